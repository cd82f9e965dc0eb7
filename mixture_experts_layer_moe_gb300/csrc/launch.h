// Host-side launchers of the MoE kernels (internal; the public ABI is moe.h).
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Launch with programmatic stream serialisation: the kernel may be scheduled
// before the previous kernel in the stream completes (it must call pdl_wait()
// before touching memory that earlier kernels use).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tensor-map encoding (cuTensorMapEncodeTiled through the runtime's driver
// entry point), innermost dimension first, dense strides; and the SM count.
bool tensor_maps_available();
bool make_tensor_map(CUtensorMap *m, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                     int rank, const uint64_t *dims, const uint32_t *box,
                     CUtensorMapSwizzle swizzle);
int num_sms();

// Router: logits (fp32 [n][E] scratch) -> softmax -> top-k -> gates.
// parts (nullable, parts_bytes long) is scratch for partial logits when the
// tensor-core router splits its reduction over more SMs.
// tile_count (nullable): ceil(n / 128) zeroed ints, which let a router with
// at most 32 experts and a split reduction run its selection in the GEMM.
cudaError_t launch_route(const moe_config &c, const void *x, const void *Wg, const float *bias,
                         float *logits, float *parts, size_t parts_bytes, int32_t *topk_idx,
                         float *topk_gate, float *probs, int *status, cudaStream_t s,
                         int *tile_count = nullptr);
// Kernels launch_route launches for these shapes (1 when the selection runs
// in the router's GEMM, else 2).
int route_kernels(const moe_config &c, size_t parts_bytes, bool have_counters);
// The router's linear layer alone: logits [n][E] fp32.
cudaError_t launch_route_logits(const moe_config &c, const void *x, const void *Wg,
                                const float *bias, float *logits, int *status, cudaStream_t s);

// Device address of moe_route_noalloc's status word on the current device.
moe_status noalloc_status_word(int **out);

// Routing statistics: P [E], f [E] and aux (one float) from probs [n][E] and
// the top-1 column of topk_idx.
cudaError_t launch_route_stats(const moe_config &c, const float *probs, const int32_t *topk_idx,
                               float alpha, float *P, float *f, float *aux, int *status,
                               cudaStream_t s);

// Stable counting sort of P pairs by expert (one CTA).
// From kDispatchManyMinPairs pairs on, the sort runs over one CTA per SM (two
// launches) when scratch holds SMs * E int32 (per-range counts); otherwise one
// CTA.  Both give the same arrays.
constexpr int kDispatchManyMinPairs = 16384;
cudaError_t launch_dispatch(int P, int E, const int32_t *topk_idx, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv_perm, int *status,
                            cudaStream_t s, void *scratch = nullptr, size_t scratch_bytes = 0);
// Kernels launch_dispatch launches for these arguments (1 or 2).
int dispatch_kernels(int P, int E, const void *scratch, size_t scratch_bytes);

// x_perm[q] = x[perm[q] / k]; rows of row_bytes (multiple of 16).
// x_perm[inv_perm[t*k + j]] = x[t] in token order: each x row read once
// (pairs with inv_perm < 0 skipped, >= P reported).
cudaError_t launch_scatter_rows(const void *x, const int32_t *inv_perm, int P, int k, int n,
                                int64_t row_bytes, void *x_perm, int *status, cudaStream_t s);
cudaError_t launch_gather(const void *x, const int32_t *perm, int P, int k, int n,
                          int64_t row_bytes, void *x_perm, int *status, cudaStream_t s);

// y[t] = sum_j g[t][j] * y_perm[inv[t*k+j]] (+ y_shared[t]).
cudaError_t launch_combine(int act_dtype, const void *y_perm, const int32_t *inv_perm,
                           const float *gates, const void *y_shared, void *y, int n, int k,
                           int d, int *status, cudaStream_t s);

// One grouped GEMM stage on CUDA cores (fp32 accumulate):
//   out[q][j] = epi( sum_i A[q][i] * B_e[j][i] )  for q in segment e.
// epi: 0 = none, 1 = relu, 2 = swiglu (B3 gives the linear branch),
//      3 = fp32 output + col_bias[j] (router logits; tensor-core path only).
// offsets == nullptr means one segment [0, rows) using expert 0.
// Internal element type: f16 activation copies feeding the MXFP4 tensor-core path.
constexpr int kF16 = 3;

struct GemmStage {
  int a_dtype;          // MOE_F32 / MOE_BF16 / kF16
  int b_dtype;          // MOE_F32 / MOE_BF16 / MOE_MXFP4
  int out_dtype;        // MOE_F32 / MOE_BF16
  int epi;
  const void *A;
  const int32_t *offsets;
  int num_experts;
  int rows;             // total rows of A (P)
  int N, K;
  const void *B;        // [E][N][K] (or codes [E][N][K/2])
  const uint8_t *SB;    // scales [E][N][K/32]
  const void *B3;
  const uint8_t *SB3;
  void *out;            // [rows][N]
  const float *col_bias; // epi 3: per-column bias or nullptr
  void *out16;          // MXFP4 path: f16 copy of out (next projection's input) or nullptr
  int ksplit;           // epi 3 on tensor cores: k ranges per row tile; > 1 writes
                        // partial sums to planes out[p][rows][N] without the bias
  // epi 3 with N <= 32 on tensor cores: top-k selection fused into the GEMM
  // when sel_idx is set (logits [rows][N] written, probs optional); with
  // ksplit > 1 it needs tile_count, one zeroed int per 128-row tile
  int32_t *sel_idx;
  float *sel_gate;
  float *sel_probs;
  float *logits;
  int *tile_count;
  int top_k, gate_mode;
};
cudaError_t launch_gemm_simt(const GemmStage &g, int *status, cudaStream_t s);

// The same stage on tcgen05 tensor cores (fp32 accumulate in TMEM, TMA-fed):
// MXFP4 weights go to gemm_mx.cu, bf16 expert projections (epi 0-2) to the
// SM-pair kernel of gemm_t2.cu, the router (epi 3) to gemm_tc.cu;
// gemm_tc_supported() says whether the shape/dtypes qualify.
bool gemm_tc_supported(const GemmStage &g);
cudaError_t launch_gemm_tc(const GemmStage &g, int *status, cudaStream_t s);
// Split of the router's reduction that fills the SMs (1: no split), given
// room in bytes for the fp32 partial planes.
int gemm_tc_router_ksplit(const GemmStage &g, size_t plane_room);
// Whether launch_gemm_tc runs this router stage with the selection fused.
bool gemm_tc_router_fuses(const GemmStage &g);
// The bf16 grouped GEMM (epi 0, 1, 2) on SM pairs: tcgen05.mma.cta_group::2
// with 256 weight rows on M and up to 256 tokens on N (gemm_t2.cu).
bool gemm_t2_supported(const GemmStage &g);
cudaError_t launch_gemm_t2(const GemmStage &g, int *status, cudaStream_t s);
// MXFP4 grouped GEMM with the dequantised weights as the tcgen05 A operand in
// tensor memory (f16 activation copies in, bf16 out; epi 0, 1 or 2).
bool gemm_mx_supported(const GemmStage &g);
cudaError_t launch_gemm_mx(const GemmStage &g, int *status, cudaStream_t s);

// Picks the tensor-core kernel when it applies, else the CUDA-core one.
inline cudaError_t launch_gemm(const GemmStage &g, int *status, cudaStream_t s) {
  if (g.rows == 0) return cudaSuccess;
  return gemm_tc_supported(g) ? launch_gemm_tc(g, status, s) : launch_gemm_simt(g, status, s);
}

// Small-batch MXFP4 path over the selected experts only, weights streamed
// once and dequantised in registers.  part 0: f16 copies of the activation
// rows in segment order (x [n][d] gathered through perm, or x_perm [P][d] when
// perm is nullptr) into act16, then up + activation -> h [P][d_ff] (bf16, and
// an f16 copy in act16).  part 1: down -> y_perm [P][d].  act16 is workspace
// of mx_act16_bytes(c).
constexpr int kDecodeMaxPairs = 256;
bool decode_supported(const moe_config &c);
// Workspace for f16 copies of the activation rows ([P][d] then [P][d_ff]) used
// by both MXFP4 paths; 0 for other configurations.
size_t mx_act16_bytes(const moe_config &c);
// dst[q] = f16(src[perm[q] / top_k]) (perm given) or f16(src[q]); rows of K.
// dst[inv_perm[t*k + j]] = f16(src[t]) in token order, each row converted once.
cudaError_t launch_rows_to_f16_scatter(const void *src, const int32_t *inv_perm, int top_k, int n,
                                       int K, void *dst, int *status, cudaStream_t s);
cudaError_t launch_rows_to_f16(const void *src, const int32_t *perm, int top_k, int P, int K,
                               void *dst, int *status, cudaStream_t s);
// part 0 with act == nullptr: act16 already holds the f16 x rows in token order
// (as launch_decode_route writes them), read through perm.  With a pool, an
// expert e with pool->slot_of[e] >= 0 is read from that slot of the pool.
cudaError_t launch_decode_ffn(const moe_config &c, int part, const void *act,
                              const int32_t *perm, const int32_t *offsets, const moe_weights &w,
                              void *h, void *y_perm, void *act16, int *status, cudaStream_t s,
                              const moe_expert_pool *pool = nullptr);
cudaError_t launch_decode_ffn_nvfp4(const moe_config &c, int part, const void *act,
                                    const int32_t *perm, const int32_t *offsets,
                                    const moe_weights &w, void *h, void *y_perm, void *act16,
                                    int *status, cudaStream_t s);
cudaError_t launch_decode_ffn_pooled(const moe_config &c, int part, const void *act,
                                     const int32_t *perm, const int32_t *offsets,
                                     const moe_weights &w, void *h, void *y_perm, void *act16,
                                     int *status, cudaStream_t s, const moe_expert_pool &pool);
// Small-batch routing in one launch (decode_supported configurations with a
// bf16 x): selection and gates from the logits, counts / offsets / perm /
// inv_perm of the stable dispatch, and the f16 x rows in token order (act16,
// as launch_decode_ffn part 0 reads them with act == nullptr).
bool decode_route_supported(const moe_config &c);
// With a pool, CTA 0 also classifies the selected experts against it (state,
// miss_list, pool_counts as moe_classify_experts writes them; each nullable).
cudaError_t launch_decode_route(const moe_config &c, const float *logits, const void *x,
                                int32_t *topk_idx, float *topk_gate, int32_t *counts,
                                int32_t *offsets, int32_t *perm, int32_t *inv_perm, void *act16,
                                int *status, cudaStream_t s,
                                const moe_expert_pool *pool = nullptr, int32_t *state = nullptr,
                                int32_t *miss_list = nullptr, int32_t *pool_counts = nullptr);
// The whole small-batch layer in one cooperative launch (decode_layer.cu):
// router, selection, dispatch, both expert projections and combine, for
// SwiGLU experts with d <= 3072: MXFP4 (also from a pool) with n <= 16
// tokens, NVFP4 (no pool) with n <= 8.  The chained launches above cover the
// rest, and are faster beyond those sizes.  It writes the workspace
// arrays the chained path writes; sync is decode_layer_sync_bytes() of
// zeroed counters.
struct DecodeLayerBuffers {
  float *logits;
  int32_t *topk_idx;
  float *topk_gate;
  int32_t *counts, *offsets, *perm, *inv_perm;
  void *act16, *h, *y_perm, *y;
  int *sync;
  int *status;
  int32_t *state, *miss_list, *pool_counts;   // with a pool (each nullable)
};
bool decode_layer_supported(const moe_config &c, bool pooled);
size_t decode_layer_sync_bytes();
cudaError_t launch_decode_layer(const moe_config &c, const void *x, const moe_weights &w,
                                const moe_expert_pool *pool, const DecodeLayerBuffers &b,
                                cudaStream_t s);
// Hit/miss classification of topk_idx against slot_of (one CTA; E <= 256).
cudaError_t launch_classify(const moe_config &c, const int32_t *topk_idx, const int32_t *slot_of,
                            int n_slots, int32_t *state, int32_t *miss_list, int32_t *counts,
                            int *status, cudaStream_t s);

}  // namespace moe
