// Router kernels: logits = x Wg^T (+ b) in fp32, row softmax, top-k, gates.
//
// "How Mixture of Experts Scales Model Parameters", section "Routing: a router
// scores the experts, and the top one runs": the router is one d x E linear
// layer followed by a softmax over each row.  Section "Top-K: several experts,
// added up by weight": the K highest-scoring experts, weights renormalised
// over the chosen K.  The softmax subtracts the row maximum first (the safe
// softmax of the online-softmax section of "Inference Optimization: The
// Bandwidth Wall, PagedAttention, and FlashAttention").
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "select.cuh"

namespace moe {
namespace {

constexpr int RT_M = 64, RT_E = 64, RT_K = 32, RT_THREADS = 256;
// From this many tokens on, the bf16 router GEMM runs on the tensor cores
// (fp32 accumulation in TMEM); smaller batches use the CUDA-core kernel.
constexpr int kTensorCoreRouterMinTokens = 128;
// Up to this many tokens, the bf16 router runs one warp per expert.
constexpr int kSmallRouterMaxTokens = 96;

// logits[t][e] = sum_i x[t][i] * Wg[e][i] (+ bias[e]): each 32-wide chunk of i
// is summed with fp32 FMA into a fresh partial, and the partials are added up,
// which keeps the rounding error of long rows (d in the thousands) near 1e-7.
template <typename T>
__global__ void __launch_bounds__(RT_THREADS)
route_logits_kernel(const T *__restrict__ x, const T *__restrict__ Wg,
                    const float *__restrict__ bias, float *__restrict__ logits, int n, int d,
                    int E) {
  __shared__ float xs[RT_K][RT_M + 4];
  __shared__ float gs[RT_K][RT_E + 4];
  const int m0 = blockIdx.x * RT_M, e0 = blockIdx.y * RT_E;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += RT_K) {
    for (int i = threadIdx.x; i < RT_M * RT_K; i += RT_THREADS) {
      const int r = i / RT_K, kk = i % RT_K, gk = k0 + kk;
      const int gm = m0 + r, ge = e0 + r;
      xs[kk][r] = (gm < n && gk < d) ? Elem<T>::load(x + (size_t)gm * d + gk) : 0.f;
      gs[kk][r] = (ge < E && gk < d) ? Elem<T>::load(Wg + (size_t)ge * d + gk) : 0.f;
    }
    __syncthreads();
    float part[4][4] = {};
#pragma unroll 8
    for (int kk = 0; kk < RT_K; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = gs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] += part[i][j];
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= n) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ge = e0 + tx * 4 + j;
      if (ge < E) logits[(size_t)gm * E + ge] = acc[i][j] + (bias ? bias[ge] : 0.f);
    }
  }
}

// Small batches (decode): one warp per expert, RS_TOK tokens per CTA row.
// Lane l walks the row in 8-element pieces (l*8, l*8 + 256, ...); each piece
// is a fresh fp32 partial added to the token's sum, and the 32 lane sums are
// combined by a shuffle tree.  A lane's Wg pieces are loaded into registers
// while the CTA copies its tokens' x rows into shared memory, so the whole
// CTA waits on one round of memory latency; the dot products then read x
// from shared memory.
constexpr int RS_WARPS = 8, RS_TOK = 4, RS_MAXV = 12;    // d <= 32 * 8 * RS_MAXV = 3072

__global__ void __launch_bounds__(32 * RS_WARPS)
route_logits_small_kernel(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ Wg,
                          const float *__restrict__ bias, float *__restrict__ logits, int n, int d,
                          int E) {
  extern __shared__ __align__(16) uint4 xs[];             // [RS_TOK][d / 8]
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * RS_WARPS + warp;
  const int t0 = blockIdx.y * RS_TOK;
  const int nt = min(RS_TOK, n - t0);
  const int vpr = d / 8;
  const int nv = (vpr - lane + 31) / 32;                  // pieces of this lane: k0 = (lane + 32 v) * 8
  uint4 wv[RS_MAXV];
  if (e < E) {
    const __nv_bfloat16 *wrow = Wg + (size_t)e * d;
#pragma unroll
    for (int v = 0; v < RS_MAXV; ++v)
      if (v < nv) wv[v] = *reinterpret_cast<const uint4 *>(wrow + (size_t)(lane + 32 * v) * 8);
  }
  // all of a thread's x pieces in flight at once (at most RS_TOK * d / 8 /
  // threads = 12), then stored
  const uint4 *xsrc = reinterpret_cast<const uint4 *>(x + (size_t)t0 * d);
  constexpr int RS_STAGE = RS_TOK * 32 * 8 * RS_MAXV / 8 / (32 * RS_WARPS);
  uint4 xv_st[RS_STAGE];
#pragma unroll
  for (int j = 0; j < RS_STAGE; ++j) {
    const int i = threadIdx.x + j * 32 * RS_WARPS;
    if (i < nt * vpr) xv_st[j] = xsrc[i];
  }
#pragma unroll
  for (int j = 0; j < RS_STAGE; ++j) {
    const int i = threadIdx.x + j * 32 * RS_WARPS;
    if (i < nt * vpr) xs[i] = xv_st[j];
  }
  __syncthreads();
  if (e >= E) return;
  // the RS_TOK tokens' sums side by side, so their shuffle trees interleave
  float acc[RS_TOK];
#pragma unroll
  for (int j = 0; j < RS_TOK; ++j) acc[j] = 0.f;
#pragma unroll
  for (int v = 0; v < RS_MAXV; ++v) {
    if (v < nv) {
#pragma unroll
      for (int j = 0; j < RS_TOK; ++j)
        if (j < nt) acc[j] += bf16x8_dot(wv[v], xs[j * vpr + lane + 32 * v]);
    }
  }
  float mine = 0.f;
#pragma unroll
  for (int j = 0; j < RS_TOK; ++j) {
    acc[j] = warp_sum_xor(acc[j]);
    if (lane == j) mine = acc[j];
  }
  if (lane < nt) logits[(size_t)(t0 + lane) * E + e] = mine + (bias ? bias[e] : 0.f);
}

// One warp per token (selection and gates as in select_topk_lanes; NV =
// ceil(E / 32) logits per lane).  With nparts > 0 the logits are first
// assembled from the router's partial planes parts[p][n][E], added in plane
// order, then the bias; they are stored to logits and selected from registers.
template <int NV>
__global__ void __launch_bounds__(256)
route_select_kernel(float *__restrict__ logits, const float *__restrict__ parts, int nparts,
                    const float *__restrict__ bias, int n, int E, int k, int gate_mode,
                    int32_t *__restrict__ topk_idx, float *__restrict__ topk_gate,
                    float *__restrict__ probs) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = 0.f;
    if (e < E) {
      if (nparts > 0) {
        float a = parts[(size_t)warp * E + e];
        for (int p = 1; p < nparts; ++p) a += parts[((size_t)p * n + warp) * E + e];
        v[i] = a + (bias ? bias[e] : 0.f);
        logits[(size_t)warp * E + e] = v[i];
      } else {
        v[i] = logits[(size_t)warp * E + e];
      }
    }
  }
  select_topk_lanes<NV>(v, E, k, gate_mode, lane, topk_idx + (size_t)warp * k,
                        topk_gate + (size_t)warp * k, probs ? probs + (size_t)warp * E : nullptr);
}

}  // namespace

// Selection outputs for a router whose selection may be fused into its GEMM.
struct RouteSel {
  int32_t *idx;
  float *gate;
  float *probs;
  int *tile_count;   // zeroed [ceil(n / 128)] ints, or nullptr
};

// The tensor-core router stage for these shapes (rows >= 128, bf16), with the
// reduction split when parts has room, and the selection fused when sel is
// given and the GEMM can take it (at most 32 experts).
static GemmStage router_stage(const moe_config &c, const void *x, const void *Wg,
                              const float *bias, float *logits, float *parts, size_t parts_bytes,
                              const RouteSel *sel) {
  GemmStage g{};
  g.a_dtype = c.act_dtype;
  g.b_dtype = c.act_dtype;
  g.out_dtype = MOE_F32;
  g.epi = 3;
  g.A = x;
  g.offsets = nullptr;
  g.num_experts = 1;
  g.rows = c.n;
  g.N = c.n_experts;
  g.K = c.d;
  g.B = Wg;
  g.out = logits;
  g.col_bias = bias;
  if (c.n < kTensorCoreRouterMinTokens || !gemm_tc_supported(g)) {
    g.rows = 0;   // not on the tensor cores
    return g;
  }
  g.ksplit = parts ? gemm_tc_router_ksplit(g, parts_bytes) : 1;
  if (g.ksplit > 1) g.out = parts;
  if (sel) {
    g.sel_idx = sel->idx;
    g.sel_gate = sel->gate;
    g.sel_probs = sel->probs;
    g.logits = logits;
    g.tile_count = sel->tile_count;
    g.top_k = c.top_k;
    g.gate_mode = c.gate;
    if (!gemm_tc_router_fuses(g)) g.sel_idx = nullptr;
  }
  return g;
}

// The router's linear layer into logits, or (*nparts > 1) into nparts partial
// planes at parts that the selection adds up, or (*fused) with the selection
// done as well.
static cudaError_t route_logits(const moe_config &c, const void *x, const void *Wg,
                                const float *bias, float *logits, float *parts,
                                size_t parts_bytes, const RouteSel *sel, int *status,
                                cudaStream_t s, int *nparts, bool *fused) {
  cudaError_t err = cudaSuccess;
  *nparts = 1;
  *fused = false;
  const GemmStage g = router_stage(c, x, Wg, bias, logits, parts, parts_bytes, sel);
  dim3 grid((c.n + RT_M - 1) / RT_M, (c.n_experts + RT_E - 1) / RT_E);
  if (g.rows > 0) {
    if (g.ksplit > 1) *nparts = g.ksplit;
    *fused = g.sel_idx != nullptr;
    err = launch_gemm_tc(g, status, s);
  }
  else if (c.act_dtype == MOE_BF16 && c.n <= kSmallRouterMaxTokens && c.d <= 32 * 8 * RS_MAXV)
    err = launch_pdl(route_logits_small_kernel,
                     dim3((c.n_experts + RS_WARPS - 1) / RS_WARPS, (c.n + RS_TOK - 1) / RS_TOK),
                     dim3(32 * RS_WARPS), (size_t)RS_TOK * c.d * 2, s, (const __nv_bfloat16 *)x,
                     (const __nv_bfloat16 *)Wg, bias, logits, c.n, c.d, c.n_experts);
  else if (c.act_dtype == MOE_F32)
    route_logits_kernel<float><<<grid, RT_THREADS, 0, s>>>(
        (const float *)x, (const float *)Wg, bias, logits, c.n, c.d, c.n_experts);
  else
    route_logits_kernel<__nv_bfloat16><<<grid, RT_THREADS, 0, s>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wg, bias, logits, c.n, c.d,
        c.n_experts);
  if (err == cudaSuccess) err = cudaGetLastError();
  return err;
}

int route_kernels(const moe_config &c, size_t parts_bytes, bool have_counters) {
  // (the pointers only need to be non-null to decide)
  float dummy;
  int32_t didx;
  int dcount;
  const RouteSel sel{&didx, &dummy, nullptr, have_counters ? &dcount : nullptr};
  const GemmStage g = router_stage(c, &dummy, &dummy, nullptr, &dummy,
                                   parts_bytes ? &dummy : nullptr, parts_bytes, &sel);
  return (g.rows > 0 && g.sel_idx != nullptr) ? 1 : 2;
}

cudaError_t launch_route_logits(const moe_config &c, const void *x, const void *Wg,
                                const float *bias, float *logits, int *status, cudaStream_t s) {
  int nparts = 1;
  bool fused = false;
  return route_logits(c, x, Wg, bias, logits, nullptr, 0, nullptr, status, s, &nparts, &fused);
}

cudaError_t launch_route(const moe_config &c, const void *x, const void *Wg, const float *bias,
                         float *logits, float *parts, size_t parts_bytes, int32_t *topk_idx,
                         float *topk_gate, float *probs, int *status, cudaStream_t s,
                         int *tile_count) {
  int nparts = 1;
  bool fused = false;
  const RouteSel sel{topk_idx, topk_gate, probs, tile_count};
  cudaError_t err = route_logits(c, x, Wg, bias, logits, parts, parts_bytes, &sel, status, s,
                                 &nparts, &fused);
  if (err != cudaSuccess || fused) return err;
  const int warps_per_block = 8;
  const dim3 grid((c.n + warps_per_block - 1) / warps_per_block), block(32 * warps_per_block);
  const int np = nparts > 1 ? nparts : 0;
  const int E = c.n_experts;
  if (E <= 32)
    route_select_kernel<1><<<grid, block, 0, s>>>(logits, parts, np, bias, c.n, E, c.top_k,
                                                  c.gate, topk_idx, topk_gate, probs);
  else if (E <= 64)
    route_select_kernel<2><<<grid, block, 0, s>>>(logits, parts, np, bias, c.n, E, c.top_k,
                                                  c.gate, topk_idx, topk_gate, probs);
  else if (E <= 128)
    route_select_kernel<4><<<grid, block, 0, s>>>(logits, parts, np, bias, c.n, E, c.top_k,
                                                  c.gate, topk_idx, topk_gate, probs);
  else
    route_select_kernel<8><<<grid, block, 0, s>>>(logits, parts, np, bias, c.n, E, c.top_k,
                                                  c.gate, topk_idx, topk_gate, probs);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Routing statistics ("How Mixture of Experts Scales Model Parameters",
// section "Load balancing: how collapse happens, and how it's kept in check"):
//   P_i = (1/n) sum_t p_i(t),  f_i = (1/n) #{t : argmax_e p_e(t) = i},
//   aux = alpha * E * sum_i f_i P_i.
// One CTA per 32 experts: lane = expert, warp w takes rows w, w+8, ...; each
// run of 64 rows is summed into a fresh partial, the warp partials are added
// in warp order, so the result does not depend on scheduling.
namespace moe {
namespace {

constexpr int ST_WARPS = 8;

__global__ void __launch_bounds__(32 * ST_WARPS)
route_stats_kernel(const float *__restrict__ probs, const int32_t *__restrict__ topk_idx, int n,
                   int E, int k, float *__restrict__ P, float *__restrict__ f, int *status) {
  __shared__ float ps[ST_WARPS][32];
  __shared__ int pc[ST_WARPS][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  float sum = 0.f, part = 0.f;
  int count = 0, in_part = 0;
  for (int t = warp; t < n; t += ST_WARPS) {
    if (e < E) part += probs[(size_t)t * E + e];
    const int a = topk_idx[(size_t)t * k];
    if (a < 0 || a >= E) {
      if (lane == 0 && blockIdx.x == 0) set_status(status, MOE_ERR_BAD_INDEX, t * k);
    } else if (a == e) {
      ++count;
    }
    if (++in_part == 64) {
      sum += part;
      part = 0.f;
      in_part = 0;
    }
  }
  ps[warp][lane] = sum + part;
  pc[warp][lane] = count;
  __syncthreads();
  if (warp == 0 && e < E) {
    float s = 0.f;
    int c = 0;
    for (int w = 0; w < ST_WARPS; ++w) {
      s += ps[w][lane];
      c += pc[w][lane];
    }
    P[e] = s / (float)n;
    f[e] = (float)c / (float)n;
  }
}

// aux = alpha * E * sum_i f_i P_i, a fixed-order tree over one CTA.
__global__ void __launch_bounds__(256)
route_aux_kernel(const float *__restrict__ P, const float *__restrict__ f, int E, float alpha,
                 float *__restrict__ aux) {
  __shared__ float v[256];
  v[threadIdx.x] = threadIdx.x < E ? f[threadIdx.x] * P[threadIdx.x] : 0.f;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (threadIdx.x < o) v[threadIdx.x] += v[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *aux = alpha * (float)E * v[0];
}

}  // namespace

cudaError_t launch_route_stats(const moe_config &c, const float *probs, const int32_t *topk_idx,
                               float alpha, float *P, float *f, float *aux, int *status,
                               cudaStream_t s) {
  route_stats_kernel<<<(c.n_experts + 31) / 32, 32 * ST_WARPS, 0, s>>>(
      probs, topk_idx, c.n, c.n_experts, c.top_k, P, f, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  route_aux_kernel<<<1, 256, 0, s>>>(P, f, c.n_experts, alpha, aux);
  return cudaGetLastError();
}

}  // namespace moe
