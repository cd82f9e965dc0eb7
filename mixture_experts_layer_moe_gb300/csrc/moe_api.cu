// The C ABI (include/moe.h): argument validation, workspace layout, and the
// launch sequence of the MoE layer forward pass.
#include <stdint.h>
#include <string.h>

#include "launch.h"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool ok_ptr(const void *p) { return p != nullptr && aligned(p, 16); }
cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }
int act_size(const moe_config &c) { return c.act_dtype == MOE_F32 ? 4 : 2; }
int h_size(const moe_config &c) { return c.act_dtype == MOE_F32 ? 4 : 2; }

moe_status check_config(const moe_config *c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->n < 1 || c->d < 1 || c->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->n_experts > 256) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->weight_dtype != MOE_F32 && c->weight_dtype != MOE_BF16 && c->weight_dtype != MOE_MXFP4 &&
      c->weight_dtype != MOE_NVFP4)
    return MOE_ERR_INVALID_ARG;
  if (c->gate != MOE_GATE_TOP_PROB && c->gate != MOE_GATE_RENORM) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->d_ff_shared < 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)c->n * c->top_k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
  // fp32 activations go with fp32 weights; bf16 activations with bf16 or MXFP4
  if (c->act_dtype == MOE_F32 && c->weight_dtype != MOE_F32) return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype == MOE_BF16 && c->weight_dtype == MOE_F32) return MOE_ERR_UNSUPPORTED;
  // rows must be whole 16-byte vectors
  const int vec = c->act_dtype == MOE_F32 ? 4 : 8;
  if (c->d % vec || c->d_ff % vec || c->d_ff_shared % vec) return MOE_ERR_UNSUPPORTED;
  const bool fp4 = c->weight_dtype == MOE_MXFP4 || c->weight_dtype == MOE_NVFP4;
  if (fp4 && (c->d % 32 || c->d_ff % 32)) return MOE_ERR_UNSUPPORTED;
  // NVFP4 runs on the small-batch path only
  if (c->weight_dtype == MOE_NVFP4 &&
      (c->act_dtype != MOE_BF16 || (int64_t)c->n * c->top_k > kDecodeMaxPairs))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_router_weights(const moe_config &c, const moe_weights *w) {
  if (w == nullptr || !ok_ptr(w->Wg)) return MOE_ERR_INVALID_ARG;
  if (w->router_bias != nullptr && !aligned(w->router_bias, 4)) return MOE_ERR_INVALID_ARG;
  (void)c;
  return MOE_OK;
}

moe_status check_expert_weights(const moe_config &c, const moe_weights *w) {
  if (w == nullptr || !ok_ptr(w->W1) || !ok_ptr(w->W2)) return MOE_ERR_INVALID_ARG;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (swiglu != (w->W3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (swiglu && !ok_ptr(w->W3)) return MOE_ERR_INVALID_ARG;
  const bool nv = c.weight_dtype == MOE_NVFP4;
  if (nv) {
    if (!w->G1 || !w->G2 || !aligned(w->G1, 4) || !aligned(w->G2, 4)) return MOE_ERR_INVALID_ARG;
    if (swiglu != (w->G3 != nullptr) || (swiglu && !aligned(w->G3, 4))) return MOE_ERR_INVALID_ARG;
  } else if (w->G1 || w->G2 || w->G3) {
    return MOE_ERR_INVALID_ARG;
  }
  if (c.weight_dtype == MOE_MXFP4 || nv) {
    if (!ok_ptr(w->S1) || !ok_ptr(w->S2)) return MOE_ERR_INVALID_ARG;
    if (swiglu != (w->S3 != nullptr)) return MOE_ERR_INVALID_ARG;
    if (swiglu && !ok_ptr(w->S3)) return MOE_ERR_INVALID_ARG;
  } else if (w->S1 || w->S2 || w->S3) {
    return MOE_ERR_INVALID_ARG;
  }
  if (c.d_ff_shared > 0) {
    if (!ok_ptr(w->Ws1) || !ok_ptr(w->Ws3) || !ok_ptr(w->Ws2)) return MOE_ERR_INVALID_ARG;
  } else if (w->Ws1 || w->Ws3 || w->Ws2) {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

struct Layout {
  size_t status, route_count, sync, logits, topk_idx, topk_gate, counts, offsets, perm, inv_perm,
      x_perm, h, y_perm, y_shared, h_shared, act16, total;
};

Layout layout_of(const moe_config &c) {
  Layout L{};
  const size_t n = c.n, E = c.n_experts, P = (size_t)c.n * c.top_k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  L.status = take(kAlign);
  // right after the status word, so that one memset clears them all: per
  // 128-row router tile, the CTAs of a split reduction that have finished it;
  // then the counters of the fused small-batch layer launch
  L.route_count = take(((size_t)c.n + 127) / 128 * 4);
  L.sync = take(decode_layer_sync_bytes());
  L.logits = take(n * E * 4);
  L.topk_idx = take(P * 4);
  L.topk_gate = take(P * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(P * 4);
  L.inv_perm = take(P * 4);
  L.x_perm = take(P * c.d * act_size(c));
  L.h = take(P * c.d_ff * h_size(c));
  L.y_perm = take(P * c.d * act_size(c));
  L.y_shared = c.d_ff_shared ? take(n * c.d * act_size(c)) : 0;
  L.h_shared = c.d_ff_shared ? take(n * c.d_ff_shared * h_size(c)) : 0;
  const size_t a16 = mx_act16_bytes(c);
  L.act16 = a16 ? take(a16) : 0;
  L.total = off;
  return L;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

moe_status check_ws(const moe_config &c, const void *ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout_of(c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Bytes from the status word through the per-launch counters (one memset
// clears them all before a forward pass).
size_t cleared_bytes(const Layout &L) { return L.sync - L.status + decode_layer_sync_bytes(); }

#define MOE_TRY(expr)                   \
  do {                                  \
    const moe_status _st = (expr);      \
    if (_st != MOE_OK) return _st;      \
  } while (0)

// The two GEMM stages of the MXFP4 tensor-core path (f16 activations).
void mx_stages(const moe_config &c, const int32_t *offsets, const moe_weights *w, void *ws,
               void *y_perm, GemmStage &up, GemmStage &dn) {
  const Layout L = layout_of(c);
  const int P = c.n * c.top_k;
  uint16_t *x16 = at<uint16_t>(ws, L.act16);
  uint16_t *h16 = x16 + (size_t)P * c.d;
  up = GemmStage{};
  up.a_dtype = kF16;
  up.b_dtype = MOE_MXFP4;
  up.out_dtype = MOE_BF16;
  up.epi = c.act == MOE_ACT_RELU ? 1 : 2;
  up.A = x16;
  up.offsets = offsets;
  up.num_experts = c.n_experts;
  up.rows = P;
  up.N = c.d_ff;
  up.K = c.d;
  up.B = w->W1;
  up.SB = w->S1;
  up.B3 = w->W3;
  up.SB3 = w->S3;
  up.out = at<void>(ws, L.h);
  up.out16 = h16;
  dn = up;
  dn.epi = 0;
  dn.A = h16;
  dn.N = c.d;
  dn.K = c.d_ff;
  dn.B = w->W2;
  dn.SB = w->S2;
  dn.B3 = nullptr;
  dn.SB3 = nullptr;
  dn.out = y_perm;
  dn.out16 = nullptr;
}

bool mx_tc_path(const moe_config &c) {
  if (c.weight_dtype != MOE_MXFP4 || c.act_dtype != MOE_BF16 || decode_supported(c)) return false;
  moe_weights w{};
  GemmStage up, dn;
  mx_stages(c, nullptr, &w, nullptr, nullptr, up, dn);
  up.offsets = dn.offsets = reinterpret_cast<const int32_t *>(16);   // shape check only
  return gemm_tc_supported(up) && gemm_tc_supported(dn);
}

// MXFP4 prefill on tensor cores: f16 copies of the expert-ordered rows (x
// scattered in token order through inv_perm: the dispatch's gather of the
// rows, run before the FFN stage begins; or x_perm converted in place), then
// the up and down grouped GEMMs with on-the-fly dequantisation.
template <typename StageFn>
moe_status run_mx_ffn(const moe_config &c, const void *act, const int32_t *inv_perm,
                      const int32_t *offsets, const moe_weights *w, void *y_perm, void *ws,
                      cudaStream_t s, StageFn &&stage) {
  const Layout L = layout_of(c);
  int *status = at<int>(ws, L.status);
  GemmStage up, dn;
  mx_stages(c, offsets, w, ws, y_perm, up, dn);
  if (inv_perm) {
    MOE_TRY(cuda_status(launch_rows_to_f16_scatter(act, inv_perm, c.top_k, c.n, c.d,
                                                   at<void>(ws, L.act16), status, s)));
    stage(MOE_STAGE_FFN_UP, 1);
  } else {
    stage(MOE_STAGE_FFN_UP, 2);
    MOE_TRY(cuda_status(launch_rows_to_f16(act, nullptr, c.top_k, c.n * c.top_k, c.d,
                                           at<void>(ws, L.act16), status, s)));
  }
  MOE_TRY(cuda_status(launch_gemm_tc(up, status, s)));
  stage(MOE_STAGE_FFN_DOWN, 1);
  return cuda_status(launch_gemm_tc(dn, status, s));
}

template <typename StageFn>
moe_status run_expert_ffn(const moe_config &c, const void *x_perm, const int32_t *offsets,
                          const moe_weights *w, void *y_perm, void *ws, cudaStream_t s,
                          StageFn &&stage) {
  const Layout L = layout_of(c);
  int *status = at<int>(ws, L.status);
  if (decode_supported(c)) {
    stage(MOE_STAGE_FFN_UP, 2);
    MOE_TRY(cuda_status(launch_decode_ffn(c, 0, x_perm, nullptr, offsets, *w, at<void>(ws, L.h),
                                          y_perm, at<void>(ws, L.act16), status, s)));
    stage(MOE_STAGE_FFN_DOWN, 1);
    return cuda_status(launch_decode_ffn(c, 1, x_perm, nullptr, offsets, *w, at<void>(ws, L.h),
                                         y_perm, at<void>(ws, L.act16), status, s));
  }
  if (mx_tc_path(c)) return run_mx_ffn(c, x_perm, nullptr, offsets, w, y_perm, ws, s, stage);
  const int P = c.n * c.top_k;
  const int hdt = c.act_dtype == MOE_F32 ? MOE_F32 : MOE_BF16;
  GemmStage up{};
  up.a_dtype = c.act_dtype;
  up.b_dtype = c.weight_dtype;
  up.out_dtype = hdt;
  up.epi = c.act == MOE_ACT_RELU ? 1 : 2;
  up.A = x_perm;
  up.offsets = offsets;
  up.num_experts = c.n_experts;
  up.rows = P;
  up.N = c.d_ff;
  up.K = c.d;
  up.B = w->W1;
  up.SB = w->S1;
  up.B3 = w->W3;
  up.SB3 = w->S3;
  up.out = at<void>(ws, L.h);
  stage(MOE_STAGE_FFN_UP, 1);
  MOE_TRY(cuda_status(launch_gemm(up, status, s)));
  GemmStage dn = up;
  dn.a_dtype = hdt;
  dn.epi = 0;
  dn.A = up.out;
  dn.N = c.d;
  dn.K = c.d_ff;
  dn.B = w->W2;
  dn.SB = w->S2;
  dn.B3 = nullptr;
  dn.SB3 = nullptr;
  dn.out = y_perm;
  stage(MOE_STAGE_FFN_DOWN, 1);
  return cuda_status(launch_gemm(dn, status, s));
}

// The small-batch forward.  MXFP4 SwiGLU layers within the fused kernel's
// range run as one cooperative launch (decode_layer.cu).  Otherwise: the
// router's linear layer, selection + dispatch + f16 x rows in one launch
// (plus the hit/miss classification against the pool, if any), the two FFN
// kernels streaming the selected experts (from their pool slots where
// resident), combine.  Both write the same workspace arrays.
template <typename StageFn>
moe_status run_small_batch(const moe_config &c, const void *x, const moe_weights *w,
                           const moe_expert_pool *pool, void *y, int32_t *state,
                           int32_t *miss_list, int32_t *pool_counts, void *ws, cudaStream_t s,
                           StageFn &&stage) {
  const Layout L = layout_of(c);
  int *status = at<int>(ws, L.status);
  int32_t *offsets = at<int32_t>(ws, L.offsets);
  int32_t *perm = at<int32_t>(ws, L.perm);
  int32_t *inv_perm = at<int32_t>(ws, L.inv_perm);
  float *gates = at<float>(ws, L.topk_gate);
  if (decode_layer_supported(c, pool != nullptr)) {
    DecodeLayerBuffers b{};
    b.logits = at<float>(ws, L.logits);
    b.topk_idx = at<int32_t>(ws, L.topk_idx);
    b.topk_gate = gates;
    b.counts = at<int32_t>(ws, L.counts);
    b.offsets = offsets;
    b.perm = perm;
    b.inv_perm = inv_perm;
    b.act16 = at<void>(ws, L.act16);
    b.h = at<void>(ws, L.h);
    b.y_perm = at<void>(ws, L.y_perm);
    b.y = y;
    b.sync = at<int>(ws, L.sync);
    b.status = status;
    b.state = state;
    b.miss_list = miss_list;
    b.pool_counts = pool_counts;
    stage(MOE_STAGE_FUSED, 1);
    MOE_TRY(cuda_status(launch_decode_layer(c, x, *w, pool, b, s)));
    stage(MOE_STAGE_END, 0);
    return MOE_OK;
  }
  stage(MOE_STAGE_ROUTE, 1);
  MOE_TRY(cuda_status(launch_route_logits(c, x, w->Wg, w->router_bias, at<float>(ws, L.logits),
                                          status, s)));
  stage(MOE_STAGE_DISPATCH, 1);
  MOE_TRY(cuda_status(launch_decode_route(c, at<float>(ws, L.logits), x,
                                          at<int32_t>(ws, L.topk_idx), gates,
                                          at<int32_t>(ws, L.counts), offsets, perm, inv_perm,
                                          at<void>(ws, L.act16), status, s, pool, state, miss_list,
                                          pool_counts)));
  stage(MOE_STAGE_FFN_UP, 1);
  MOE_TRY(cuda_status(launch_decode_ffn(c, 0, nullptr, perm, offsets, *w, at<void>(ws, L.h),
                                        at<void>(ws, L.y_perm), at<void>(ws, L.act16), status, s,
                                        pool)));
  stage(MOE_STAGE_FFN_DOWN, 1);
  MOE_TRY(cuda_status(launch_decode_ffn(c, 1, nullptr, perm, offsets, *w, at<void>(ws, L.h),
                                        at<void>(ws, L.y_perm), at<void>(ws, L.act16), status, s,
                                        pool)));
  stage(MOE_STAGE_COMBINE, 1);
  MOE_TRY(cuda_status(launch_combine(c.act_dtype, at<void>(ws, L.y_perm), inv_perm, gates, nullptr,
                                     y, c.n, c.top_k, c.d, status, s)));
  stage(MOE_STAGE_END, 0);
  return MOE_OK;
}

moe_status check_pool(const moe_config &c, const moe_expert_pool *p) {
  if (p == nullptr || !ok_ptr(p->slot_of) || p->n_slots < 1) return MOE_ERR_INVALID_ARG;
  const bool swiglu = c.act == MOE_ACT_SWIGLU;
  if (!ok_ptr(p->W1) || !ok_ptr(p->W2) || !ok_ptr(p->S1) || !ok_ptr(p->S2))
    return MOE_ERR_INVALID_ARG;
  if (swiglu != (p->W3 != nullptr) || swiglu != (p->S3 != nullptr)) return MOE_ERR_INVALID_ARG;
  if (swiglu && (!ok_ptr(p->W3) || !ok_ptr(p->S3))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status run_shared_expert(const moe_config &c, const void *x, const moe_weights *w, void *ws,
                             cudaStream_t s) {
  const Layout L = layout_of(c);
  int *status = at<int>(ws, L.status);
  const int hdt = c.act_dtype == MOE_F32 ? MOE_F32 : MOE_BF16;
  GemmStage up{};
  up.a_dtype = c.act_dtype;
  up.b_dtype = c.act_dtype;
  up.out_dtype = hdt;
  up.epi = 2;
  up.A = x;
  up.offsets = nullptr;
  up.num_experts = 1;
  up.rows = c.n;
  up.N = c.d_ff_shared;
  up.K = c.d;
  up.B = w->Ws1;
  up.B3 = w->Ws3;
  up.out = at<void>(ws, L.h_shared);
  MOE_TRY(cuda_status(launch_gemm(up, status, s)));
  GemmStage dn = up;
  dn.a_dtype = hdt;
  dn.epi = 0;
  dn.A = up.out;
  dn.N = c.d;
  dn.K = c.d_ff_shared;
  dn.B = w->Ws2;
  dn.B3 = nullptr;
  dn.out = at<void>(ws, L.y_shared);
  return cuda_status(launch_gemm(dn, status, s));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes) {
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(*cfg).total;
  return MOE_OK;
}

moe_status moe_workspace_layout_of(const moe_config *cfg, moe_workspace_layout *out) {
  MOE_TRY(check_config(cfg));
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  out->status = L.status;
  out->logits = L.logits;
  out->topk_idx = L.topk_idx;
  out->topk_gate = L.topk_gate;
  out->counts = L.counts;
  out->offsets = L.offsets;
  out->perm = L.perm;
  out->inv_perm = L.inv_perm;
  out->x_perm = L.x_perm;
  out->h = L.h;
  out->y_perm = L.y_perm;
  out->y_shared = L.y_shared;
  out->h_shared = L.h_shared;
  out->act16 = L.act16;
  out->total = L.total;
  return MOE_OK;
}

moe_status moe_route(const moe_config *cfg, const void *x, const moe_weights *w,
                     int32_t *topk_idx, float *topk_gate, float *probs, void *ws,
                     size_t ws_bytes, void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  MOE_TRY(check_router_weights(c, w));
  if (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(topk_gate)) return MOE_ERR_INVALID_ARG;
  if (probs != nullptr && !aligned(probs, 16)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  // (the h region is scratch for the router's partial logits)
  return cuda_status(launch_route(c, x, w->Wg, w->router_bias, at<float>(ws, L.logits),
                                  at<float>(ws, L.h), (size_t)c.n * c.top_k * c.d_ff * h_size(c),
                                  topk_idx, topk_gate, probs, at<int>(ws, L.status),
                                  as_stream(stream)));
}

moe_status moe_route_stats(const moe_config *cfg, const float *probs, const int32_t *topk_idx,
                           float alpha, float *P, float *f, float *aux, void *ws,
                           size_t ws_bytes, void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (!ok_ptr(probs) || !ok_ptr(topk_idx) || !ok_ptr(P) || !ok_ptr(f) || aux == nullptr ||
      !aligned(aux, 4))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  return cuda_status(launch_route_stats(c, probs, topk_idx, alpha, P, f, aux,
                                        at<int>(ws, L.status), as_stream(stream)));
}

moe_status moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                        int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                        void *x_perm, void *ws, size_t ws_bytes, void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (!ok_ptr(topk_idx) || !ok_ptr(counts) || !ok_ptr(offsets) || !ok_ptr(perm) ||
      !ok_ptr(inv_perm))
    return MOE_ERR_INVALID_ARG;
  if (x_perm != nullptr && !ok_ptr(x)) return MOE_ERR_INVALID_ARG;
  if (x_perm != nullptr && !ok_ptr(x_perm)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  int *status = at<int>(ws, L.status);
  const int P = c.n * c.top_k;
  cudaStream_t s = as_stream(stream);
  MOE_TRY(cuda_status(
      launch_dispatch(P, c.n_experts, topk_idx, counts, offsets, perm, inv_perm, status, s,
                      at<void>(ws, L.h), (size_t)P * c.d_ff * h_size(c))));
  if (x_perm != nullptr)
    MOE_TRY(cuda_status(launch_gather(x, perm, P, c.top_k, c.n, (int64_t)c.d * act_size(c),
                                      x_perm, status, s)));
  return MOE_OK;
}

moe_status moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets,
                          const moe_weights *w, void *y_perm, void *ws, size_t ws_bytes,
                          void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (c.d_ff_shared != 0) {
    // the routed experts only; shared-expert weights are not read here
    moe_config c2 = c;
    c2.d_ff_shared = 0;
    moe_weights w2 = w ? *w : moe_weights{};
    w2.Ws1 = w2.Ws2 = w2.Ws3 = nullptr;
    MOE_TRY(check_expert_weights(c2, &w2));
  } else {
    MOE_TRY(check_expert_weights(c, w));
  }
  if (!ok_ptr(x_perm) || !ok_ptr(offsets) || !ok_ptr(y_perm)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  return run_expert_ffn(c, x_perm, offsets, w, y_perm, ws, as_stream(stream), [](int, int) {});
}

moe_status moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *inv_perm,
                       const float *topk_gate, const void *y_shared, void *y, void *ws,
                       size_t ws_bytes, void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (!ok_ptr(y_perm) || !ok_ptr(inv_perm) || !ok_ptr(topk_gate) || !ok_ptr(y))
    return MOE_ERR_INVALID_ARG;
  if (y_shared != nullptr && !aligned(y_shared, 16)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  return cuda_status(launch_combine(c.act_dtype, y_perm, inv_perm, topk_gate, y_shared, y, c.n,
                                    c.top_k, c.d, at<int>(ws, L.status), as_stream(stream)));
}

moe_status moe_forward_staged(const moe_config *cfg, const void *x, const moe_weights *w, void *y,
                              void *ws, size_t ws_bytes, void *stream, moe_stage_hook hook,
                              void *user) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  MOE_TRY(check_router_weights(c, w));
  MOE_TRY(check_expert_weights(c, w));
  if (!ok_ptr(x) || !ok_ptr(y)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  cudaStream_t s = as_stream(stream);
  int *status = at<int>(ws, L.status);
  const int P = c.n * c.top_k;
  int launched = 0;
  auto stage = [&](int id, int kernels) {
    if (hook) hook(id, launched, user);
    launched += kernels;
  };
  // the status word, the router's tile counts and the fused layer's counters
  MOE_TRY(cuda_status(cudaMemsetAsync(status, 0, cleared_bytes(L), s)));
  int32_t *topk_idx = at<int32_t>(ws, L.topk_idx);
  float *gates = at<float>(ws, L.topk_gate);
  int32_t *offsets = at<int32_t>(ws, L.offsets);
  int32_t *perm = at<int32_t>(ws, L.perm);
  int32_t *inv_perm = at<int32_t>(ws, L.inv_perm);
  const bool decode = decode_supported(c);
  const bool mx_tc = mx_tc_path(c);
  if (decode && decode_route_supported(c))
    return run_small_batch(c, x, w, nullptr, y, nullptr, nullptr, nullptr, ws, s, stage);
  // (the h buffer is free until the FFN: scratch for the router's partial
  // logits, then for a many-CTA sort)
  stage(MOE_STAGE_ROUTE, route_kernels(c, (size_t)P * c.d_ff * h_size(c), true));
  MOE_TRY(cuda_status(launch_route(c, x, w->Wg, w->router_bias, at<float>(ws, L.logits),
                                   at<float>(ws, L.h), (size_t)P * c.d_ff * h_size(c), topk_idx,
                                   gates, nullptr, status, s, at<int>(ws, L.route_count))));
  // (the sort, plus the copy of x rows into segment order: bf16/fp32 rows, or
  // the f16 copies the MXFP4 tensor-core path reads)
  stage(MOE_STAGE_DISPATCH,
        dispatch_kernels(P, c.n_experts, at<void>(ws, L.h), (size_t)P * c.d_ff * h_size(c)) +
            (decode ? 0 : 1));
  MOE_TRY(cuda_status(launch_dispatch(P, c.n_experts, topk_idx, at<int32_t>(ws, L.counts), offsets,
                                      perm, inv_perm, status, s, at<void>(ws, L.h),
                                      (size_t)P * c.d_ff * h_size(c))));
  if (decode) {
    // small batch: the FFN reads x rows through perm, no x_perm copy
    stage(MOE_STAGE_FFN_UP, 2);
    MOE_TRY(cuda_status(launch_decode_ffn(c, 0, x, perm, offsets, *w, at<void>(ws, L.h),
                                          at<void>(ws, L.y_perm), at<void>(ws, L.act16), status,
                                          s)));
    stage(MOE_STAGE_FFN_DOWN, 1);
    MOE_TRY(cuda_status(launch_decode_ffn(c, 1, x, perm, offsets, *w, at<void>(ws, L.h),
                                          at<void>(ws, L.y_perm), at<void>(ws, L.act16), status,
                                          s)));
  } else if (mx_tc) {
    // prefill over MXFP4 weights: the f16 staging gathers the rows itself
    MOE_TRY(run_mx_ffn(c, x, inv_perm, offsets, w, at<void>(ws, L.y_perm), ws, s, stage));
  } else {
    MOE_TRY(cuda_status(launch_scatter_rows(x, inv_perm, P, c.top_k, c.n,
                                            (int64_t)c.d * act_size(c), at<void>(ws, L.x_perm),
                                            status, s)));
    MOE_TRY(run_expert_ffn(c, at<void>(ws, L.x_perm), offsets, w, at<void>(ws, L.y_perm), ws, s,
                           stage));
  }
  const void *y_shared = nullptr;
  if (c.d_ff_shared) {
    stage(MOE_STAGE_SHARED, 2);
    MOE_TRY(run_shared_expert(c, x, w, ws, s));
    y_shared = at<void>(ws, L.y_shared);
  }
  stage(MOE_STAGE_COMBINE, 1);
  MOE_TRY(cuda_status(launch_combine(c.act_dtype, at<void>(ws, L.y_perm), inv_perm, gates, y_shared,
                                     y, c.n, c.top_k, c.d, status, s)));
  stage(MOE_STAGE_END, 0);
  return MOE_OK;
}

moe_status moe_forward(const moe_config *cfg, const void *x, const moe_weights *w, void *y,
                       void *ws, size_t ws_bytes, void *stream) {
  return moe_forward_staged(cfg, x, w, y, ws, ws_bytes, stream, nullptr, nullptr);
}

moe_status moe_classify_experts(const moe_config *cfg, const int32_t *topk_idx,
                                const int32_t *slot_of, int32_t n_slots, int32_t *state,
                                int32_t *miss_list, int32_t *counts, void *ws, size_t ws_bytes,
                                void *stream) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (!ok_ptr(topk_idx) || !ok_ptr(slot_of) || n_slots < 1 || !ok_ptr(state) ||
      !ok_ptr(miss_list) || !ok_ptr(counts))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  return cuda_status(launch_classify(c, topk_idx, slot_of, n_slots, state, miss_list, counts,
                                     at<int>(ws, L.status), as_stream(stream)));
}

moe_status moe_forward_pooled(const moe_config *cfg, const void *x, const moe_weights *w,
                              const moe_expert_pool *pool, void *y, int32_t *state,
                              int32_t *miss_list, int32_t *counts, void *ws, size_t ws_bytes,
                              void *stream) {
  return moe_forward_pooled_staged(cfg, x, w, pool, y, state, miss_list, counts, ws, ws_bytes,
                                   stream, nullptr, nullptr);
}

moe_status moe_forward_pooled_staged(const moe_config *cfg, const void *x, const moe_weights *w,
                                     const moe_expert_pool *pool, void *y, int32_t *state,
                                     int32_t *miss_list, int32_t *counts, void *ws,
                                     size_t ws_bytes, void *stream, moe_stage_hook hook,
                                     void *user) {
  MOE_TRY(check_config(cfg));
  const moe_config &c = *cfg;
  if (!decode_route_supported(c)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_router_weights(c, w));
  MOE_TRY(check_expert_weights(c, w));
  MOE_TRY(check_pool(c, pool));
  if (!ok_ptr(x) || !ok_ptr(y)) return MOE_ERR_INVALID_ARG;
  if ((state && !ok_ptr(state)) || (miss_list && !ok_ptr(miss_list)) || (counts && !ok_ptr(counts)))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  const Layout L = layout_of(c);
  cudaStream_t s = as_stream(stream);
  MOE_TRY(cuda_status(cudaMemsetAsync(at<int>(ws, L.status), 0, cleared_bytes(L), s)));
  int launched = 0;
  auto stage = [&](int id, int kernels) {
    if (hook) hook(id, launched, user);
    launched += kernels;
  };
  return run_small_batch(c, x, w, pool, y, state, miss_list, counts, ws, s, stage);
}

moe_status moe_status_check(const void *ws, void *stream, int32_t *detail) {
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t word[2] = {0, 0};
  if (cudaMemcpy(word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (detail) *detail = word[1];
  return static_cast<moe_status>(word[0]);
}

moe_status moe_status_clear(void *ws, void *stream) {
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, 2 * sizeof(int32_t), as_stream(stream)));
}

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: configuration not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime error";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX: index out of range on the device";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: device pipeline wait ran out";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE: MXFP4 block scale outside the exact range";
    case MOE_ERR_F16_RANGE:
      return "MOE_ERR_F16_RANGE: MXFP4 layer activation outside the f16 operand range";
  }
  return "unknown moe_status";
}

}  // extern "C"
