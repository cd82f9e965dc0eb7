// Top-k selection and gates of one token by one warp, shared by the router's
// selection kernel, the small-batch routing cluster and the one-launch
// small-batch layer.
//
// "How Mixture of Experts Scales Model Parameters", section "Routing: a router
// scores the experts, and the top one runs" (softmax over the router scores)
// and section "Top-K: several experts, added up by weight" (the K highest
// scores; weights renormalised over the chosen K).
#pragma once
#include <math.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Order-preserving 32-bit key of a score: a larger score has a larger key
// (-0 counts as +0; NaN is mapped to -inf before), and every score's key,
// -inf's included, is above 0.
__device__ __forceinline__ uint32_t score_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Lane l holds experts l, l+32, ... (E <= 256).  Selection works on the fp32
// logits: larger first, lower index on equal values; NaN scores rank below
// everything.  Gates:
//   top_prob: g_j = exp(l_j - m) / sum_e exp(l_e - m)
//   renorm:   g_j = exp(l_j - m) / sum_{chosen} exp(l_c - m)
// idx[j] and gate[j] (j < k) are written in rank order; probs (nullable) gets
// the E softmax probabilities.
//
// NV = ceil(E / 32) register slots per lane; l[i] is expert lane + 32 i (any
// value where that is >= E).  Each rank takes two warp reductions
// (redux.sync): the largest key among the lanes' best candidates, then the
// lowest expert index holding it.  The full softmax sum is formed only when
// the gates or probs need it (renorm gates divide by the chosen k's sum
// alone).
template <int NV>
__device__ __forceinline__ void select_topk_lanes(const float (&l)[NV], int E, int k,
                                                  int gate_mode, int lane, int32_t *idx,
                                                  float *gate, float *probs) {
  float v[NV];
  uint32_t key[NV];   // 0: not a candidate (past E, or already chosen)
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float t = (e < E) ? l[i] : -INFINITY;
    if (isnan(t)) t = -INFINITY;
    v[i] = t;
    key[i] = (e < E) ? score_key(t) : 0u;
  }
  // the lane's best candidate: the largest key, the lowest index on a tie
  uint32_t bk, be;
  auto lane_best = [&]() {
    bk = 0u;
    be = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (key[i] > bk) {
        bk = key[i];
        be = (uint32_t)(lane + 32 * i);
      }
  };
  lane_best();
  uint32_t top = __reduce_max_sync(0xffffffffu, bk);
  const float mx = key_score(top);   // the largest score
  float sum = 0.f;
  if (gate_mode != MOE_GATE_RENORM || probs != nullptr) {
    float ex[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      ex[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
      sum += ex[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (probs) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E) probs[e] = ex[i] / sum;
      }
    }
  }
  float gx[NV];   // rank j's exponential, kept by lane j % 32 at [j / 32] (k <= E)
#pragma unroll
  for (int i = 0; i < NV; ++i) gx[i] = 0.f;
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    if (j > 0) {
      lane_best();
      top = __reduce_max_sync(0xffffffffu, bk);
    }
    const uint32_t w = __reduce_min_sync(0xffffffffu, bk == top ? be : 0xffffffffu);
    if ((int)(w & 31u) == lane) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (i == (int)(w >> 5)) key[i] = 0u;
    }
    const float exj = expf(key_score(top) - mx);
    sel_sum += exj;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (j == lane + 32 * i) gx[i] = exj;
    if (lane == 0) idx[j] = (int32_t)w;
  }
  const float denom = (gate_mode == MOE_GATE_RENORM) ? sel_sum : sum;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int j = lane + 32 * i;
    if (j < k) gate[j] = gx[i] / denom;
  }
}

// The same selection with the argmax as a shuffle tree over (value, index)
// pairs and the chosen exponentials in an indexed array (local memory): the
// form the small-batch routing cluster keeps.  Same results bit for bit.  In
// that kernel the redux form above, though faster on its own, made chains of
// back-to-back layers slower (8 us per layer at 32-64 tokens, graph replay,
// same box), so the cluster stays on this one.
template <int NV>
__device__ __forceinline__ void select_topk_lanes_shfl(const float (&l)[NV], int E, int k,
                                                  int gate_mode, int lane, int32_t *idx,
                                                  float *gate, float *probs) {
  float v[NV];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float t = (e < E) ? l[i] : -INFINITY;
    if (isnan(t)) t = -INFINITY;
    v[i] = t;
    mx = fmaxf(mx, t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  if (gate_mode != MOE_GATE_RENORM || probs != nullptr) {
    float ex[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      ex[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
      sum += ex[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (probs) {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E) probs[e] = ex[i] / sum;
      }
    }
  }
  unsigned taken = 0;
  float sel_ex[NV];   // slot j kept by lane j % 32 at [j / 32] (k <= E)
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        if (v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    const float exj = expf(bv - mx);
    sel_sum += exj;
    if ((j & 31) == lane) sel_ex[j >> 5] = exj;
    if (lane == 0) idx[j] = bi;
  }
  const float denom = (gate_mode == MOE_GATE_RENORM) ? sel_sum : sum;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int j = lane + 32 * i;
    if (j < k) gate[j] = sel_ex[i] / denom;
  }
}

// The same reading the E logits from memory (l[e]).
template <int NV>
__device__ __forceinline__ void select_topk_mem(const float *__restrict__ l, int E, int k,
                                                int gate_mode, int lane, int32_t *idx,
                                                float *gate, float *probs) {
  float v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? l[e] : -INFINITY;
  }
  select_topk_lanes<NV>(v, E, k, gate_mode, lane, idx, gate, probs);
}
__device__ __forceinline__ void select_topk_warp(const float *__restrict__ l, int E, int k,
                                                 int gate_mode, int lane, int32_t *idx,
                                                 float *gate, float *probs) {
  if (E <= 128) select_topk_mem<4>(l, E, k, gate_mode, lane, idx, gate, probs);
  else select_topk_mem<8>(l, E, k, gate_mode, lane, idx, gate, probs);
}
__device__ __forceinline__ void select_topk_warp_shfl(const float *__restrict__ l, int E, int k,
                                                      int gate_mode, int lane, int32_t *idx,
                                                      float *gate, float *probs) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? l[e] : -INFINITY;
  }
  select_topk_lanes_shfl<8>(v, E, k, gate_mode, lane, idx, gate, probs);
}

}  // namespace moe
