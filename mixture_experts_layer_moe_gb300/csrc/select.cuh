// Top-k selection and gates of one token by one warp, shared by the router's
// selection kernel and the fused small-batch routing kernel.
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

// Lane l holds experts l, l+32, ... (E <= 256).  Selection works on the fp32
// logits: larger first, lower index on equal values; NaN scores rank below
// everything.  Gates:
//   top_prob: g_j = exp(l_j - m) / sum_e exp(l_e - m)
//   renorm:   g_j = exp(l_j - m) / sum_{chosen} exp(l_c - m)
// idx[j] and gate[j] (j < k) are written in rank order; probs (nullable) gets
// the E softmax probabilities.
__device__ __forceinline__ void select_topk_warp(const float *__restrict__ l, int E, int k,
                                                 int gate_mode, int lane, int32_t *idx,
                                                 float *gate, float *probs) {
  float v[8];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float t = (e < E) ? l[e] : -INFINITY;
    if (isnan(t)) t = -INFINITY;
    v[i] = t;
    mx = fmaxf(mx, t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  float ex[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ex[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.f;
    sum += ex[i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (probs) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) probs[e] = ex[i] / sum;
    }
  }
  unsigned taken = 0;
  float sel_ex[8];   // slot j kept by lane j % 32 at [j / 32]
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
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
  for (int i = 0; i < 8; ++i) {
    const int j = lane + 32 * i;
    if (j < k) gate[j] = sel_ex[i] / denom;
  }
}

}  // namespace moe
