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
//
// NV = ceil(E / 32) register slots per lane; l[i] is expert lane + 32 i (any
// value where that is >= E).  The full softmax sum is formed only when the
// gates or probs need it (renorm gates divide by the chosen k's sum alone).
// COMPACT keeps the chosen exponentials in an indexed array (local memory)
// rather than unrolled registers: fewer registers for kernels that must stay
// small, the same values.
template <int NV, bool COMPACT = false>
__device__ __forceinline__ void select_topk_lanes(const float (&l)[NV], int E, int k,
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
    if (COMPACT) {
      if ((j & 31) == lane) sel_ex[j >> 5] = exj;
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (j == lane + 32 * i) sel_ex[i] = exj;
    }
    if (lane == 0) idx[j] = bi;
  }
  const float denom = (gate_mode == MOE_GATE_RENORM) ? sel_sum : sum;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int j = lane + 32 * i;
    if (j < k) gate[j] = sel_ex[i] / denom;
  }
}

// The same reading the E logits from memory (l[e]), in the compact form for
// any E <= 256 (the small-batch routing cluster, whose register count decides
// how soon the next kernel's CTAs fit beside it).
__device__ __forceinline__ void select_topk_warp(const float *__restrict__ l, int E, int k,
                                                 int gate_mode, int lane, int32_t *idx,
                                                 float *gate, float *probs) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? l[e] : -INFINITY;
  }
  select_topk_lanes<8, true>(v, E, k, gate_mode, lane, idx, gate, probs);
}

}  // namespace moe
