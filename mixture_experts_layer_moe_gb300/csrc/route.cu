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

namespace moe {
namespace {

constexpr int RT_M = 64, RT_E = 64, RT_K = 32, RT_THREADS = 256;

// logits[t][e] = sum_i x[t][i] * Wg[e][i], each thread accumulating its 4x4
// outputs sequentially in i with fp32 FMA, then + bias[e].
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
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
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

// One warp per token.  Lane l holds experts l, l+32, ... (E <= 256).
// Selection works on the fp32 logits: larger first, lower index on equal
// values; NaN scores rank below everything.  Gates:
//   top_prob: g_j = exp(l_j - m) / sum_e exp(l_e - m)
//   renorm:   g_j = exp(l_j - m) / sum_{chosen} exp(l_c - m)
__global__ void __launch_bounds__(256)
route_select_kernel(const float *__restrict__ logits, int n, int E, int k, int gate_mode,
                    int32_t *__restrict__ topk_idx, float *__restrict__ topk_gate,
                    float *__restrict__ probs) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= n) return;
  const float *l = logits + (size_t)warp * E;
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
      if (e < E) probs[(size_t)warp * E + e] = ex[i] / sum;
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
    if (lane == 0) topk_idx[(size_t)warp * k + j] = bi;
  }
  const float denom = (gate_mode == MOE_GATE_RENORM) ? sel_sum : sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = lane + 32 * i;
    if (j < k) topk_gate[(size_t)warp * k + j] = sel_ex[i] / denom;
  }
}

}  // namespace

cudaError_t launch_route(const moe_config &c, const void *x, const void *Wg, const float *bias,
                         float *logits, int32_t *topk_idx, float *topk_gate, float *probs,
                         int *status, cudaStream_t s) {
  (void)status;
  dim3 grid((c.n + RT_M - 1) / RT_M, (c.n_experts + RT_E - 1) / RT_E);
  if (c.act_dtype == MOE_F32)
    route_logits_kernel<float><<<grid, RT_THREADS, 0, s>>>(
        (const float *)x, (const float *)Wg, bias, logits, c.n, c.d, c.n_experts);
  else
    route_logits_kernel<__nv_bfloat16><<<grid, RT_THREADS, 0, s>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)Wg, bias, logits, c.n, c.d,
        c.n_experts);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int warps_per_block = 8;
  route_select_kernel<<<(c.n + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0,
                        s>>>(logits, c.n, c.n_experts, c.top_k, c.gate, topk_idx, topk_gate,
                             probs);
  return cudaGetLastError();
}

}  // namespace moe
