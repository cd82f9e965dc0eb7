// Dispatch: regroup the (token, slot) pairs into one contiguous segment per
// expert, in token order inside a segment, and gather the rows of x.
//
// "How Mixture of Experts Scales Model Parameters", section "The forward
// pass: dispatch, then combine": tokens are pulled into one matrix per chosen
// expert; an expert may receive no tokens at all.  Here the regrouping is a
// stable counting sort, so the result is unique and bit-exact:
//   counts[e], offsets[e] (exclusive prefix sum, offsets[E] = P),
//   perm[q]     = pair index t*k + j at segment position q,
//   inv_perm[p] = segment position of pair p.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int DP_THREADS = 1024;
constexpr int DP_WARPS = DP_THREADS / 32;
constexpr int DP_PREFETCH = 8;            // groups of 32 pair indices loaded ahead

// One CTA.  Warp w owns the pair range [w*chunk, (w+1)*chunk) and walks it in
// groups of 32 in increasing pair order, so a pair's rank inside its expert is
// (pairs of that expert in earlier warps) + (earlier groups of this warp) +
// (lower lanes of this group).  hist is [DP_WARPS][E] in shared memory.
__global__ void __launch_bounds__(DP_THREADS)
dispatch_kernel(const int32_t *__restrict__ topk_idx, int P, int E, int32_t *__restrict__ counts,
                int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                int32_t *__restrict__ inv_perm, int *status) {
  extern __shared__ int smem[];
  int *hist = smem;                       // [DP_WARPS][E]
  int *tot = smem + DP_WARPS * E;         // [E] -> exclusive offsets
  __shared__ int warp_sums[DP_WARPS];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = ((P + DP_WARPS - 1) / DP_WARPS + 31) & ~31;
  const int beg = min(P, w * chunk), end = min(P, beg + chunk);
  int *my = hist + w * E;

  for (int i = threadIdx.x; i < DP_WARPS * E; i += DP_THREADS) hist[i] = 0;
  __syncthreads();

  // pass 1: per-warp histogram (DP_PREFETCH groups of 32 loaded ahead)
  for (int base0 = beg; base0 < end; base0 += 32 * DP_PREFETCH) {
    int ev[DP_PREFETCH];
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      ev[u] = (p < end) ? topk_idx[p] : -1;
    }
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      int e = ev[u];
      const bool bad = (p < end) && (e < 0 || e >= E);
      if (bad) {
        set_status(status, MOE_ERR_BAD_INDEX, p);
        e = -1;
      }
      if (p >= end) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // per-expert totals and per-warp exclusive prefixes (warps in pair order)
  for (int e = threadIdx.x; e < E; e += DP_THREADS) {
    int run = 0;
    for (int ww = 0; ww < DP_WARPS; ++ww) {
      const int c = hist[ww * E + e];
      hist[ww * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();

  // exclusive scan of tot over experts (E <= 256 <= DP_THREADS)
  {
    const int e = threadIdx.x;
    int v = (e < E) ? tot[e] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      int s = warp_sums[lane];
      int si = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, si, o);
        if (lane >= o) si += t;
      }
      warp_sums[lane] = si - s;   // exclusive prefix of warp totals
    }
    __syncthreads();
    const int excl = incl - v + warp_sums[w];
    if (e < E) {
      counts[e] = v;
      offsets[e] = excl;
      tot[e] = excl;
    }
    if (e == E - 1) offsets[E] = excl + v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < DP_WARPS * E; i += DP_THREADS) hist[i] += tot[i % E];
  __syncthreads();

  // pass 2: scatter in pair order
  for (int base0 = beg; base0 < end; base0 += 32 * DP_PREFETCH) {
    int ev[DP_PREFETCH];
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      ev[u] = (p < end) ? topk_idx[p] : -1;
    }
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      int e = ev[u];
      if (e >= E || e < 0 || p >= end) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      int pos = 0;
      if (e >= 0) pos = my[e] + __popc(peers & lanemask_lt());
      __syncwarp();
      if (e >= 0) {
        perm[pos] = p;
        inv_perm[p] = pos;
        if (lane == __ffs(peers) - 1) my[e] += __popc(peers);
      } else if (p < end) {
        inv_perm[p] = -1;
      }
      __syncwarp();
    }
  }
}

// x_perm[q] = x[perm[q] / k], 16-byte vectors; one row per CTA iteration so
// the source row is resolved once per row.  perm entries outside [0, P) are
// reported and their row is zero-filled.
__global__ void __launch_bounds__(256)
gather_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ perm, int P, int k, int n,
              int vec_per_row, uint4 *__restrict__ x_perm, int *status) {
  for (int q = blockIdx.x; q < P; q += gridDim.x) {
    const int p = perm[q];
    const bool ok = p >= 0 && p < P && p / k < n;
    if (!ok && threadIdx.x == 0) set_status(status, MOE_ERR_BAD_INDEX, q);
    const uint4 *src = x + (int64_t)(ok ? p / k : 0) * vec_per_row;
    uint4 *dst = x_perm + (int64_t)q * vec_per_row;
    for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x)
      dst[v] = ok ? src[v] : make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

cudaError_t launch_dispatch(int P, int E, const int32_t *topk_idx, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv_perm, int *status,
                            cudaStream_t s) {
  const size_t smem = (size_t)(DP_WARPS + 1) * E * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(dispatch_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dispatch_kernel<<<1, DP_THREADS, smem, s>>>(topk_idx, P, E, counts, offsets, perm, inv_perm,
                                              status);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void *x, const int32_t *perm, int P, int k, int n,
                          int64_t row_bytes, void *x_perm, int *status, cudaStream_t s) {
  const int vpr = (int)(row_bytes / 16);
  int blocks = P < 152 * 16 ? P : 152 * 16;
  if (blocks < 1) blocks = 1;
  gather_kernel<<<blocks, 256, 0, s>>>((const uint4 *)x, perm, P, k, n, vpr, (uint4 *)x_perm,
                                       status);
  return cudaGetLastError();
}

}  // namespace moe
