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

// ------------------------------------------------------------------ many CTAs
// For large batches the same sort runs over one CTA per SM, each owning a
// contiguous range of pairs:
//   1. dispatch_hist_kernel: counts per expert in each range -> hist[g][e]
//   2. dispatch_scatter_kernel: every CTA sums hist over all ranges (totals,
//      hence counts and offsets) and over the ranges before its own (base),
//      then ranks its pairs as the single-CTA kernel does (earlier warps,
//      earlier groups, lower lanes) from offsets[e] + base[e]
// so every pair lands where the single-CTA kernel puts it.  The scatter
// kernel starts early (programmatic dependent launch) and builds its own
// per-warp counts while the first kernel finishes.

constexpr int DM_THREADS = 1024;
constexpr int DM_WARPS = DM_THREADS / 32;

// Per-warp counts of this CTA's range (hist: [DM_WARPS][E] in shared memory,
// zeroed by the caller); warp w takes the w-th of DM_WARPS equal sub-ranges,
// whole groups of 32 pairs in pair order.
__device__ __forceinline__ void range_hist(const int32_t *__restrict__ topk_idx, int beg, int end,
                                           int E, int *hist, int *status, bool report) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = end - beg;
  const int chunk = ((n + DM_WARPS - 1) / DM_WARPS + 31) & ~31;
  const int wb = min(end, beg + w * chunk), we = min(end, wb + chunk);
  int *my = hist + w * E;
  for (int base0 = wb; base0 < we; base0 += 32 * DP_PREFETCH) {
    int ev[DP_PREFETCH];
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      ev[u] = (p < we) ? topk_idx[p] : -1;
    }
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      int e = ev[u];
      if (p < we && (e < 0 || e >= E)) {
        if (report) set_status(status, MOE_ERR_BAD_INDEX, p);
        e = -1;
      }
      if (p >= we) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
    }
  }
}

__global__ void __launch_bounds__(DM_THREADS)
dispatch_hist_kernel(const int32_t *__restrict__ topk_idx, int P, int E, int range,
                     int32_t *__restrict__ hist_out, int *status) {
  extern __shared__ int smem[];
  pdl_launch_dependents();
  int *hist = smem;                                   // [DM_WARPS][E]
  for (int i = threadIdx.x; i < DM_WARPS * E; i += DM_THREADS) hist[i] = 0;
  __syncthreads();
  const int beg = min(P, (int)blockIdx.x * range), end = min(P, beg + range);
  range_hist(topk_idx, beg, end, E, hist, status, true);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += DM_THREADS) {
    int t = 0;
    for (int w = 0; w < DM_WARPS; ++w) t += hist[w * E + e];
    hist_out[(size_t)blockIdx.x * E + e] = t;
  }
}

__global__ void __launch_bounds__(DM_THREADS)
dispatch_scatter_kernel(const int32_t *__restrict__ topk_idx, int P, int E, int range, int G,
                        const int32_t *__restrict__ hist_g, int32_t *__restrict__ counts,
                        int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                        int32_t *__restrict__ inv_perm) {
  extern __shared__ int smem[];
  int *hist = smem;                                   // [DM_WARPS][E] -> running positions
  int *part_tot = hist + DM_WARPS * E;                // [DM_THREADS]: partial sums over ranges
  int *part_bef = part_tot + DM_THREADS;              // [DM_THREADS]: the same, earlier ranges
  int *start = part_bef + DM_THREADS;                 // [E]: offsets[e] + base of this range
  __shared__ int warp_sums[DM_WARPS];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < DM_WARPS * E; i += DM_THREADS) hist[i] = 0;
  __syncthreads();
  const int beg = min(P, (int)blockIdx.x * range), end = min(P, beg + range);
  range_hist(topk_idx, beg, end, E, hist, nullptr, false);

  // totals over all ranges and over the ranges before this one: thread t sums
  // expert t % E over its share of the ranges
  pdl_wait();
  {
    const int parts = DM_THREADS / E;
    const int t = threadIdx.x, e = t % E, part = t / E;
    int tot = 0, bef = 0;
    if (part < parts) {
      const int per = (G + parts - 1) / parts;
      const int g0 = part * per, g1 = min(G, g0 + per);
      for (int g = g0; g < g1; ++g) {
        const int c = hist_g[(size_t)g * E + e];
        tot += c;
        bef += (g < (int)blockIdx.x) ? c : 0;
      }
    }
    part_tot[t] = tot;
    part_bef[t] = bef;
  }
  __syncthreads();
  {
    // exclusive scan of the totals over experts (E <= 256 <= DM_THREADS)
    const int e = threadIdx.x, parts = DM_THREADS / E;
    int v = 0, bef = 0;
    if (e < E)
      for (int q = 0; q < parts; ++q) {
        v += part_tot[q * E + e];
        bef += part_bef[q * E + e];
      }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      const int sv = warp_sums[lane];
      int si = sv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, si, o);
        if (lane >= o) si += u;
      }
      warp_sums[lane] = si - sv;
    }
    __syncthreads();
    const int excl = incl - v + warp_sums[w];
    if (e < E) {
      start[e] = excl + bef;
      if (blockIdx.x == 0) {
        counts[e] = v;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + v;
      }
    }
  }
  __syncthreads();
  // per-warp start positions: the range's start plus earlier warps' pairs
  for (int e = threadIdx.x; e < E; e += DM_THREADS) {
    int run = start[e];
    for (int ww = 0; ww < DM_WARPS; ++ww) {
      const int c = hist[ww * E + e];
      hist[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int n = end - beg;
  const int chunk = ((n + DM_WARPS - 1) / DM_WARPS + 31) & ~31;
  const int wb = min(end, beg + w * chunk), we = min(end, wb + chunk);
  int *my = hist + w * E;
  for (int base0 = wb; base0 < we; base0 += 32 * DP_PREFETCH) {
    int ev[DP_PREFETCH];
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      ev[u] = (p < we) ? topk_idx[p] : -1;
    }
#pragma unroll
    for (int u = 0; u < DP_PREFETCH; ++u) {
      const int p = base0 + 32 * u + lane;
      int e = ev[u];
      if (e >= E || e < 0 || p >= we) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      int pos = 0;
      if (e >= 0) pos = my[e] + __popc(peers & lanemask_lt());
      __syncwarp();
      if (e >= 0) {
        perm[pos] = p;
        inv_perm[p] = pos;
        if (lane == __ffs(peers) - 1) my[e] += __popc(peers);
      } else if (p < we) {
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

// The same copy in token order: a CTA reads each x row once and writes it to
// the segment positions of the token's k pairs (inv_perm), so x is read from
// HBM once however large k is.  Pairs without a position (inv_perm < 0, an
// out-of-range expert id already reported by the sort) are skipped; their
// rows lie past every segment and are never read.
constexpr int SC_VEC = 4;                     // 16-byte vectors per thread in flight
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ inv_perm, int P,
                    int k, int n, int vec_per_row, uint4 *__restrict__ x_perm, int *status) {
  for (int t = blockIdx.x; t < n; t += gridDim.x) {
    const uint4 *src = x + (int64_t)t * vec_per_row;
    for (int v0 = 0; v0 < vec_per_row; v0 += SC_VEC * 256) {
      uint4 r[SC_VEC];
#pragma unroll
      for (int u = 0; u < SC_VEC; ++u) {
        const int v = v0 + threadIdx.x + u * 256;
        if (v < vec_per_row) r[u] = src[v];
      }
      for (int j = 0; j < k; ++j) {
        const int q = inv_perm[(int64_t)t * k + j];
        if (q < 0) continue;
        if (q >= P) {
          if (threadIdx.x == 0 && v0 == 0) set_status(status, MOE_ERR_BAD_INDEX, t * k + j);
          continue;
        }
        uint4 *dst = x_perm + (int64_t)q * vec_per_row;
#pragma unroll
        for (int u = 0; u < SC_VEC; ++u) {
          const int v = v0 + threadIdx.x + u * 256;
          if (v < vec_per_row) dst[v] = r[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_scatter_rows(const void *x, const int32_t *inv_perm, int P, int k, int n,
                                int64_t row_bytes, void *x_perm, int *status, cudaStream_t s) {
  if (P == 0 || n == 0) return cudaSuccess;
  const int vpr = (int)(row_bytes / 16);
  int blocks = n < 152 * 8 ? n : 152 * 8;
  if (blocks < 1) blocks = 1;
  scatter_rows_kernel<<<blocks, 256, 0, s>>>((const uint4 *)x, inv_perm, P, k, n, vpr,
                                             (uint4 *)x_perm, status);
  return cudaGetLastError();
}

// many CTAs once there is enough to share out and the scratch holds hist + base
static bool dispatch_many(int P, int E, const void *scratch, size_t scratch_bytes) {
  return P >= kDispatchManyMinPairs && scratch != nullptr &&
         scratch_bytes >= (size_t)num_sms() * E * sizeof(int32_t);
}

int dispatch_kernels(int P, int E, const void *scratch, size_t scratch_bytes) {
  return dispatch_many(P, E, scratch, scratch_bytes) ? 2 : 1;
}

cudaError_t launch_dispatch(int P, int E, const int32_t *topk_idx, int32_t *counts,
                            int32_t *offsets, int32_t *perm, int32_t *inv_perm, int *status,
                            cudaStream_t s, void *scratch, size_t scratch_bytes) {
  const int G = num_sms();
  if (dispatch_many(P, E, scratch, scratch_bytes)) {
    int32_t *hist = static_cast<int32_t *>(scratch);
    const int range = (P + G - 1) / G;
    const size_t smem1 = (size_t)DM_WARPS * E * sizeof(int);
    dispatch_hist_kernel<<<G, DM_THREADS, smem1, s>>>(topk_idx, P, E, range, hist, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem2 = smem1 + (2 * (size_t)DM_THREADS + E) * sizeof(int);
    return launch_pdl(dispatch_scatter_kernel, dim3((unsigned)G), dim3(DM_THREADS), smem2, s,
                      topk_idx, P, E, range, G, (const int32_t *)hist, counts, offsets, perm,
                      inv_perm);
  }
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
