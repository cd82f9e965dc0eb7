// Small-batch routing in one launch: top-k selection and gates for every
// token, the stable dispatch arrays, and the f16 copies of the x rows that
// the small-batch expert FFN reads.
//
// "How Mixture of Experts Scales Model Parameters", sections "Top-K: several
// experts, added up by weight" (selection, renormalised gates) and "The
// forward pass: dispatch, then combine" (tokens regrouped per chosen expert).
// A cluster of CTAs selects for the n tokens (n * k <= 256 pairs, one token
// per warp), CTA 0 then derives the dispatch arrays, and every CTA converts a
// share of the x rows to f16 in token order, which the small-batch FFN reads
// through perm.
#include "common.cuh"
#include "launch.h"
#include "classify.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int DR_CLUSTER = 8;        // CTAs of the routing cluster
constexpr int DR_THREADS = 256;
constexpr int DR_WARPS = DR_THREADS / 32;
constexpr int DR_UNROLL = 4;          // x vectors in flight per thread

// Standalone classification from topk_idx: one CTA.
__global__ void __launch_bounds__(256)
classify_kernel(const int32_t *__restrict__ topk_idx, int P, int E,
                const int32_t *__restrict__ slot_of, int n_slots, int32_t *state,
                int32_t *miss_list, int32_t *counts, int *status) {
  __shared__ int s_cnt[256];
  for (int e = threadIdx.x; e < 256; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = topk_idx[p];
    if (e < 0 || e >= E) set_status(status, MOE_ERR_BAD_INDEX, p);
    else atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (threadIdx.x < 32)
    classify_warp(s_cnt, E, slot_of, n_slots, P, state, miss_list, counts, status);
}

// Every CTA converts its share of the x rows to f16 in token order
// (act16[t] = f16(x[t]), clamped to the f16 range).  The first cluster also
// routes: token t is selected by warp (t / DR_CLUSTER) % DR_WARPS of CTA
// t % DR_CLUSTER, the cluster meets on its barrier, and CTA 0 derives the
// dispatch arrays from the selections (and, given a slot table, classifies
// the selected experts against the resident pool).
struct PoolOut {
  const int32_t *slot_of;   // nullptr: no classification
  int n_slots;
  int32_t *state, *miss_list, *counts;
};

__global__ void __cluster_dims__(DR_CLUSTER, 1, 1) __launch_bounds__(DR_THREADS)
decode_route_kernel(const float *__restrict__ logits, int n, int E, int k, int gate_mode,
                    const __nv_bfloat16 *__restrict__ x, int d, int32_t *__restrict__ topk_idx,
                    float *__restrict__ topk_gate, int32_t *__restrict__ counts,
                    int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                    int32_t *__restrict__ inv_perm, uint16_t *__restrict__ act16, PoolOut pool,
                    int *status) {
  __shared__ int32_t s_idx[kDecodeMaxPairs];
  __shared__ int s_cnt[256];
  __shared__ int s_off[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = n * k;
  pdl_launch_dependents();
  pdl_wait();
  // (the x conversion below may record MOE_ERR_F16_RANGE while other CTAs
  // start, so CTAs can read different answers here: only the conversion
  // depends on it; the selection and the dispatch arrays are always built)
  const bool failed = status_failed(status);
  const bool router = blockIdx.x < DR_CLUSTER;

  if (router)
    for (int t = blockIdx.x + DR_CLUSTER * warp; t < n; t += DR_CLUSTER * DR_WARPS)
      select_topk_warp_shfl(logits + (size_t)t * E, E, k, gate_mode, lane,
                            topk_idx + (size_t)t * k, topk_gate + (size_t)t * k, nullptr);
  if (!failed) {
    const int nvec = n * (d / 8);
    const int stride = gridDim.x * DR_THREADS;
    const uint4 *xs = reinterpret_cast<const uint4 *>(x);
    uint4 *xd = reinterpret_cast<uint4 *>(act16);
    for (int base = blockIdx.x * DR_THREADS + threadIdx.x; base < nvec;
         base += DR_UNROLL * stride) {
      uint4 r[DR_UNROLL];
#pragma unroll
      for (int j = 0; j < DR_UNROLL; ++j)
        if (base + j * stride < nvec) r[j] = xs[base + j * stride];
#pragma unroll
      for (int j = 0; j < DR_UNROLL; ++j)
        if (base + j * stride < nvec)
          xd[base + j * stride] =
              bf16x8_to_f16x8_checked(r[j], status, (base + j * stride) / (d / 8));
    }
  }
  if (!router) return;
  for (int e = threadIdx.x; e < 256; e += DR_THREADS) s_cnt[e] = 0;
  // every thread of the cluster arrives (none has left): the selections are
  // visible to CTA 0 after the wait
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
  if (blockIdx.x != 0) return;

  for (int p = threadIdx.x; p < P; p += DR_THREADS) {
    int e = topk_idx[p];
    if (e < 0 || e >= E) {   // (the selection writes indices in range)
      set_status(status, MOE_ERR_BAD_INDEX, p);
      e = -1;
    }
    s_idx[p] = e;
    if (e >= 0) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (warp == 1 && pool.slot_of)
    classify_warp(s_cnt, E, pool.slot_of, pool.n_slots, P, pool.state, pool.miss_list,
                  pool.counts, status);
  if (warp == 0) {
    // exclusive prefix sum of the counts (lane l owns experts 8l .. 8l+7)
    int c[8], run = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = s_cnt[8 * lane + j];
      run += c[j];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int base = incl - run;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 8 * lane + j;
      s_off[e] = base;
      if (e < E) {
        counts[e] = c[j];
        offsets[e] = base;
      }
      base += c[j];
    }
    if (lane == 31) offsets[E] = incl;   // = P
    // stable positions: walk the pairs in order, 32 at a time; a pair's rank
    // among equal experts is the number of earlier pairs with that expert
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      const int e = p < P ? s_idx[p] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int pos = s_off[e] + __popc(peers & lanemask_lt());
        perm[pos] = p;
        inv_perm[p] = pos;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) s_off[e] += __popc(peers);
      __syncwarp();
    }
  }
}

}  // namespace

bool decode_route_supported(const moe_config &c) {
  return decode_supported(c) && c.n_experts <= 256 && c.d % 8 == 0 && c.d_ff_shared == 0;
}

cudaError_t launch_decode_route(const moe_config &c, const float *logits, const void *x,
                                int32_t *topk_idx, float *topk_gate, int32_t *counts,
                                int32_t *offsets, int32_t *perm, int32_t *inv_perm, void *act16,
                                int *status, cudaStream_t s, const moe_expert_pool *pool,
                                int32_t *state, int32_t *miss_list, int32_t *pool_counts) {
  // enough clusters that every thread converts at most DR_UNROLL x vectors
  const long vec = (long)c.n * (c.d / 8);
  const long per_cluster = (long)DR_CLUSTER * DR_THREADS * DR_UNROLL;
  long clusters = (vec + per_cluster - 1) / per_cluster;
  const long max_clusters = num_sms() / DR_CLUSTER;
  if (clusters > max_clusters) clusters = max_clusters;
  if (clusters < 1) clusters = 1;
  PoolOut po{};
  if (pool) {
    po.slot_of = pool->slot_of;
    po.n_slots = pool->n_slots;
    po.state = state;
    po.miss_list = miss_list;
    po.counts = pool_counts;
  }
  return launch_pdl(decode_route_kernel, dim3((unsigned)(clusters * DR_CLUSTER)), dim3(DR_THREADS),
                    0, s, logits, c.n, c.n_experts, c.top_k, (int)c.gate,
                    static_cast<const __nv_bfloat16 *>(x), c.d, topk_idx, topk_gate, counts,
                    offsets, perm, inv_perm, static_cast<uint16_t *>(act16), po, status);
}

cudaError_t launch_classify(const moe_config &c, const int32_t *topk_idx, const int32_t *slot_of,
                            int n_slots, int32_t *state, int32_t *miss_list, int32_t *counts,
                            int *status, cudaStream_t s) {
  classify_kernel<<<1, 256, 0, s>>>(topk_idx, c.n * c.top_k, c.n_experts, slot_of, n_slots, state,
                                    miss_list, counts, status);
  return cudaGetLastError();
}

}  // namespace moe
