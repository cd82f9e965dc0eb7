// Hit/miss classification of the selected experts against a resident slot
// pool, shared by the small-batch routing kernel and the fused layer kernel.
#pragma once

#include "common.cuh"

namespace moe {

// Hit/miss classification by one warp from the per-expert selection counts
// (FreeToken paper summary post, section "3. Decode: Exploit Expert
// Locality": a selected expert in GPU memory is a hit, otherwise a miss).
// Experts are visited in ascending order, 32 at a time, so the miss list is
// sorted.  A slot outside [-1, n_slots) is reported and counted as a miss.
__device__ __forceinline__ void classify_warp(const int *cnt, int E,
                                              const int32_t *__restrict__ slot_of, int n_slots,
                                              int lookups, int32_t *state, int32_t *miss_list,
                                              int32_t *counts, int *status) {
  const int lane = threadIdx.x & 31;
  int misses = 0, selected = 0, resident = 0, served = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const int c = e < E ? cnt[e] : 0;
    int slot = -1;
    if (e < E) {
      slot = slot_of[e];
      if (slot < -1 || slot >= n_slots) {
        set_status(status, MOE_ERR_BAD_INDEX, e);
        slot = -1;
      }
    }
    const bool chosen = c > 0, hit = chosen && slot >= 0, miss = chosen && slot < 0;
    if (state && e < E) state[e] = chosen ? (hit ? 1 : 0) : -1;
    const unsigned mm = __ballot_sync(0xffffffffu, miss);
    if (miss && miss_list) miss_list[misses + __popc(mm & lanemask_lt())] = e;
    misses += __popc(mm);
    selected += __popc(__ballot_sync(0xffffffffu, chosen));
    resident += __popc(__ballot_sync(0xffffffffu, hit));
    served += hit ? c : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) served += __shfl_xor_sync(0xffffffffu, served, o);
  if (miss_list)
    for (int i = misses + lane; i < E; i += 32) miss_list[i] = -1;
  if (counts && lane == 0) {
    counts[MOE_POOL_SELECTED] = selected;
    counts[MOE_POOL_RESIDENT] = resident;
    counts[MOE_POOL_LOOKUPS] = lookups;
    counts[MOE_POOL_SERVED] = served;
  }
}

}  // namespace moe
