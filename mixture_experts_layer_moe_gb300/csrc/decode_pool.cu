// Small-batch (decode) expert FFN reading resident experts from a slot pool
// (expert-slot indirection): the pool instantiations of decode_kernel.cuh,
// compiled apart from the plain ones.
#include "decode_kernel.cuh"

namespace moe {

cudaError_t launch_decode_ffn_pooled(const moe_config &c, int part, const void *act,
                                     const int32_t *perm, const int32_t *offsets,
                                     const moe_weights &w, void *h, void *y_perm, void *act16,
                                     int *status, cudaStream_t s, const moe_expert_pool &pool) {
  return run_decode_ffn<true, 0>(c, part, act, perm, offsets, w, h, y_perm, act16, status, s, &pool);
}

}  // namespace moe
