// Small-batch (decode) expert FFN over NVFP4 weights (E2M1 codes, an E4M3
// scale per 16 elements, one fp32 scale per matrix): the NVFP4 instantiations
// of decode_kernel.cuh, compiled apart from the MXFP4 ones.
#include "decode_kernel.cuh"

namespace moe {

cudaError_t launch_decode_ffn_nvfp4(const moe_config &c, int part, const void *act,
                                    const int32_t *perm, const int32_t *offsets,
                                    const moe_weights &w, void *h, void *y_perm, void *act16,
                                    int *status, cudaStream_t s) {
  return run_decode_ffn<false, 1>(c, part, act, perm, offsets, w, h, y_perm, act16, status, s,
                                  nullptr);
}

}  // namespace moe
