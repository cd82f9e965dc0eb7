// Host helpers shared by the TMA-fed kernels: tensor-map encoding through the
// driver entry point (no link-time dependency on libcuda) and the SM count.
#include <cudaTypedefs.h>

#include "launch.h"

namespace moe {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool tensor_maps_available() { return encode_fn() != nullptr; }

bool make_tensor_map(CUtensorMap *m, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                     int rank, const uint64_t *dims, const uint32_t *box,
                     CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr || rank < 1 || rank > 3) return false;
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t gbox[3], estr[3] = {1, 1, 1};
  uint64_t stride = dims[0] * (uint64_t)elem_bytes;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    gbox[i] = box[i];
    if (i + 1 < rank) {
      gstride[i] = stride;
      stride *= dims[i + 1];
    }
  }
  return fn(m, dtype, rank, const_cast<void *>(base), gdim, gstride, gbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace moe
