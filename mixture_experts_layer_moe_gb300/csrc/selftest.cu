// Diagnostics: the bounded device wait every pipeline kernel uses, run
// against an mbarrier that nothing arrives on, so that a test can check that
// such a wait ends by itself and reports MOE_ERR_TIMEOUT through the status
// word, with the context still usable afterwards.  The word is a workspace's,
// or (ws == NULL) the one moe_route_noalloc reports through.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, int *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncwarp();
  // nothing arrives: the wait gives up after limit_ns and raises the flag
  const bool ok = tc::mbar_wait(&bar, 0, &abort_flag, limit_ns);
  if (__all_sync(0xffffffffu, !ok) && threadIdx.x == 0) set_status(status, MOE_ERR_TIMEOUT, -1);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_wait_timeout(void *ws, uint64_t limit_ns, void *stream) {
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return MOE_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;
  int *word = static_cast<int *>(ws);
  if (word == nullptr) {
    const moe_status st = moe::noalloc_status_word(&word);
    if (st != MOE_OK) return st;
  }
  moe::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, word);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
