// moe_route_noalloc: the router for callers that cannot allocate device memory.
//
// moe_route needs a caller-allocated workspace because the router keeps its
// fp32 logits (n x E) in scratch memory between its two kernels.  Some callers
// cannot provide one: code that runs while a CUDA graph is being captured in
// a framework whose allocator is not capture-safe, plugins that are handed
// only their input and output tensors by a host runtime that owns all device
// memory, and fixed-arena embedded runtimes whose memory is budgeted before
// the model runs.  This entry point takes only inputs and outputs and keeps
// the logits in a file-scope device array instead.
//
// That array is a static __device__ object, so every GPU that loads this
// library holds it (16 MiB) until the process exits.  Its host-side name is
// only a stand-in, not a device address, so the address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made while it is current.  That first call should come before
// any stream capture begins.  All calls share the one array and it keeps the
// last call's contents; calls that overlap on the GPU (different streams, or
// several threads) race on it and must be serialised by the caller.  Nothing
// in it has to start at zero: each call writes every logit it reads.
#include <mutex>

#include "launch.h"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kMaxLogits = (size_t)4 << 20;   // n * E <= 4,194,304 fp32 values (16 MiB)
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_route_logits[kMaxLogits];

std::mutex g_lock;
float *g_logits_ptr[kMaxDevices] = {};

// Device address of g_route_logits on the current device (looked up once).
moe_status logits_scratch(float **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_logits_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_logits) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_logits_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_logits_ptr[dev];
  return MOE_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const moe_config *cfg, const void *x, const moe_weights *w,
                                        int32_t *topk_idx, float *topk_gate, float *probs,
                                        void *stream) {
  using namespace moe;
  size_t ws_bytes = 0;   // host-only shape check shared with every other entry point
  const moe_status st = moe_workspace_size(cfg, &ws_bytes);
  if (st != MOE_OK) return st;
  if (w == nullptr || !aligned16(w->Wg)) return MOE_ERR_INVALID_ARG;
  if (w->router_bias != nullptr && (reinterpret_cast<uintptr_t>(w->router_bias) & 3))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_gate)) return MOE_ERR_INVALID_ARG;
  if (probs != nullptr && (reinterpret_cast<uintptr_t>(probs) & 15)) return MOE_ERR_INVALID_ARG;
  if ((size_t)cfg->n * (size_t)cfg->n_experts > kMaxLogits) return MOE_ERR_WORKSPACE;
  float *logits = nullptr;
  const moe_status ss = logits_scratch(&logits);
  if (ss != MOE_OK) return ss;
  const cudaError_t e =
      launch_route(*cfg, x, w->Wg, w->router_bias, logits, nullptr, 0, topk_idx, topk_gate, probs,
                   nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
