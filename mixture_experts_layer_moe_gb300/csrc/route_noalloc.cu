// moe_route_noalloc: the router for callers that cannot allocate device memory.
//
// moe_route needs a caller-allocated workspace because the router keeps its
// fp32 logits (n x E) in scratch memory between its two kernels.  Some callers
// cannot provide one: code that runs while a CUDA graph is being captured in
// a framework whose allocator is not capture-safe, plugins that are handed
// only their input and output tensors by a host runtime that owns all device
// memory, and fixed-arena embedded runtimes whose memory is budgeted before
// the model runs.  This entry point takes only inputs and outputs and keeps
// the logits in a file-scope device array instead, next to a status word of
// its own (the workspace's status word has no home here).
//
// Both arrays are static __device__ objects, so every GPU that loads this
// library holds them (16 MiB + 16 bytes) until the process exits.  Their
// host-side names are only stand-ins, not device addresses, so the addresses
// are looked up with cudaGetSymbolAddress once per device and CUDA context,
// with that device current, on the first call made in that context.  That
// first call should come before any stream capture begins.  All calls share
// the one pair of arrays and they keep the last call's contents; calls that
// overlap on the GPU (different streams, or several threads) race on them and
// must be serialised by the caller.  Each call clears the status word on its
// stream before its kernels run; the logits need no clearing (each call
// writes every logit it reads).
#include <cudaTypedefs.h>

#include <mutex>

#include "launch.h"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kMaxLogits = (size_t)4 << 20;   // n * E <= 4,194,304 fp32 values (16 MiB)
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_route_logits[kMaxLogits];
__device__ __align__(16) int g_route_status[4];   // status, detail, spare

struct Scratch {
  CUcontext ctx;   // the context the addresses belong to
  float *logits;
  int *status;
};

std::mutex g_lock;
Scratch g_scratch[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 ctx_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }
  return fn;
}

// Device addresses of the two arrays in the current device's current context
// (looked up again when the context changed, e.g. after cudaDeviceReset).
moe_status scratch_of_current(Scratch *out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  auto get_ctx = ctx_fn();
  CUcontext ctx = nullptr;
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  if (ctx == nullptr) {
    // no context current yet: a symbol lookup makes the device's primary one current
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_status) != cudaSuccess) return MOE_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> guard(g_lock);
  Scratch &s = g_scratch[dev];
  if (s.ctx != ctx || s.logits == nullptr || s.status == nullptr) {
    void *pl = nullptr, *ps = nullptr;
    if (cudaGetSymbolAddress(&pl, g_route_logits) != cudaSuccess || pl == nullptr)
      return MOE_ERR_CUDA;
    if (cudaGetSymbolAddress(&ps, g_route_status) != cudaSuccess || ps == nullptr)
      return MOE_ERR_CUDA;
    s.ctx = ctx;
    s.logits = static_cast<float *>(pl);
    s.status = static_cast<int *>(ps);
  }
  *out = s;
  return MOE_OK;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

// The status word of moe_route_noalloc on the current device (diagnostics).
moe_status noalloc_status_word(int **out) {
  Scratch s{};
  const moe_status st = scratch_of_current(&s);
  if (st == MOE_OK) *out = s.status;
  return st;
}

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
  Scratch s{};
  const moe_status ss = scratch_of_current(&s);
  if (ss != MOE_OK) return ss;
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(s.status, 0, 2 * sizeof(int), strm) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t e = launch_route(*cfg, x, w->Wg, w->router_bias, s.logits, nullptr, 0,
                                     topk_idx, topk_gate, probs, s.status, strm);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_route_noalloc_status(void *stream, int32_t *detail) {
  using namespace moe;
  int *word = nullptr;
  const moe_status st = noalloc_status_word(&word);
  if (st != MOE_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v[2] = {0, 0};
  if (cudaMemcpy(v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = v[1];
  return static_cast<moe_status>(v[0]);
}
