// Internal helpers shared by the kernels of the MoE library (device side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------- status word
// The first 256 bytes of every workspace: int32 status, int32 detail, spare.
struct DevStatus {
  int status;
  int detail;
};

__device__ __forceinline__ void set_status(int *st, int code, int detail) {
  if (st == nullptr) return;
  if (atomicCAS(st, 0, code) == 0) {
    atomicExch(st + 1, detail);
  }
}

__device__ __forceinline__ bool status_failed(const int *st) {
  return st != nullptr && *reinterpret_cast<const volatile int *>(st) != 0;
}

// -------------------------------------------------------- f16 operand staging
// The MXFP4 paths feed the tensor cores f16 activations (E2M1 weights are
// exact in f16).  A bf16 or fp32 value converts exactly when it is zero or
// |v| lies in [2^-14, 65504]; a smaller magnitude rounds to an f16 subnormal
// (absolute error at most 2^-25).  |v| > 65504 or NaN cannot be represented:
// the value is clamped to +-65504 and MOE_ERR_F16_RANGE is recorded (detail:
// the row), so the layer's result is reported invalid instead of being wrong.
__device__ __forceinline__ uint16_t f16_bits_checked(float v, int *status, int row) {
  if (!(fabsf(v) <= 65504.f)) {
    set_status(status, MOE_ERR_F16_RANGE, row);
    v = v > 0.f ? 65504.f : -65504.f;
  }
  const __half h = __float2half_rn(v);
  return *reinterpret_cast<const uint16_t *>(&h);
}

// 8 bf16 values of row `row` -> f16 bit patterns, each through f16_bits_checked.
__device__ __forceinline__ uint4 bf16x8_to_f16x8_checked(uint4 raw, int *status, int row) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
    o[j] = (uint32_t)f16_bits_checked(lo, status, row) |
           ((uint32_t)f16_bits_checked(hi, status, row) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ----------------------------------------------------------- router dot product
// One 8-element piece of a bf16 router row against the same piece of a bf16 x
// row: a fresh fp32 partial, products added with fmaf in element order.  The
// small-batch router kernels add these partials piece by piece (lane l takes
// pieces l, l + 32, ...) and then combine the 32 lane sums with
// warp_sum_xor, so that every kernel that computes router logits this way
// gets the same bits.
__device__ __forceinline__ float bf16x8_dot(const uint4 &w, const uint4 &x) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  const uint32_t xx[4] = {x.x, x.y, x.z, x.w};
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    part = fmaf(__uint_as_float(ww[i] << 16), __uint_as_float(xx[i] << 16), part);
    part = fmaf(__uint_as_float(ww[i] & 0xffff0000u), __uint_as_float(xx[i] & 0xffff0000u), part);
  }
  return part;
}

// Sum over the warp by a butterfly (xor 16, 8, 4, 2, 1): every lane gets it.
__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------- programmatic dependent launch
// A kernel launched with launch_pdl may start while the previous kernel in the
// stream is still running: it calls pdl_launch_dependents() to let the next
// kernel start in turn, and pdl_wait() before touching any global memory that
// an earlier kernel writes or reads (the wait returns once the previous grid
// has completed and its writes are visible).  Both are no-ops in a kernel
// launched without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------- element types
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float *p) { return *p; }
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// ------------------------------------------------------------------- MXFP4
// E2M1 element (OCP MX v1.0): sign bit 3, exponent bits 2..1 (bias 1),
// mantissa bit 0; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_to_float(uint32_t code) {
  const uint32_t e = (code >> 1) & 3u;
  const uint32_t m = code & 1u;
  // normal: 2^(e-1) * (1 + m/2) -> fp32 bits: exponent e-1+127, mantissa m<<22
  // subnormal (e == 0): m * 0.5
  float mag = (e == 0) ? (m ? 0.5f : 0.0f) : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (code & 8u) ? -mag : mag;
}

// E8M0 scale: 2^(s-127); s = 0 is the fp32 subnormal 2^-127; s = 255 is NaN.
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
  if (s == 0u) return __uint_as_float(0x00400000u);
  if (s == 255u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float(s << 23);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace moe
