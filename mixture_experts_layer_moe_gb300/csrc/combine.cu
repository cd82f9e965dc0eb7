// Combine: gate scaling fused with the un-permute back to token order.
//
// "How Mixture of Experts Scales Model Parameters", section "The forward
// pass: dispatch, then combine": each expert's output rows are multiplied by
// the probability the token was routed with, and combine puts the weighted
// rows back in the tokens' original order.  With top-K ("Top-K: several
// experts, added up by weight") the K weighted outputs of a token are added.
//   y[t] = sum_{j<k} g[t][j] * y_perm[inv_perm[t*k + j]]  (+ y_shared[t])
// fp32 accumulation in slot order, then one rounding to the output type.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *f);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float *f);
template <>
__device__ __forceinline__ uint4 pack16<float>(const float *f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Thread = one 16-byte vector of an output row.  The slots are taken eight at
// a time: their indices and gates, then their rows, are all loaded before the
// sum, which runs in slot order.
constexpr int CB_SLOTS = 8;

template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ inv_perm,
               const float *__restrict__ gates, const uint4 *__restrict__ y_shared,
               uint4 *__restrict__ y, int n, int k, int vec_per_row, int *status) {
  constexpr int V = Vec16<T>::N;
  pdl_launch_dependents();
  pdl_wait();
  const int P = n * k;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)n * vec_per_row;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / vec_per_row);
    const int v = (int)(i - (int64_t)t * vec_per_row);
    float acc[V];
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] = 0.f;
    for (int j0 = 0; j0 < k; j0 += CB_SLOTS) {
      int q[CB_SLOTS];
      float g[CB_SLOTS];
      uint4 r[CB_SLOTS];
#pragma unroll
      for (int u = 0; u < CB_SLOTS; ++u) {
        q[u] = -1;
        if (j0 + u < k) {
          q[u] = inv_perm[(int64_t)t * k + j0 + u];
          g[u] = gates[(int64_t)t * k + j0 + u];
        }
      }
#pragma unroll
      for (int u = 0; u < CB_SLOTS; ++u)
        if (q[u] >= 0 && q[u] < P) r[u] = y_perm[(int64_t)q[u] * vec_per_row + v];
#pragma unroll
      for (int u = 0; u < CB_SLOTS; ++u) {
        if (j0 + u >= k) continue;
        if (q[u] < 0 || q[u] >= P) {
          if (v == 0) set_status(status, MOE_ERR_BAD_INDEX, t * k + j0 + u);
          continue;
        }
        float f[V];
        unpack16<T>(r[u], f);
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] = fmaf(g[u], f[c], acc[c]);
      }
    }
    if (y_shared) {
      float f[V];
      unpack16<T>(y_shared[i], f);
#pragma unroll
      for (int c = 0; c < V; ++c) acc[c] += f[c];
    }
    y[i] = pack16<T>(acc);
  }
}

// Row-oriented variant: CTA (t, c) takes vectors [c * 256 * VB, ...) of token
// t's row.  The token's k inverse indices and gates are loaded once into
// shared memory; a thread then loads its VB vectors of the rows CR_SLOTS
// slots at a time before summing them in slot order, as above.
constexpr int CR_SLOTS = 4;
template <typename T, int VB>
__global__ void __launch_bounds__(256)
combine_rows_kernel(const uint4 *__restrict__ y_perm, const int32_t *__restrict__ inv_perm,
                    const float *__restrict__ gates, const uint4 *__restrict__ y_shared,
                    uint4 *__restrict__ y, int n, int k, int vec_per_row, int *status) {
  constexpr int V = Vec16<T>::N;
  __shared__ int s_q[256];
  __shared__ float s_g[256];
  pdl_launch_dependents();
  pdl_wait();
  const int P = n * k;
  const int t = blockIdx.x;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    int q = inv_perm[(int64_t)t * k + j];
    if (q < 0 || q >= P) {
      if (blockIdx.y == 0) set_status(status, MOE_ERR_BAD_INDEX, t * k + j);
      q = -1;
    }
    s_q[j] = q;
    s_g[j] = gates[(int64_t)t * k + j];
  }
  __syncthreads();
  const int v0 = blockIdx.y * 256 * VB + threadIdx.x;
  float acc[VB][V];
#pragma unroll
  for (int b = 0; b < VB; ++b)
#pragma unroll
    for (int c = 0; c < V; ++c) acc[b][c] = 0.f;
  for (int j0 = 0; j0 < k; j0 += CR_SLOTS) {
    uint4 r[CR_SLOTS][VB];
#pragma unroll
    for (int u = 0; u < CR_SLOTS; ++u) {
      const int q = (j0 + u < k) ? s_q[j0 + u] : -1;
#pragma unroll
      for (int b = 0; b < VB; ++b)
        if (q >= 0 && v0 + b * 256 < vec_per_row)
          r[u][b] = y_perm[(int64_t)q * vec_per_row + v0 + b * 256];
    }
#pragma unroll
    for (int u = 0; u < CR_SLOTS; ++u) {
      if (j0 + u >= k || s_q[j0 + u] < 0) continue;
      const float g = s_g[j0 + u];
#pragma unroll
      for (int b = 0; b < VB; ++b) {
        if (v0 + b * 256 < vec_per_row) {
          float f[V];
          unpack16<T>(r[u][b], f);
#pragma unroll
          for (int c = 0; c < V; ++c) acc[b][c] = fmaf(g, f[c], acc[b][c]);
        }
      }
    }
  }
#pragma unroll
  for (int b = 0; b < VB; ++b) {
    const int v = v0 + b * 256;
    if (v < vec_per_row) {
      const int64_t i = (int64_t)t * vec_per_row + v;
      if (y_shared) {
        float f[V];
        unpack16<T>(y_shared[i], f);
#pragma unroll
        for (int c = 0; c < V; ++c) acc[b][c] += f[c];
      }
      y[i] = pack16<T>(acc[b]);
    }
  }
}

template <typename T>
cudaError_t launch_rows(const void *y_perm, const int32_t *inv_perm, const float *gates,
                        const void *y_shared, void *y, int n, int k, int vpr, int *status,
                        cudaStream_t s) {
  // two vectors per thread where that still leaves two CTAs per SM
  const bool two = (int64_t)n * ((vpr + 511) / 512) >= 2 * 152;
  if (two)
    return launch_pdl(combine_rows_kernel<T, 2>, dim3((unsigned)n, (unsigned)((vpr + 511) / 512)),
                      dim3(256), 0, s, (const uint4 *)y_perm, inv_perm, gates,
                      (const uint4 *)y_shared, (uint4 *)y, n, k, vpr, status);
  return launch_pdl(combine_rows_kernel<T, 1>, dim3((unsigned)n, (unsigned)((vpr + 255) / 256)),
                    dim3(256), 0, s, (const uint4 *)y_perm, inv_perm, gates,
                    (const uint4 *)y_shared, (uint4 *)y, n, k, vpr, status);
}

}  // namespace

cudaError_t launch_combine(int act_dtype, const void *y_perm, const int32_t *inv_perm,
                           const float *gates, const void *y_shared, void *y, int n, int k,
                           int d, int *status, cudaStream_t s) {
  const int esz = act_dtype == MOE_F32 ? 4 : 2;
  const int vpr = d * esz / 16;
  // row-oriented once there are rows enough to fill the GPU (k <= 256: the
  // indices fit shared memory)
  if (n >= 2 * 152 && k <= 256) {
    if (act_dtype == MOE_F32)
      return launch_rows<float>(y_perm, inv_perm, gates, y_shared, y, n, k, vpr, status, s);
    return launch_rows<__nv_bfloat16>(y_perm, inv_perm, gates, y_shared, y, n, k, vpr, status, s);
  }
  const int64_t total = (int64_t)n * vpr;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  if (act_dtype == MOE_F32)
    return launch_pdl(combine_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s,
                      (const uint4 *)y_perm, inv_perm, gates, (const uint4 *)y_shared, (uint4 *)y,
                      n, k, vpr, status);
  return launch_pdl(combine_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, s,
                    (const uint4 *)y_perm, inv_perm, gates, (const uint4 *)y_shared, (uint4 *)y, n,
                    k, vpr, status);
}

}  // namespace moe
