// Small-batch (decode) expert FFN over MXFP4 weights: the launches without a
// resident pool, and the f16 staging of activation rows.  The kernel itself
// is in decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace moe {
namespace {

// Expert-ordered activation rows as f16: dst[q] = src[perm[q] / top_k] (perm
// given) or src[q] (f16_bits_checked: values beyond the f16 range are reported).
__global__ void rows_to_f16_kernel(const __nv_bfloat16 *__restrict__ src,
                                   const int32_t *__restrict__ perm, int top_k, int P, int K,
                                   uint16_t *__restrict__ dst, int *status) {
  const int vpr = K / 8;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < P * vpr; i += gridDim.x * blockDim.x) {
    const int q = i / vpr, v = i - q * vpr;
    int row = q;
    if (perm) {
      const int p = perm[q];
      row = (p >= 0 && p < P) ? p / top_k : -1;
      if (row < 0 && v == 0) set_status(status, MOE_ERR_BAD_INDEX, q);
    }
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (row >= 0) raw = *reinterpret_cast<const uint4 *>(src + (size_t)row * K + v * 8);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
      o[j] = (uint32_t)f16_bits_checked(lo, status, q) |
             ((uint32_t)f16_bits_checked(hi, status, q) << 16);
    }
    *reinterpret_cast<uint4 *>(dst + (size_t)q * K + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The same staging in token order: dst[inv_perm[t*k + j]] = f16(src[t]), each
// x row read and converted once (pairs with inv_perm < 0 skipped, >= P
// reported).
constexpr int RF16_VEC = 4;                   // 16-byte vectors per thread in flight
__global__ void __launch_bounds__(256)
rows_to_f16_scatter_kernel(const __nv_bfloat16 *__restrict__ src,
                           const int32_t *__restrict__ inv_perm, int top_k, int n, int P, int K,
                           uint16_t *__restrict__ dst, int *status) {
  const int vpr = K / 8;
  for (int t = blockIdx.x; t < n; t += gridDim.x) {
    for (int v0 = 0; v0 < vpr; v0 += RF16_VEC * 256) {
      uint4 o[RF16_VEC];
#pragma unroll
      for (int u = 0; u < RF16_VEC; ++u) {
        const int v = v0 + threadIdx.x + u * 256;
        if (v < vpr) {
          const uint4 raw = *reinterpret_cast<const uint4 *>(src + (size_t)t * K + v * 8);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t h[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xffff0000u);
            h[j] = (uint32_t)f16_bits_checked(lo, status, t) |
                   ((uint32_t)f16_bits_checked(hi, status, t) << 16);
          }
          o[u] = make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
      for (int j = 0; j < top_k; ++j) {
        const int q = inv_perm[(size_t)t * top_k + j];
        if (q < 0) continue;
        if (q >= P) {
          if (threadIdx.x == 0 && v0 == 0) set_status(status, MOE_ERR_BAD_INDEX, t * top_k + j);
          continue;
        }
#pragma unroll
        for (int u = 0; u < RF16_VEC; ++u) {
          const int v = v0 + threadIdx.x + u * 256;
          if (v < vpr) *reinterpret_cast<uint4 *>(dst + (size_t)q * K + v * 8) = o[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_rows_to_f16_scatter(const void *src, const int32_t *inv_perm, int top_k, int n,
                                       int K, void *dst, int *status, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  int blocks = n < 152 * 8 ? n : 152 * 8;
  rows_to_f16_scatter_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src),
                                                    inv_perm, top_k, n, n * top_k, K,
                                                    static_cast<uint16_t *>(dst), status);
  return cudaGetLastError();
}

bool decode_supported(const moe_config &c) {
  return (c.weight_dtype == MOE_MXFP4 || c.weight_dtype == MOE_NVFP4) &&
         c.act_dtype == MOE_BF16 && c.d % 32 == 0 &&
         c.d_ff % 32 == 0 && (int64_t)c.n * c.top_k <= kDecodeMaxPairs;
}

size_t mx_act16_bytes(const moe_config &c) {
  if ((c.weight_dtype != MOE_MXFP4 && c.weight_dtype != MOE_NVFP4) || c.act_dtype != MOE_BF16)
    return 0;
  const size_t P = (size_t)c.n * c.top_k;
  return P * (size_t)c.d * 2 + P * (size_t)c.d_ff * 2;
}

cudaError_t launch_rows_to_f16(const void *src, const int32_t *perm, int top_k, int P, int K,
                               void *dst, int *status, cudaStream_t s) {
  const int vec = P * (K / 8);
  int blocks = (vec + 255) / 256;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  if (blocks < 1) blocks = 1;
  rows_to_f16_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), perm, top_k,
                                           P, K, static_cast<uint16_t *>(dst), status);
  return cudaGetLastError();
}

cudaError_t launch_decode_ffn(const moe_config &c, int part, const void *act,
                              const int32_t *perm, const int32_t *offsets, const moe_weights &w,
                              void *h, void *y_perm, void *act16, int *status, cudaStream_t s,
                              const moe_expert_pool *pool) {
  if (c.weight_dtype == MOE_NVFP4)
    return pool ? cudaErrorNotSupported
                : launch_decode_ffn_nvfp4(c, part, act, perm, offsets, w, h, y_perm, act16, status,
                                          s);
  if (pool) return launch_decode_ffn_pooled(c, part, act, perm, offsets, w, h, y_perm, act16,
                                            status, s, *pool);
  return run_decode_ffn<false, 0>(c, part, act, perm, offsets, w, h, y_perm, act16, status, s,
                                  nullptr);
}

}  // namespace moe
