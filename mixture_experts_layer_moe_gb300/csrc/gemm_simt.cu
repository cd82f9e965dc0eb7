// Grouped expert GEMM on CUDA cores (fp32 FMA accumulation).
//
// Runs each expert's FFN projection on its dispatched segment ("How Mixture of
// Experts Scales Model Parameters", sections "Dense models" and "The forward
// pass: dispatch, then combine").  This is the fp32 path (fp32 tensor-core
// modes cannot hold a 1e-4 relative error) and the path for shapes the
// tensor-core kernels do not take.  MXFP4 weights (E2M1 codes, one E8M0 scale
// per 32 elements along the reduction dimension) are decoded while the tile is
// staged in shared memory.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int SB_M = 64, SB_N = 64, SB_K = 32, SB_THREADS = 256;

template <int BT>
__device__ __forceinline__ float load_b(const void *B, const uint8_t *S, size_t row, int K, int k) {
  if constexpr (BT == MOE_F32) {
    return static_cast<const float *>(B)[row * K + k];
  } else if constexpr (BT == MOE_BF16) {
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(B)[row * K + k]);
  } else {
    const uint8_t byte = static_cast<const uint8_t *>(B)[row * (K / 2) + (k >> 1)];
    const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
    return e2m1_to_float(code) * e8m0_to_float(S[row * (K / 32) + (k >> 5)]);
  }
}

template <typename TA, int BT, typename TO, int EPI>
__global__ void __launch_bounds__(SB_THREADS) gemm_simt_kernel(GemmStage g, int *status) {
  __shared__ float as[SB_K][SB_M + 4];
  __shared__ float bs[SB_K][SB_N + 4];
  __shared__ float b3s[EPI == 2 ? SB_K : 1][SB_N + 4];
  if (status_failed(status)) return;

  // locate (expert, row range) of this M tile
  int e = -1, row0 = 0, seg_end = 0;
  const int tile = blockIdx.x;
  if (g.offsets == nullptr) {
    e = 0;
    row0 = tile * SB_M;
    seg_end = g.rows;
    if (row0 >= seg_end) return;
  } else {
    int acc = 0;
    for (int ee = 0; ee < g.num_experts; ++ee) {
      const int beg = g.offsets[ee], end = g.offsets[ee + 1];
      if (beg < 0 || end < beg || end > g.rows) {
        if (threadIdx.x == 0) set_status(status, MOE_ERR_BAD_INDEX, ee);
        return;
      }
      const int nt = (end - beg + SB_M - 1) / SB_M;
      if (tile < acc + nt) {
        e = ee;
        row0 = beg + (tile - acc) * SB_M;
        seg_end = end;
        break;
      }
      acc += nt;
    }
    if (e < 0) return;
  }
  const int n0 = blockIdx.y * SB_N;
  const int N = g.N, K = g.K;
  const TA *A = static_cast<const TA *>(g.A);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {}, acc3[4][4] = {};

  for (int k0 = 0; k0 < K; k0 += SB_K) {
    for (int i = threadIdx.x; i < SB_M * SB_K; i += SB_THREADS) {
      const int r = i / SB_K, kk = i % SB_K, gk = k0 + kk;
      const int gr = row0 + r, gn = n0 + r;
      as[kk][r] = (gr < seg_end && gk < K) ? Elem<TA>::load(A + (size_t)gr * K + gk) : 0.f;
      const bool bok = gn < N && gk < K;
      const size_t brow = (size_t)e * N + gn;
      bs[kk][r] = bok ? load_b<BT>(g.B, g.SB, brow, K, gk) : 0.f;
      if constexpr (EPI == 2) b3s[kk][r] = bok ? load_b<BT>(g.B3, g.SB3, brow, K, gk) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], b[4], b3[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[kk][tx * 4 + j];
      if constexpr (EPI == 2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) b3[j] = b3s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if constexpr (EPI == 2) acc3[i][j] = fmaf(a[i], b3[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
  TO *out = static_cast<TO *>(g.out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gr = row0 + ty * 4 + i;
    if (gr >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j];
      if constexpr (EPI == 1) v = fmaxf(v, 0.f);
      if constexpr (EPI == 2) v = v / (1.f + expf(-v)) * acc3[i][j];
      out[(size_t)gr * N + gn] = Elem<TO>::from_f(v);
    }
  }
}

template <typename TA, int BT, typename TO>
cudaError_t launch_epi(const GemmStage &g, int *status, cudaStream_t s) {
  const int mt = g.offsets ? (g.rows + SB_M - 1) / SB_M + g.num_experts
                           : (g.rows + SB_M - 1) / SB_M;
  dim3 grid(mt, (g.N + SB_N - 1) / SB_N);
  switch (g.epi) {
    case 0: gemm_simt_kernel<TA, BT, TO, 0><<<grid, SB_THREADS, 0, s>>>(g, status); break;
    case 1: gemm_simt_kernel<TA, BT, TO, 1><<<grid, SB_THREADS, 0, s>>>(g, status); break;
    default: gemm_simt_kernel<TA, BT, TO, 2><<<grid, SB_THREADS, 0, s>>>(g, status); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmStage &g, int *status, cudaStream_t s) {
  if (g.rows == 0) return cudaSuccess;
  if (g.a_dtype == MOE_F32) {
    if (g.b_dtype != MOE_F32 || g.out_dtype != MOE_F32) return cudaErrorInvalidValue;
    return launch_epi<float, MOE_F32, float>(g, status, s);
  }
  if (g.out_dtype != MOE_BF16) return cudaErrorInvalidValue;
  if (g.b_dtype == MOE_BF16) return launch_epi<__nv_bfloat16, MOE_BF16, __nv_bfloat16>(g, status, s);
  if (g.b_dtype == MOE_MXFP4) return launch_epi<__nv_bfloat16, MOE_MXFP4, __nv_bfloat16>(g, status, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
