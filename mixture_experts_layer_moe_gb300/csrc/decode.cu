// Small-batch (decode) expert FFN over MXFP4 weights: stream only the
// selected experts' weights, once, and dequantise them in registers.
//
// The decode step touches a few experts per token, so its time is the time
// to read those experts' weight bytes from HBM ("Inference Optimization: The
// Bandwidth Wall, PagedAttention, and FlashAttention": decode is bound by the
// bytes of weights read per token).  Weights are MXFP4 (feed post "What is
// MXFP4?": 4-bit elements in blocks of 32 sharing one scale; E2M1 elements and
// E8M0 scales per the OCP MX v1.0 format).
//
// Work unit: one CTA = one selected expert x 16 output rows (one MMA M tile);
// its warps split the reduction.  Codes arrive by TMA (128-byte boxes of 16
// rows, 128-byte swizzle).  16 bytes of a row are exactly one MX block (32
// elements, one scale); lane (g = lane/4, t = lane%4) reads word t of the block
// for rows g and g+8 and converts its bytes with cvt.rn.f16x2.e2m1x2 straight
// into the A fragment of mma.sync.m16n8k16.  The expert's tokens (up to 8 per
// pass, N = 8) sit in shared memory as f16 and form the B fragment.  Each
// 32-element block is multiplied with unscaled E2M1 values into a fresh fp32
// partial, which is then scaled by the block's E8M0 scale and added to the
// fp32 accumulator.
//
// Activations enter the tensor core as f16 (E2M1 values are exact in f16);
// an activation beyond the f16 range (|v| > 65504) is clamped to it.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int DV_WARPS = 8;                 // warps per CTA = row groups x reduction splits
constexpr int DV_BOXB = 128;                // bytes of a row per TMA box: 8 MX blocks
constexpr int DV_BOX = 16 * DV_BOXB;        // one box: 16 rows x 128 bytes (128-byte swizzle)
constexpr int DV_STAGES_MAX = 2;            // boxes in flight per warp and matrix
constexpr int DV_TOK = 8;                   // tokens per pass (MMA N)

struct DecodeArgs {
  const int32_t *offsets;
  int num_experts;
  int P;
  const uint16_t *act16;          // f16 activation rows in segment order [P][K]
  int row_groups;                 // 16-row groups per CTA (1 or 4); DV_WARPS / row_groups splits
  int stages;                     // ring depth per warp (<= DV_STAGES_MAX)
  const uint8_t *S, *S3;          // scales [E][R][K/32] (S3: SwiGLU linear branch or nullptr)
  int R, K;
  __nv_bfloat16 *out;             // [P][R]
  uint16_t *out16;                // f16 copy of out (the next projection's input), or nullptr
  int *status;
};

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(d)
      : "r"(byte));
  return d;
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One MX block (32 elements) of rows g and g+8 against 8 tokens.  The block's
// 32 elements are fed to the two K=16 MMAs in a permuted order that both
// operands share: lane (g, t) owns word t of each row (elements 8t..8t+7) and
// the same 8 elements of its token's activation row.  MMA 1 takes bytes 0, 1
// of the word (elements 8t..8t+3), MMA 2 bytes 2, 3 (8t+4..8t+7).  A
// reduction does not depend on the order of its terms.
__device__ __forceinline__ void mx_block(float (&acc)[4], uint32_t wg, uint32_t wh, float sg,
                                         float sh, const uint4 &b) {
  float p[4] = {0.f, 0.f, 0.f, 0.f};
  mma_16816(p, e2m1x2_to_f16x2(wg), e2m1x2_to_f16x2(wh), e2m1x2_to_f16x2(wg >> 8),
            e2m1x2_to_f16x2(wh >> 8), b.x, b.y);
  mma_16816(p, e2m1x2_to_f16x2(wg >> 16), e2m1x2_to_f16x2(wh >> 16), e2m1x2_to_f16x2(wg >> 24),
            e2m1x2_to_f16x2(wh >> 24), b.z, b.w);
  acc[0] = fmaf(sg, p[0], acc[0]);
  acc[1] = fmaf(sg, p[1], acc[1]);
  acc[2] = fmaf(sh, p[2], acc[2]);
  acc[3] = fmaf(sh, p[3], acc[3]);
}

__device__ __forceinline__ uint16_t to_f16_bits(float v) {
  v = fminf(fmaxf(v, -65504.f), 65504.f);
  const __half h = __float2half_rn(v);
  return *reinterpret_cast<const uint16_t *>(&h);
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// Expert-ordered activation rows as f16: dst[q] = src[perm[q] / top_k] (perm
// given) or src[q], values clamped to the f16 range.
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
      o[j] = (uint32_t)to_f16_bits(lo) | ((uint32_t)to_f16_bits(hi) << 16);
    }
    *reinterpret_cast<uint4 *>(dst + (size_t)q * K + v * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// EPI: 0 none, 1 relu, 2 swiglu (tm3 / S3 hold the linear branch).
//
// One CTA = one selected expert x 16 * row_groups output rows.  Its DV_WARPS
// warps form row_groups groups of DV_WARPS / row_groups warps; the warps of a
// group split the reduction into contiguous runs of 128-byte boxes.  Each warp
// keeps its own ring of boxes per matrix in flight (lane 0 issues TMA and
// refills a slot once the warp has read it) and reads its fragments
// conflict-free from the 128-byte-swizzled boxes.  The B fragments (the
// tokens' f16 activation rows, a few KB that stay in L2) are loaded from
// global memory a box ahead of their use.  The partial sums of a group are
// added in warp order by its first warp, which applies the activation and
// stores.
template <int EPI>
__global__ void __launch_bounds__(32 * DV_WARPS)
decode_mxfp4_kernel(const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm3,
                    DecodeArgs a) {
  constexpr int NMAT = (EPI == 2) ? 2 : 1;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ uint64_t full[DV_WARPS][DV_STAGES_MAX];
  __shared__ uint64_t sbar;
  __shared__ int s_expert;
  __shared__ int s_abort;
  __shared__ float red[DV_WARPS][32][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (status_failed(a.status)) return;

  // slot blockIdx.y -> the blockIdx.y-th expert with a non-empty segment
  // (all offsets loaded up front: one memory latency, E <= 256)
  if (warp == 0) {
    const int slot = blockIdx.y;
    int off_lo[8], off_hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      off_lo[j] = e < a.num_experts ? a.offsets[e] : 0;
      off_hi[j] = e < a.num_experts ? a.offsets[e + 1] : 0;
    }
    int seen = 0, found = -1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int base = 32 * j;
      if (found >= 0 || base >= a.num_experts) continue;
      const bool ne = off_hi[j] > off_lo[j];
      unsigned m = __ballot_sync(0xffffffffu, ne);
      const int c = __popc(m);
      if (seen + c > slot) {
        for (int i = slot - seen; i > 0; --i) m &= m - 1;   // drop the lower set bits
        found = base + __ffs(m) - 1;
      }
      seen += c;
    }
    if (lane == 0) {
      s_expert = found;
      s_abort = 0;
      tc::mbar_init(&sbar, 1);
    }
  }
  if (lane == 0) {
    for (int st = 0; st < DV_STAGES_MAX; ++st) tc::mbar_init(&full[warp][st], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  const int e = s_expert;
  if (e < 0) return;
  const int beg = a.offsets[e], cnt = a.offsets[e + 1] - beg;
  if (beg < 0 || cnt < 0 || beg + cnt > a.P) {
    if (threadIdx.x == 0) set_status(a.status, MOE_ERR_BAD_INDEX, e);
    return;
  }
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const int K = a.K, R = a.R, S = a.stages;
  const int RG = a.row_groups, KS = DV_WARPS / RG;
  const int grp = warp / KS, split = warp - grp * KS;
  const int KB = K / 32;                                // MX blocks per row
  const int NC = (K / 2 + DV_BOXB - 1) / DV_BOXB;       // boxes per row
  const int per_warp = (NC + KS - 1) / KS;
  const int c_beg = min(NC, split * per_warp), c_end = min(NC, c_beg + per_warp);
  const int cta_rows = 16 * RG;
  const int sc_bytes = cta_rows * KB;                   // the CTA's rows, one matrix
  const int sc_pitch = (sc_bytes + 15) & ~15;
  uint8_t *ring = smem + (size_t)warp * S * NMAT * DV_BOX;
  uint8_t *scl = smem + (size_t)DV_WARPS * S * NMAT * DV_BOX;
  const int cta_r0 = blockIdx.x * cta_rows;
  const int r0 = cta_r0 + grp * 16;
  const bool active = r0 < R;
  const int g = lane >> 2, t = lane & 3;
  const int wrow = e * R + r0;                          // first code row of this warp
  volatile int *abort = &s_abort;

  auto issue = [&](int chunk, int slot) {
    tc::mbar_arrive_expect_tx(&full[warp][slot], NMAT * DV_BOX);
    uint8_t *dst = ring + (size_t)slot * NMAT * DV_BOX;
    tc::tma_load_2d(&tm1, &full[warp][slot], dst, chunk * DV_BOXB, wrow);
    if (NMAT == 2) tc::tma_load_2d(&tm3, &full[warp][slot], dst + DV_BOX, chunk * DV_BOXB, wrow);
  };

  if (threadIdx.x == 0) {
    const int rows = min(cta_rows, R - cta_r0);
    const uint32_t bytes = (uint32_t)rows * KB;         // a multiple of 16 (rows % 16 == 0)
    tc::mbar_arrive_expect_tx(&sbar, NMAT * bytes);
    bulk_load(scl, a.S + (size_t)(e * R + cta_r0) * KB, bytes, &sbar);
    if (NMAT == 2) bulk_load(scl + sc_pitch, a.S3 + (size_t)(e * R + cta_r0) * KB, bytes, &sbar);
  }
  bool scales_ready = false;
  int issued = 0, consumed = 0;
  const uint8_t *s1g = scl + (grp * 16 + g) * KB, *s1h = s1g + 8 * KB;
  const uint8_t *s3g = s1g + sc_pitch, *s3h = s1h + sc_pitch;

  for (int tg = 0; tg < cnt; tg += DV_TOK) {
    // every thread sees the same decision: a warp that timed out stops the CTA
    if (__syncthreads_or(*abort)) break;
    if (active && lane == 0) {
      for (int c = c_beg; c < c_end && c - c_beg < S; ++c) issue(c, (issued++) % S);
    }
    bool ok = true;
    if (active && !scales_ready) {
      scales_ready = __all_sync(0xffffffffu, tc::mbar_wait(&sbar, 0, abort));
      ok = scales_ready;
    }
    const bool xrow_ok = g < cnt - tg;                  // token g of this pass exists
    const uint16_t *xrow = a.act16 + (size_t)(beg + tg + (xrow_ok ? g : 0)) * K + 8 * t;
    float acc1[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = c_beg; active && c < c_end && ok; ++c) {
      const int nb = min(8, KB - c * 8);
      uint4 bx[8];
#pragma unroll
      for (int bl = 0; bl < 8; ++bl)
        bx[bl] = (xrow_ok && bl < nb) ? __ldg(reinterpret_cast<const uint4 *>(xrow + (c * 8 + bl) * 32))
                                      : make_uint4(0u, 0u, 0u, 0u);
      const int slot = consumed % S;
      const uint32_t parity = (consumed / S) & 1;
      ++consumed;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[warp][slot], parity, abort));
      if (!ok) break;
      const uint8_t *st = ring + (size_t)slot * NMAT * DV_BOX;
#pragma unroll
      for (int bl = 0; bl < 8; ++bl) {
        if (bl < nb) {
          const int bg = c * 8 + bl;
          const int off = ((bl ^ g) << 4) + 4 * t;
          const uint32_t wg = *reinterpret_cast<const uint32_t *>(st + g * DV_BOXB + off);
          const uint32_t wh = *reinterpret_cast<const uint32_t *>(st + (g + 8) * DV_BOXB + off);
          mx_block(acc1, wg, wh, e8m0_to_float(s1g[bg]), e8m0_to_float(s1h[bg]), bx[bl]);
          if constexpr (NMAT == 2) {
            const uint32_t vg =
                *reinterpret_cast<const uint32_t *>(st + DV_BOX + g * DV_BOXB + off);
            const uint32_t vh =
                *reinterpret_cast<const uint32_t *>(st + DV_BOX + (g + 8) * DV_BOXB + off);
            mx_block(acc3, vg, vh, e8m0_to_float(s3g[bg]), e8m0_to_float(s3h[bg]), bx[bl]);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && c + S < c_end) {
        // the slot was read through the generic proxy; order those reads
        // before the TMA engine overwrites it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(c + S, (issued++) % S);
      }
    }
    // partial sums -> the first warp of the group, added in warp order
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      red[warp][lane][i] = acc1[i];
      red[warp][lane][4 + i] = acc3[i];
    }
    if (__syncthreads_or(!ok)) continue;   // an aborted pass stores nothing
    if (split == 0 && active) {
      float s1[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w = warp; w < warp + KS; ++w)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s1[i] += red[w][lane][i];
          s3[i] += red[w][lane][4 + i];
        }
      // c0, c1: row g, tokens 2t, 2t+1; c2, c3: row g+8
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v;
        if constexpr (EPI == 2) v = s1[i] / (1.f + __expf(-s1[i])) * s3[i];
        else if constexpr (EPI == 1) v = fmaxf(s1[i], 0.f);
        else v = s1[i];
        const int tok = tg + 2 * t + (i & 1);
        const int row = r0 + g + ((i >> 1) ? 8 : 0);
        if (tok < cnt && row < R) {
          const __nv_bfloat16 hb = __float2bfloat16_rn(v);
          a.out[(size_t)(beg + tok) * R + row] = hb;
          if (a.out16) a.out16[(size_t)(beg + tok) * R + row] = to_f16_bits(__bfloat162float(hb));
        }
      }
    }
  }
  if (*abort) {
    // let the copies this CTA issued land before it exits
    if (lane == 0) {
      for (int j = consumed; j < issued; ++j)
        tc::mbar_wait_drain(&full[warp][j % S], (j / S) & 1, 100000000ull);
    }
    if (threadIdx.x == 0) {
      tc::mbar_wait_drain(&sbar, 0, 100000000ull);
      set_status(a.status, MOE_ERR_TIMEOUT, blockIdx.x);
    }
  }
}

size_t decode_smem(int nmat, int K, int row_groups, int stages) {
  const int KB = K / 32;
  const size_t sc_pitch = (size_t)((16 * row_groups * KB + 15) & ~15);
  return 1024 + (size_t)DV_WARPS * stages * nmat * DV_BOX + (size_t)nmat * sc_pitch;
}

template <int EPI>
cudaError_t launch_one(DecodeArgs a, const uint8_t *W, const uint8_t *W3, int num_experts,
                       int slots, cudaStream_t s) {
  constexpr int NMAT = (EPI == 2) ? 2 : 1;
  const int KS = DV_WARPS / a.row_groups;
  const int NC = (a.K / 2 + DV_BOXB - 1) / DV_BOXB;
  const int per_warp = (NC + KS - 1) / KS;
  a.stages = per_warp < DV_STAGES_MAX ? (per_warp > 0 ? per_warp : 1) : DV_STAGES_MAX;
  const size_t smem = decode_smem(NMAT, a.K, a.row_groups, a.stages);
  static size_t smem_set = 0;
  if (smem > 48 * 1024 && smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_mxfp4_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  CUtensorMap m1, m3;
  const uint64_t dims[2] = {(uint64_t)a.K / 2, (uint64_t)num_experts * a.R};
  const uint32_t box[2] = {DV_BOXB, 16};
  if (!make_tensor_map(&m1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W, 2, dims, box,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (NMAT == 2) {
    if (!make_tensor_map(&m3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W3, 2, dims, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    m3 = m1;
  }
  const int cta_rows = 16 * a.row_groups;
  dim3 grid((a.R + cta_rows - 1) / cta_rows, slots);
  decode_mxfp4_kernel<EPI><<<grid, 32 * DV_WARPS, smem, s>>>(m1, m3, a);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(const moe_config &c) {
  return c.weight_dtype == MOE_MXFP4 && c.act_dtype == MOE_BF16 && c.d % 32 == 0 &&
         c.d_ff % 32 == 0 && (int64_t)c.n * c.top_k <= kDecodeMaxPairs;
}

size_t mx_act16_bytes(const moe_config &c) {
  if (c.weight_dtype != MOE_MXFP4 || c.act_dtype != MOE_BF16) return 0;
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
                              void *h, void *y_perm, void *act16, int *status, cudaStream_t s) {
  const int P = c.n * c.top_k;
  const int slots = P < c.n_experts ? P : c.n_experts;
  uint16_t *x16 = static_cast<uint16_t *>(act16);
  uint16_t *h16 = x16 + (size_t)P * c.d;
  DecodeArgs a{};
  a.offsets = offsets;
  a.num_experts = c.n_experts;
  a.P = P;
  a.status = status;
  // few tokens per expert: eight reduction splits per 16 rows for parallelism;
  // more tokens: 64 rows per CTA, each staged B fragment serving more weights
  a.row_groups = c.n <= 2 ? 1 : 4;
  if (part == 0) {
    cudaError_t e = launch_rows_to_f16(act, perm, c.top_k, P, c.d, x16, status, s);
    if (e != cudaSuccess) return e;
    a.act16 = x16;
    a.S = w.S1;
    a.S3 = w.S3;
    a.R = c.d_ff;
    a.K = c.d;
    a.out = static_cast<__nv_bfloat16 *>(h);
    a.out16 = h16;
    const uint8_t *W1 = static_cast<const uint8_t *>(w.W1), *W3 = static_cast<const uint8_t *>(w.W3);
    return c.act == MOE_ACT_SWIGLU ? launch_one<2>(a, W1, W3, c.n_experts, slots, s)
                                   : launch_one<1>(a, W1, nullptr, c.n_experts, slots, s);
  }
  a.act16 = h16;
  a.S = w.S2;
  a.S3 = nullptr;
  a.R = c.d;
  a.K = c.d_ff;
  a.out = static_cast<__nv_bfloat16 *>(y_perm);
  a.out16 = nullptr;
  return launch_one<0>(a, static_cast<const uint8_t *>(w.W2), nullptr, c.n_experts, slots, s);
}

}  // namespace moe
