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

// The four code pairs of a 32-bit word (bytes 0..3) as four f16 pairs; each
// pair's low half is the low nibble (the even element).
struct F16x2x4 {
  uint32_t v[4];
};
__device__ __forceinline__ F16x2x4 e2m1x8_to_f16x2x4(uint32_t w) {
  F16x2x4 r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
      : "r"(w));
  return r;
}

// d = A * B (+ c), m16n8k16, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_16816_first(float (&c)[4], uint32_t a0, uint32_t a1,
                                                uint32_t a2, uint32_t a3, uint32_t b0,
                                                uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// E8M0 byte -> 2^(s-127) (s = 0 is the fp32 subnormal 2^-127; s = 255, not a
// valid scale, gives +inf).
__device__ __forceinline__ float e8m0_fast(uint32_t s) {
  return __uint_as_float(s ? (s << 23) : 0x00400000u);
}

// One MX block (32 elements) of rows g and g+8 against 8 tokens.  The block's
// 32 elements are fed to the two K=16 MMAs in a permuted order that both
// operands share: lane (g, t) owns word t of each row (elements 8t..8t+7) and
// the same 8 elements of its token's activation row.  MMA 1 takes bytes 0, 1
// of the word (elements 8t..8t+3), MMA 2 bytes 2, 3 (8t+4..8t+7).  A
// reduction does not depend on the order of its terms.
__device__ __forceinline__ void mx_block(float (&acc)[4], uint32_t wg, uint32_t wh, float sg,
                                         float sh, const uint4 &b) {
  const F16x2x4 ag = e2m1x8_to_f16x2x4(wg), ah = e2m1x8_to_f16x2x4(wh);
  float p[4];
  mma_16816_first(p, ag.v[0], ah.v[0], ag.v[1], ah.v[1], b.x, b.y);
  mma_16816(p, ag.v[2], ah.v[2], ag.v[3], ah.v[3], b.z, b.w);
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
// Persistent: the grid is sized to the GPU and each CTA walks its share of the
// work units (selected expert x 16 * row_groups output rows), slot-major.  Its
// DV_WARPS warps form row_groups groups of DV_WARPS / row_groups warps; the
// warps of a group split the reduction into contiguous runs of 128-byte
// boxes.  Each warp keeps its own ring of boxes per matrix in flight; lane 0
// refills a slot as soon as the warp has read it, with the next box of the
// warp's sequence — across token passes and units — so the weight stream
// does not stop at unit boundaries.  Block scales of the next unit are copied
// while the current one runs (two buffers).  B fragments (the tokens' f16
// activation rows, a few KB in L2) are loaded a box ahead of their use.  The
// partial sums of a group are added in warp order by its first warp, which
// applies the activation and stores.
template <int EPI>
__global__ void __launch_bounds__(32 * DV_WARPS)
decode_mxfp4_kernel(const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm3,
                    DecodeArgs a) {
  constexpr int NMAT = (EPI == 2) ? 2 : 1;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ uint64_t full[DV_WARPS][DV_STAGES_MAX];
  __shared__ uint64_t sbar[2];
  __shared__ int s_abort;
  __shared__ int s_nactive;
  __shared__ int s_active[257];
  __shared__ float red[DV_WARPS][32][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (status_failed(a.status)) return;

  // the experts with a non-empty segment, in order (E <= 256, one round of loads)
  if (warp == 0) {
    int off_lo[8], off_hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      off_lo[j] = e < a.num_experts ? a.offsets[e] : 0;
      off_hi[j] = e < a.num_experts ? a.offsets[e + 1] : 0;
    }
    int seen = 0, bad = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      const bool ne = e < a.num_experts && off_hi[j] > off_lo[j];
      if (e < a.num_experts && (off_lo[j] < 0 || off_hi[j] < off_lo[j] || off_hi[j] > a.P)) bad = 1;
      const unsigned m = __ballot_sync(0xffffffffu, ne);
      if (ne) s_active[seen + __popc(m & lanemask_lt())] = e;
      seen += __popc(m);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_nactive = bad ? 0 : seen;
      if (bad) set_status(a.status, MOE_ERR_BAD_INDEX, -1);
      s_abort = 0;
      tc::mbar_init(&sbar[0], 1);
      tc::mbar_init(&sbar[1], 1);
    }
  }
  if (lane == 0) {
    for (int st = 0; st < DV_STAGES_MAX; ++st) tc::mbar_init(&full[warp][st], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const int K = a.K, R = a.R, S = a.stages;
  const int RG = a.row_groups, KS = DV_WARPS / RG;
  const int grp = warp / KS, split = warp - grp * KS;
  const int KB = K / 32;                                // MX blocks per row
  const int NC = (K / 2 + DV_BOXB - 1) / DV_BOXB;       // boxes per row
  const int per_warp = (NC + KS - 1) / KS;
  const int c_beg = min(NC, split * per_warp), c_end = min(NC, c_beg + per_warp);
  const int cta_rows = 16 * RG;
  const int row_blocks = (R + cta_rows - 1) / cta_rows;
  const int total = s_nactive * row_blocks;
  const int sc_bytes = cta_rows * KB;                   // one unit's rows, one matrix
  const int sc_pitch = (sc_bytes + 15) & ~15;
  uint8_t *ring = smem + (size_t)warp * S * NMAT * DV_BOX;
  uint8_t *scl_base = smem + (size_t)DV_WARPS * S * NMAT * DV_BOX;
  const int g = lane >> 2, t = lane & 3;
  volatile int *abort = &s_abort;

  // unit i of this CTA -> (expert, first row); token passes of a unit
  auto unit_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };
  auto expert_of = [&](int u) { return s_active[u / row_blocks]; };
  auto row0_of = [&](int u) { return (u % row_blocks) * cta_rows; };
  auto passes_of = [&](int u) {
    const int e = expert_of(u);
    return (a.offsets[e + 1] - a.offsets[e] + DV_TOK - 1) / DV_TOK;
  };
  // scales of unit i -> buffer i & 1 (thread 0 only; sf_phase: parity of the
  // last copy issued into each buffer, -1 if none)
  int sf_phase[2] = {-1, -1};
  auto fetch_scales = [&](int i) {
    const int u = unit_of(i);
    if (u >= total) return;
    sf_phase[i & 1] = (i >> 1) & 1;
    const int e = expert_of(u), r0 = row0_of(u);
    const int rows = min(cta_rows, R - r0);
    const uint32_t bytes = (uint32_t)rows * KB;         // a multiple of 16 (rows % 16 == 0)
    uint8_t *dst = scl_base + (size_t)(i & 1) * NMAT * sc_pitch;
    tc::mbar_arrive_expect_tx(&sbar[i & 1], NMAT * bytes);
    bulk_load(dst, a.S + ((size_t)e * R + r0) * KB, bytes, &sbar[i & 1]);
    if (NMAT == 2) bulk_load(dst + sc_pitch, a.S3 + ((size_t)e * R + r0) * KB, bytes, &sbar[i & 1]);
  };
  // the producer's cursor over this warp's boxes: (unit i, pass p, box c)
  int pi = 0, pp = 0, pc = c_beg, issued = 0;
  bool pvalid = c_beg < c_end && unit_of(0) < total;
  auto issue_next = [&]() {
    if (!pvalid) return;
    const int u = unit_of(pi);
    const int r0 = row0_of(u) + grp * 16;
    const int slot = issued % S;
    if (r0 < R) {
      tc::mbar_arrive_expect_tx(&full[warp][slot], NMAT * DV_BOX);
      uint8_t *dst = ring + (size_t)slot * NMAT * DV_BOX;
      const int wrow = expert_of(u) * R + r0;
      tc::tma_load_2d(&tm1, &full[warp][slot], dst, pc * DV_BOXB, wrow);
      if (NMAT == 2) tc::tma_load_2d(&tm3, &full[warp][slot], dst + DV_BOX, pc * DV_BOXB, wrow);
    } else {
      tc::mbar_arrive(&full[warp][slot]);   // a group past the last row: keep the phases in step
    }
    ++issued;
    if (++pc == c_end) {
      pc = c_beg;
      if (++pp == passes_of(u)) {
        pp = 0;
        ++pi;
        pvalid = unit_of(pi) < total;
      }
    }
  };

  if (threadIdx.x == 0) {
    fetch_scales(0);
    fetch_scales(1);
  }
  if (lane == 0)
    for (int st = 0; st < S; ++st) issue_next();
  int consumed = 0;

  for (int i = 0; unit_of(i) < total; ++i) {
    const int u = unit_of(i);
    const int e = expert_of(u);
    const int r0 = row0_of(u) + grp * 16;
    const bool active = r0 < R;
    const int beg = a.offsets[e], cnt = a.offsets[e + 1] - beg;
    const uint8_t *scl = scl_base + (size_t)(i & 1) * NMAT * sc_pitch;
    const uint8_t *s1g = scl + (grp * 16 + g) * KB, *s1h = s1g + 8 * KB;
    const uint8_t *s3g = s1g + sc_pitch, *s3h = s1h + sc_pitch;
    bool scales_ready = false;
    for (int tg = 0; tg < cnt; tg += DV_TOK) {
      // every thread sees the same decision: a warp that timed out stops the CTA
      if (__syncthreads_or(*abort)) goto done;
      bool ok = true;
      if (!scales_ready && c_beg < c_end) {
        scales_ready = __all_sync(0xffffffffu, tc::mbar_wait(&sbar[i & 1], (i >> 1) & 1, abort));
        ok = scales_ready;
      }
      const bool xrow_ok = g < cnt - tg;                // token g of this pass exists
      const uint16_t *xrow = a.act16 + (size_t)(beg + tg + (xrow_ok ? g : 0)) * K + 8 * t;
      float acc1[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = c_beg; c < c_end && ok; ++c) {
        const int nb = min(8, KB - c * 8);
        uint4 bx[8];
#pragma unroll
        for (int bl = 0; bl < 8; ++bl)
          bx[bl] = (active && xrow_ok && bl < nb)
                       ? __ldg(reinterpret_cast<const uint4 *>(xrow + (c * 8 + bl) * 32))
                       : make_uint4(0u, 0u, 0u, 0u);
        const int slot = consumed % S;
        const uint32_t parity = (consumed / S) & 1;
        ++consumed;
        if (active) {
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[warp][slot], parity, abort));
          if (!ok) break;
          const uint8_t *st = ring + (size_t)slot * NMAT * DV_BOX;
          auto block = [&](int bl) {
            const int bg = c * 8 + bl;
            const int off = ((bl ^ g) << 4) + 4 * t;
            const uint32_t wg = *reinterpret_cast<const uint32_t *>(st + g * DV_BOXB + off);
            const uint32_t wh = *reinterpret_cast<const uint32_t *>(st + (g + 8) * DV_BOXB + off);
            mx_block(acc1, wg, wh, e8m0_fast(s1g[bg]), e8m0_fast(s1h[bg]), bx[bl]);
            if constexpr (NMAT == 2) {
              const uint32_t vg = *reinterpret_cast<const uint32_t *>(st + DV_BOX + g * DV_BOXB + off);
              const uint32_t vh =
                  *reinterpret_cast<const uint32_t *>(st + DV_BOX + (g + 8) * DV_BOXB + off);
              mx_block(acc3, vg, vh, e8m0_fast(s3g[bg]), e8m0_fast(s3h[bg]), bx[bl]);
            }
          };
          if (nb == 8) {
            // a full box: straight-line code, so the eight blocks' independent
            // MMA chains can be interleaved
#pragma unroll
            for (int bl = 0; bl < 8; ++bl) block(bl);
          } else {
            for (int bl = 0; bl < nb; ++bl) block(bl);
          }
        }
        __syncwarp();
        if (lane == 0) {
          // the slot was read through the generic proxy; order those reads
          // before the TMA engine overwrites it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue_next();
        }
      }
      // partial sums -> the first warp of the group, added in warp order
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        red[warp][lane][q] = acc1[q];
        red[warp][lane][4 + q] = acc3[q];
      }
      if (__syncthreads_or(!ok)) goto done;   // an aborted pass stores nothing
      if (split == 0 && active) {
        float s1[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = warp; w < warp + KS; ++w)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            s1[q] += red[w][lane][q];
            s3[q] += red[w][lane][4 + q];
          }
        // c0, c1: row g, tokens 2t, 2t+1; c2, c3: row g+8
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v;
          if constexpr (EPI == 2) v = s1[q] / (1.f + __expf(-s1[q])) * s3[q];
          else if constexpr (EPI == 1) v = fmaxf(s1[q], 0.f);
          else v = s1[q];
          const int tok = tg + 2 * t + (q & 1);
          const int row = r0 + g + ((q >> 1) ? 8 : 0);
          if (tok < cnt && row < R) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(v);
            a.out[(size_t)(beg + tok) * R + row] = hb;
            if (a.out16) a.out16[(size_t)(beg + tok) * R + row] = to_f16_bits(__bfloat162float(hb));
          }
        }
      }
    }
    // unit i is done everywhere: its scale buffer takes unit i + 2
    __syncthreads();
    if (threadIdx.x == 0) fetch_scales(i + 2);
  }
done:
  if (*abort) {
    // let the copies this CTA issued land before it exits
    if (lane == 0) {
      for (int j = consumed; j < issued; ++j)
        tc::mbar_wait_drain(&full[warp][j % S], (j / S) & 1, 100000000ull);
    }
    if (threadIdx.x == 0) {
      // scale copies in flight (a completed phase returns at once)
      for (int b = 0; b < 2; ++b)
        if (sf_phase[b] >= 0) tc::mbar_wait_drain(&sbar[b], (uint32_t)sf_phase[b], 100000000ull);
      set_status(a.status, MOE_ERR_TIMEOUT, blockIdx.x);
    }
  }
}

size_t decode_smem(int nmat, int K, int row_groups, int stages) {
  const int KB = K / 32;
  const size_t sc_pitch = (size_t)((16 * row_groups * KB + 15) & ~15);
  return 1024 + (size_t)DV_WARPS * stages * nmat * DV_BOX + 2 * (size_t)nmat * sc_pitch;
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
  static int per_sm = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_mxfp4_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
    per_sm = 0;
  }
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mxfp4_kernel<EPI>,
                                                      32 * DV_WARPS, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
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
  // units: at most `slots` experts x row blocks; no more CTAs than units
  const int cta_rows = 16 * a.row_groups;
  const long units = (long)slots * ((a.R + cta_rows - 1) / cta_rows);
  long grid = (long)per_sm * num_sms();
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  decode_mxfp4_kernel<EPI><<<(unsigned)grid, 32 * DV_WARPS, smem, s>>>(m1, m3, a);
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
