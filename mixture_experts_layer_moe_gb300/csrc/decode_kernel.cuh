// Small-batch (decode) expert FFN over MXFP4 weights: stream only the
// selected experts' weights, once, and dequantise them in registers.  The
// kernel template; decode.cu instantiates it without a resident pool,
// decode_pool.cu with one.
//
// The decode step touches a few experts per token, so its time is the time
// to read those experts' weight bytes from HBM ("Inference Optimization: The
// Bandwidth Wall, PagedAttention, and FlashAttention": decode is bound by the
// bytes of weights read per token).  Weights are MXFP4 (feed post "What is
// MXFP4?": 4-bit elements in blocks of 32 sharing one scale; E2M1 elements and
// E8M0 scales per the OCP MX v1.0 format).
//
// Work unit: one selected expert x 16 * RG output rows (RG MMA M tiles); the
// warps of a 16-row group split the reduction.  Codes arrive by TMA (128-byte
// boxes of 16 rows, 128-byte swizzle).  16 bytes of a row are exactly one MX
// block (32 elements, one scale); lane (g = lane/4, t = lane%4) reads word t of
// the block for rows g and g+8 and converts its bytes with
// cvt.rn.f16x2.e2m1x2 straight into the A fragment of mma.sync.m16n8k16.  The
// expert's tokens (up to 8 per pass, N = 8) are f16 rows read from L2 into
// the B fragment.  Each 32-element block is multiplied with unscaled E2M1
// values into a fresh fp32 partial, which is then scaled by the block's E8M0
// scale and added to the fp32 accumulator.
//
// Activations enter the tensor core as f16 (E2M1 values are exact in f16);
// an activation beyond the f16 range (|v| > 65504) is reported through the
// status word (f16_bits_checked).
#pragma once

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int DV_WARPS = 8;                 // warps per CTA = row groups x reduction splits
constexpr int DV_BOXB = 128;                // bytes of a row per TMA box: 8 MX blocks
constexpr int DV_BOX = 16 * DV_BOXB;        // one box: 16 rows x 128 bytes (128-byte swizzle)
constexpr int DV_STAGES = 2;                // boxes in flight per warp and matrix (a power of 2)
constexpr int DV_TOK = 8;                   // tokens per pass (MMA N)

struct DecodeArgs {
  const int32_t *offsets;
  int num_experts;
  int P;
  const uint16_t *act16;          // f16 activation rows: segment order [P][K], or token order
  const int32_t *perm;            // (token order) segment position -> pair t*top_k + j, else nullptr
  int top_k;
  const uint8_t *S, *S3;          // scales [E][R][K/32] (S3: SwiGLU linear branch or nullptr)
  const int32_t *slot_of;         // [E] pool slot of each expert or -1; nullptr: no pool
  int n_slots;
  const uint8_t *PS, *PS3;        // pool scales [n_slots][R][K/32]
  const float *G, *G3;            // NVFP4: per-expert fp32 scales of the two matrices
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

// NVFP4 (blocks of 16): the two 16-bit halves of w, each two E4M3 bytes, ->
// two f16x2 (low byte to the low half).  E4M3 values are exact in f16.
__device__ __forceinline__ uint2 e4m3x4_to_f16x2x2(uint32_t w) {
  uint2 d;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(d.x), "=r"(d.y)
      : "r"(w));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One 16-byte chunk (two NVFP4 blocks) of rows g and g+8 against 8 tokens.
// Lane (g, t) holds word t of each row, which lies in block t / 2, so one
// scale per row covers all of the lane's elements: sgh = {s_g, s_g+8} as
// f16x2.  E2M1 x E4M3 has at most 5 significant bits and lies within
// 2^-10 .. 2688, so the scaled codes are exact in f16 and both MMAs
// accumulate straight into the fp32 accumulator.
__device__ __forceinline__ void nv_block(float (&acc)[4], uint32_t wg, uint32_t wh, uint32_t sgh,
                                         const uint4 &b) {
  const F16x2x4 ag = e2m1x8_to_f16x2x4(wg), ah = e2m1x8_to_f16x2x4(wh);
  const uint32_t sg = __byte_perm(sgh, sgh, 0x1010), sh = __byte_perm(sgh, sgh, 0x3232);
  mma_16816(acc, hmul2_bits(ag.v[0], sg), hmul2_bits(ah.v[0], sh), hmul2_bits(ag.v[1], sg),
            hmul2_bits(ah.v[1], sh), b.x, b.y);
  mma_16816(acc, hmul2_bits(ag.v[2], sg), hmul2_bits(ah.v[2], sh), hmul2_bits(ag.v[3], sg),
            hmul2_bits(ah.v[3], sh), b.z, b.w);
}


__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// Group barrier on named barrier 1 + id over n threads: returns the OR of
// pred over the group (every thread gets the same answer).
__device__ __forceinline__ bool group_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(1 + id), "r"(n)
      : "memory");
  return r != 0;
}

// Shared-memory plan of the decode kernel (bytes from the 1024-aligned base).
struct DecodePlan {
  int KB;          // MX blocks per row
  int bps;         // blocks per reduction split
  int PP;          // decoded-scale row pitch (u32) of one warp
  int spc;         // scale bytes per 16-byte code chunk: 1 (MXFP4) or 2 (NVFP4)
  int sc_pitch;    // raw scale bytes of one unit and matrix, padded to 16
  int nraw;        // raw scale buffers (two for short units: copies run two units ahead)
  size_t raw_off, pairs_off, red_off, bytes;
};

__host__ __device__ inline DecodePlan decode_plan(int nmat, int K, int rg, int fmt) {
  DecodePlan p;
  const int ks = DV_WARPS / rg;
  p.KB = K / 32;
  // an even split point keeps every warp's first raw scale byte 2-byte aligned
  p.bps = (((p.KB + ks - 1) / ks) + 1) & ~1;
  p.PP = (p.bps + 7) & ~7;
  if (p.PP % 32 == 0) p.PP += 8;   // rows g and g + 1 of a quarter-warp on other banks
  p.spc = fmt == 1 ? 2 : 1;
  p.sc_pitch = (16 * rg * p.KB * p.spc + 15) & ~15;
  p.nraw = rg == 1 ? 2 : 1;
  p.raw_off = (size_t)DV_WARPS * DV_STAGES * 2 * DV_BOX;
  p.pairs_off = p.raw_off + (size_t)p.nraw * nmat * p.sc_pitch;
  p.red_off = p.pairs_off + (size_t)DV_WARPS * nmat * 8 * p.PP * 4;
  const int red_vals = ks == 2 ? 4 : 8;
  p.bytes = p.red_off + (size_t)2 * DV_WARPS * red_vals * 32 * 4;
  return p;
}

struct ProducerState {
  int i, pass, c, passes, wrow, issued;
  bool valid, active, pool;
};

// EPI: 0 none, 1 relu, 2 swiglu (tm3 / S3 hold the linear branch), 3 none with
// 32-row groups: rows r .. r+15 and r+16 .. r+31 of the one matrix take the
// places of the two SwiGLU matrices, so each activation fragment a warp loads
// serves two rows' MMAs (the row count must be a multiple of 32).  RG: row
// groups per CTA; the KS = DV_WARPS / RG warps of a group split the reduction
// into contiguous, equal runs of MX blocks.
//
// Persistent: the grid is sized to the GPU and each CTA walks its share of the
// work units (selected expert x 16 * RG output rows), slot-major.  The groups
// of a CTA run independently: the warps of a group meet only on their own
// named barrier, once per token pass, to add their partial sums.  Each warp
// keeps its own ring of 128-byte code boxes per matrix in flight; lane 0
// refills a slot as soon as the warp has read it, with the next box of the
// warp's sequence (across token passes and units), so the weight stream does
// not stop at unit boundaries.  A unit's E8M0 bytes are bulk-copied into
// shared memory ahead of it (one unit ahead, two for short 16-row units);
// each warp decodes the part it reads into bf16 pairs (row g | row g + 8), so
// that the inner loop takes eight blocks' scales with two 16-byte loads, and
// the last warp done with a raw buffer issues the copy for the unit that uses
// it next.  B fragments (the tokens' f16 activation rows, a few KB in L2) are
// loaded at the top of each slot, and the next slot's lines are prefetched
// into L1.
template <int EPI, int RG, bool POOL, int FMT>
__global__ void __launch_bounds__(32 * DV_WARPS, 2)
decode_mxfp4_kernel(const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm3,
                    const __grid_constant__ CUtensorMap tp1, const __grid_constant__ CUtensorMap tp3,
                    DecodeArgs a) {
  constexpr bool PAIRED = EPI == 3;
  constexpr int NMAT = (EPI == 2 || PAIRED) ? 2 : 1;
  constexpr int GROWS = PAIRED ? 32 : 16;   // weight rows per group
  constexpr int KS = DV_WARPS / RG;
  constexpr int CTA_ROWS = GROWS * RG;
  constexpr int RV = KS == 2 ? 4 : 8;   // partial sums a warp hands over per lane
  constexpr int SPC = FMT == 1 ? 2 : 1; // scale bytes per 16-byte code chunk
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ uint64_t full[DV_WARPS][DV_STAGES];
  __shared__ uint64_t sbar[2];
  __shared__ int s_abort;
  __shared__ int s_nactive;
  __shared__ unsigned s_raw_done;
  // per active expert: id, segment start and length (all < 2^15: E <= 256 and
  // P <= kDecodeMaxPairs), pool slot or -1; per segment position: the
  // activation row.  16-bit where it fits: with the rest of the shared memory,
  // the SwiGLU kernel must stay within two CTAs per SM.
  __shared__ int16_t s_active[256], s_beg[256], s_cnt[256];
  __shared__ int16_t s_row[kDecodeMaxPairs];
  __shared__ int s_slot[POOL ? 256 : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    tc::prefetch_tmap(&tm1);
    if (EPI == 2) tc::prefetch_tmap(&tm3);
    if constexpr (POOL) {
      tc::prefetch_tmap(&tp1);
      if (EPI == 2) tc::prefetch_tmap(&tp3);
    }
  }
  pdl_wait();
  if (status_failed(a.status)) return;

  // the experts with a non-empty segment, in order (E <= 256, one round of loads)
  if (warp == 0) {
    int off_lo[8], off_hi[8], slot[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      off_lo[j] = e < a.num_experts ? a.offsets[e] : 0;
      off_hi[j] = e < a.num_experts ? a.offsets[e + 1] : 0;
      slot[j] = (POOL && e < a.num_experts) ? a.slot_of[e] : -1;
    }
    int seen = 0, bad = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 32 * j + lane;
      const bool ne = e < a.num_experts && off_hi[j] > off_lo[j];
      if (e < a.num_experts && (off_lo[j] < 0 || off_hi[j] < off_lo[j] || off_hi[j] > a.P)) bad = 1;
      const unsigned m = __ballot_sync(0xffffffffu, ne);
      if (ne) {
        const int q = seen + __popc(m & lanemask_lt());
        s_active[q] = (int16_t)e;
        s_beg[q] = (int16_t)off_lo[j];
        s_cnt[q] = (int16_t)(off_hi[j] - off_lo[j]);
        if constexpr (POOL) {
          // a slot outside the pool is reported and the expert read from the
          // backing arrays
          if (slot[j] < -1 || slot[j] >= a.n_slots) set_status(a.status, MOE_ERR_BAD_INDEX, e);
          s_slot[q] = (slot[j] >= 0 && slot[j] < a.n_slots) ? slot[j] : -1;
        }
      }
      seen += __popc(m);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      s_nactive = bad ? 0 : seen;
      if (bad) set_status(a.status, MOE_ERR_BAD_INDEX, -1);
      s_abort = 0;
      s_raw_done = 0;
      tc::mbar_init(&sbar[0], 1);
      tc::mbar_init(&sbar[1], 1);
    }
  }
  if (warp == 1) {
    for (int q = lane; q < a.P; q += 32) {
      int row = q;
      if (a.perm) {
        const int p = a.perm[q];
        row = (p >= 0 && p < a.P) ? p / a.top_k : 0;
        if (p < 0 || p >= a.P) set_status(a.status, MOE_ERR_BAD_INDEX, q);
      }
      s_row[q] = (int16_t)row;
    }
  }
  if (lane == 0) {
    for (int st = 0; st < DV_STAGES; ++st) tc::mbar_init(&full[warp][st], 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  const DecodePlan plan = decode_plan(NMAT, a.K, RG, FMT);
  const int K = a.K, R = a.R, KB = plan.KB, PP = plan.PP, sc_pitch = plan.sc_pitch;
  const int grp = warp / KS, split = warp - grp * KS;
  const int b_beg = min(KB, split * plan.bps), b_end = min(KB, b_beg + plan.bps);
  const int nbl = b_end - b_beg;                        // this warp's MX blocks per row
  // a ring slot holds two 16 x 128-byte boxes: the same 8 MX blocks of both
  // matrices (SwiGLU), or 16 consecutive blocks of the one matrix
  constexpr int SUB = (NMAT == 2) ? 1 : 2;              // 8-block groups per slot
  constexpr int SB = 8 * SUB;                           // MX blocks per slot
  const int nslot = (nbl + SB - 1) / SB;
  const int row_blocks = (R + CTA_ROWS - 1) / CTA_ROWS;
  const int total = s_nactive * row_blocks;
  uint8_t *ring = smem + (size_t)warp * DV_STAGES * 2 * DV_BOX;
  const int NRAW = plan.nraw;
  uint32_t *pw = reinterpret_cast<uint32_t *>(smem + plan.pairs_off) + (size_t)warp * NMAT * 8 * PP;
  float *red = reinterpret_cast<float *>(smem + plan.red_off);   // [2][DV_WARPS][RV][32]
  const int g = lane >> 2, t = lane & 3;
  // byte offset of word t of 16-byte chunk (bl ^ g) in row g of a box with
  // the 128-byte swizzle: lane_off ^ (bl << 4)
  const uint32_t lane_off = (uint32_t)(g * DV_BOXB + (g << 4) + 4 * t);
  volatile int *abort = &s_abort;

  // raw E8M0 bytes of this CTA's unit i into buffer i % NRAW (NRAW copies in
  // flight at most; a thread drains the copies it issued on abort)
  int raw_mine0 = -1, raw_mine1 = -1;   // last unit copied into buffer 0 / 1
  auto fetch_raw = [&](int i) {
    const int u = (int)blockIdx.x + i * (int)gridDim.x;
    if (u >= total) return;
    const int sl = u / row_blocks;
    const int e = s_active[sl], r0 = (u - sl * row_blocks) * CTA_ROWS;
    const uint32_t bytes = (uint32_t)min(CTA_ROWS, R - r0) * KB * SPC;   // rows % 16 == 0
    const int b = i % NRAW;
    tc::mbar_arrive_expect_tx(&sbar[b], (PAIRED ? 1 : NMAT) * bytes);
    uint8_t *dst = smem + plan.raw_off + (size_t)b * NMAT * sc_pitch;
    // the resident copy (pool slot) or the backing expert
    const int ps = POOL ? s_slot[sl] : -1;
    const uint8_t *S1 = ps >= 0 ? a.PS : a.S, *S3 = ps >= 0 ? a.PS3 : a.S3;
    const size_t row = (size_t)(ps >= 0 ? ps : e) * R + r0;
    bulk_load(dst, S1 + row * KB * SPC, bytes, &sbar[b]);
    if (EPI == 2) bulk_load(dst + sc_pitch, S3 + row * KB * SPC, bytes, &sbar[b]);
    if (b) raw_mine1 = i;
    else raw_mine0 = i;
  };

  // the producer's cursor over this warp's slots (lane 0): unit i, pass, slot
  // c of the pass, the first weight row of the warp's group, slots issued
  ProducerState P{};
  auto p_load_unit = [&]() {
    const int u = (int)blockIdx.x + P.i * (int)gridDim.x;
    P.valid = nslot > 0 && u < total;
    if (!P.valid) return;
    const int sl = u / row_blocks;
    const int r = (u - sl * row_blocks) * CTA_ROWS + grp * GROWS;
    P.active = r < R;
    P.pool = POOL && s_slot[sl] >= 0;
    P.wrow = (P.pool ? s_slot[sl] : s_active[sl]) * R + r;
    P.passes = (s_cnt[sl] + DV_TOK - 1) / DV_TOK;
  };
  auto issue_next = [&]() {
    if (!P.valid) return;
    const int sl = P.issued & (DV_STAGES - 1);
    if (P.active) {
      tc::mbar_arrive_expect_tx(&full[warp][sl], 2 * DV_BOX);
      uint8_t *dst = ring + (size_t)sl * 2 * DV_BOX;
      const int x = (b_beg + SB * P.c) * 16;            // a multiple of 16 bytes
      const int y = P.wrow;
      // each copy names its tensor map directly (a kernel-parameter address);
      // a box past the end of the row reads zeros
      if (POOL && P.pool) {
        tc::tma_load_2d(&tp1, &full[warp][sl], dst, x, y);
        if (EPI == 2) tc::tma_load_2d(&tp3, &full[warp][sl], dst + DV_BOX, x, y);
        else if (PAIRED) tc::tma_load_2d(&tp1, &full[warp][sl], dst + DV_BOX, x, y + 16);
        else tc::tma_load_2d(&tp1, &full[warp][sl], dst + DV_BOX, x + DV_BOXB, y);
      } else {
        tc::tma_load_2d(&tm1, &full[warp][sl], dst, x, y);
        if (EPI == 2) tc::tma_load_2d(&tm3, &full[warp][sl], dst + DV_BOX, x, y);
        else if (PAIRED) tc::tma_load_2d(&tm1, &full[warp][sl], dst + DV_BOX, x, y + 16);
        else tc::tma_load_2d(&tm1, &full[warp][sl], dst + DV_BOX, x + DV_BOXB, y);
      }
    } else {
      tc::mbar_arrive(&full[warp][sl]);   // a group past the last row: keep the phases in step
    }
    ++P.issued;
    if (++P.c == nslot) {
      P.c = 0;
      if (++P.pass == P.passes) {
        P.pass = 0;
        ++P.i;
        p_load_unit();
      }
    }
  };

  if (threadIdx.x == 0)
    for (int i = 0; i < NRAW; ++i) fetch_raw(i);
  if (lane == 0) {
    p_load_unit();
    for (int st = 0; st < DV_STAGES; ++st) issue_next();
  }
  int consumed = 0, npass = 0;
  bool ok = true;

  for (int i = 0;; ++i) {
    const int u = (int)blockIdx.x + i * (int)gridDim.x;
    if (u >= total) break;
    const int sl = u / row_blocks;
    const int r0 = (u - sl * row_blocks) * CTA_ROWS + grp * GROWS;
    const bool active = r0 < R;
    const int beg = s_beg[sl], cnt = s_cnt[sl];

    // this unit's scales: wait for the raw bytes, decode this warp's part into
    // pairs; the last warp to finish issues the next unit's copy
    ok = __all_sync(0xffffffffu,
                    tc::mbar_wait(&sbar[i % NRAW], (uint32_t)((i / NRAW) & 1), abort));
    // the warps of a group leave together, so none waits on a barrier alone
    if (group_sync_or(grp, 32 * KS, !ok)) { ok = false; break; }
    // raw scale row gg of "matrix" m of this warp's group: the second matrix's
    // rows (SwiGLU), or rows 16..31 of the group (paired rows), at the
    // warp's first block
    auto raw_row = [&](int m, int gg) -> const uint8_t * {
      const uint8_t *buf = smem + plan.raw_off + (size_t)(i % NRAW) * NMAT * sc_pitch;
      if constexpr (PAIRED) return buf + ((size_t)(grp * GROWS + 16 * m + gg) * KB + b_beg) * SPC;
      return buf + (size_t)m * sc_pitch + ((size_t)(grp * 16 + gg) * KB + b_beg) * SPC;
    };
    if constexpr (FMT == 1) {
      // NVFP4: lane (gg = lane / 4, q = lane % 4) takes chunks q, q + 4, ...
      // of row pair gg; a chunk's two scale bytes of row gg and of row gg + 8
      // become two byte pairs {s_gg, s_gg+8}, one per block parity, stored
      // [matrix][row pair][parity][chunk] as 16-bit values
      const int gg = lane >> 2, q = lane & 3;
      uint16_t *pw16 = reinterpret_cast<uint16_t *>(pw);
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint8_t *src = raw_row(m, gg);
        uint16_t *dst = pw16 + (size_t)(m * 8 + gg) * 2 * PP;
        for (int b = q; b < nbl; b += 4) {
          const uint32_t x = *reinterpret_cast<const uint16_t *>(src + 2 * b);
          const uint32_t y = *reinterpret_cast<const uint16_t *>(src + 2 * b + 16 * KB);
          dst[b] = (uint16_t)__byte_perm(x, y, 0x0040);
          dst[PP + b] = (uint16_t)__byte_perm(x, y, 0x0051);
        }
      }
    } else {
      // lane (gg = lane / 4, q = lane % 4) takes blocks 2q, 2q + 1, 2q + 8, ...
      // of row pair gg: two raw bytes of row gg and two of row gg + 8 per step
      // (16-bit loads where the row pitch is even: the split point always is)
      const int gg = lane >> 2, q = lane & 3;
      const bool even = (KB & 1) == 0;
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        const uint8_t *src = raw_row(m, gg);
        uint32_t *dst = pw + (m * 8 + gg) * PP;
        for (int b = 2 * q; b < nbl; b += 8) {
          const bool two = b + 1 < nbl;
          uint32_t x, y;
          if (even) {
            x = *reinterpret_cast<const uint16_t *>(src + b);
            y = *reinterpret_cast<const uint16_t *>(src + b + 8 * KB);
          } else {
            x = src[b] | (two ? (uint32_t)src[b + 1] << 8 : 0u);
            y = src[b + 8 * KB] | (two ? (uint32_t)src[b + 1 + 8 * KB] << 8 : 0u);
          }
          // bf16 of 2^(s-127): s << 7, and 0x0040 (2^-127, a subnormal) for s = 0
          const uint32_t p0 = __vmaxu2(__byte_perm(x, y, 0x7460) << 7, 0x00400040u);
          const uint32_t p1 = __vmaxu2(__byte_perm(x, y, 0x7561) << 7, 0x00400040u);
          if (two) *reinterpret_cast<uint2 *>(dst + b) = make_uint2(p0, p1);
          else dst[b] = p0;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&s_raw_done, 1u) == (unsigned)((i + 1) * DV_WARPS - 1)) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        fetch_raw(i + NRAW);
      }
    }
    const uint32_t *pr1 = pw + g * PP;
    const uint32_t *pr3 = pr1 + 8 * PP;
    // NVFP4: this lane's block parity (t / 2) row of byte pairs
    const uint16_t *pn1 = reinterpret_cast<const uint16_t *>(pw) + (size_t)(g * 2 + (t >> 1)) * PP;
    const uint16_t *pn3 = pn1 + (size_t)8 * 2 * PP;
    float gs1 = 1.f, gs3 = 1.f;   // NVFP4 matrix scales of this unit's expert
    if constexpr (FMT == 1) {
      gs1 = a.G[s_active[sl]];
      if (EPI == 2) gs3 = a.G3[s_active[sl]];
      else if (PAIRED) gs3 = gs1;
    }

    for (int tg = 0; tg < cnt; tg += DV_TOK, ++npass) {
      // token g of this pass, or the pass's last token where g is past it (its
      // results are not stored)
      const int tok = tg + min(g, cnt - tg - 1);
      const uint16_t *xrow = a.act16 + (size_t)s_row[beg + tok] * K + (size_t)b_beg * 32 + 8 * t;
      const uint16_t *xpf = a.act16 + (size_t)s_row[beg + tg + min(lane >> 2, cnt - tg - 1)] * K +
                            (size_t)b_beg * 32 + (lane & 3) * 64;
      float acc1[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
      uint4 bx[8];
      // B fragments of the 8-block group starting at local block cb
      auto load_bx = [&](int cb, int nb) {
        const uint16_t *xb = xrow + cb * 32;
#pragma unroll
        for (int bl = 0; bl < 8; ++bl)
          bx[bl] = (bl < nb) ? __ldg(reinterpret_cast<const uint4 *>(xb + bl * 32))
                             : make_uint4(0u, 0u, 0u, 0u);
      };
      // the 8-block group at local block cb: matrix 1 in box sw (matrix 3,
      // SwiGLU, in the box after it)
      auto compute8 = [&](const uint8_t *sw, int cb, int nb) {
        if constexpr (FMT == 1) {
          const uint4 n1 = *reinterpret_cast<const uint4 *>(pn1 + cb);
          uint4 n3 = n1;
          if constexpr (NMAT == 2) n3 = *reinterpret_cast<const uint4 *>(pn3 + cb);
          // the eight chunks' scale pairs {s_g, s_g+8} as f16x2
          const uint2 f1a = e4m3x4_to_f16x2x2(n1.x), f1b = e4m3x4_to_f16x2x2(n1.y),
                      f1c = e4m3x4_to_f16x2x2(n1.z), f1d = e4m3x4_to_f16x2x2(n1.w);
          const uint32_t f1[8] = {f1a.x, f1a.y, f1b.x, f1b.y, f1c.x, f1c.y, f1d.x, f1d.y};
          uint32_t f3[8] = {f1[0], f1[1], f1[2], f1[3], f1[4], f1[5], f1[6], f1[7]};
          if constexpr (NMAT == 2) {
            const uint2 a = e4m3x4_to_f16x2x2(n3.x), b = e4m3x4_to_f16x2x2(n3.y),
                        c = e4m3x4_to_f16x2x2(n3.z), d = e4m3x4_to_f16x2x2(n3.w);
            f3[0] = a.x; f3[1] = a.y; f3[2] = b.x; f3[3] = b.y;
            f3[4] = c.x; f3[5] = c.y; f3[6] = d.x; f3[7] = d.y;
          }
          auto block = [&](int bl) {
            const uint8_t *w = sw + (lane_off ^ (uint32_t)(bl << 4));
            const uint32_t wg = *reinterpret_cast<const uint32_t *>(w);
            const uint32_t wh = *reinterpret_cast<const uint32_t *>(w + 8 * DV_BOXB);
            nv_block(acc1, wg, wh, f1[bl], bx[bl]);
            if constexpr (NMAT == 2) {
              const uint32_t vg = *reinterpret_cast<const uint32_t *>(w + DV_BOX);
              const uint32_t vh = *reinterpret_cast<const uint32_t *>(w + DV_BOX + 8 * DV_BOXB);
              nv_block(acc3, vg, vh, f3[bl], bx[bl]);
            }
          };
          if (nb == 8) {
#pragma unroll
            for (int bl = 0; bl < 8; ++bl) block(bl);
          } else {
#pragma unroll
            for (int bl = 0; bl < 8; ++bl)
              if (bl < nb) block(bl);
          }
          return;
        }
        const uint4 s1a = *reinterpret_cast<const uint4 *>(pr1 + cb);
        const uint4 s1b = *reinterpret_cast<const uint4 *>(pr1 + cb + 4);
        uint4 s3a = s1a, s3b = s1b;
        if constexpr (NMAT == 2) {
          s3a = *reinterpret_cast<const uint4 *>(pr3 + cb);
          s3b = *reinterpret_cast<const uint4 *>(pr3 + cb + 4);
        }
        const uint32_t sp1[8] = {s1a.x, s1a.y, s1a.z, s1a.w, s1b.x, s1b.y, s1b.z, s1b.w};
        const uint32_t sp3[8] = {s3a.x, s3a.y, s3a.z, s3a.w, s3b.x, s3b.y, s3b.z, s3b.w};
        auto block = [&](int bl) {
          const uint8_t *w = sw + (lane_off ^ (uint32_t)(bl << 4));
          const uint32_t wg = *reinterpret_cast<const uint32_t *>(w);
          const uint32_t wh = *reinterpret_cast<const uint32_t *>(w + 8 * DV_BOXB);
          mx_block(acc1, wg, wh, __uint_as_float(sp1[bl] << 16),
                   __uint_as_float(sp1[bl] & 0xffff0000u), bx[bl]);
          if constexpr (NMAT == 2) {
            const uint32_t vg = *reinterpret_cast<const uint32_t *>(w + DV_BOX);
            const uint32_t vh = *reinterpret_cast<const uint32_t *>(w + DV_BOX + 8 * DV_BOXB);
            mx_block(acc3, vg, vh, __uint_as_float(sp3[bl] << 16),
                     __uint_as_float(sp3[bl] & 0xffff0000u), bx[bl]);
          }
        };
        if (nb == 8) {
          // a full group: straight-line code, so the eight blocks' independent
          // MMA chains can be interleaved
#pragma unroll
          for (int bl = 0; bl < 8; ++bl) block(bl);
        } else {
#pragma unroll
          for (int bl = 0; bl < 8; ++bl)
            if (bl < nb) block(bl);
        }
      };
      for (int c = 0; c < nslot; ++c) {
        const int cb = c * SB;
        const int slot = consumed & (DV_STAGES - 1);
        const uint32_t parity = (uint32_t)(consumed / DV_STAGES) & 1u;
        ++consumed;
        if (active) {
          load_bx(cb, min(8, nbl - cb));
          // the next slot's activation lines: one 128-byte line (two blocks)
          // per lane and 8-block group
#pragma unroll
          for (int h = 0; h < SUB; ++h)
            if (c + 1 < nslot && (lane & 3) * 2 < nbl - (cb + SB + 8 * h))
              asm volatile("prefetch.global.L1 [%0];" ::"l"(xpf + (cb + SB + 8 * h) * 32));
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[warp][slot], parity, abort));
          if (!ok) break;
          const uint8_t *st = ring + (size_t)slot * 2 * DV_BOX;
          compute8(st, cb, min(8, nbl - cb));
          if constexpr (SUB == 2) {
            if (nbl - cb > 8) {
              load_bx(cb + 8, min(8, nbl - cb - 8));
              compute8(st + DV_BOX, cb + 8, min(8, nbl - cb - 8));
            }
          }
        } else {
          // a group past the last row: its slots were arrived on without data
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[warp][slot], parity, abort));
          if (!ok) break;
        }
        __syncwarp();
        if (lane == 0) {
          // the slot was read through the generic proxy; order those reads
          // before the TMA engine overwrites it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          issue_next();
        }
      }
      // partial sums of the group's warps, added in warp order.  Two splits:
      // each warp finishes one row (split 0 row g, split 1 row g + 8) and hands
      // the other row's sums to its partner.  More splits: the first warp
      // finishes both rows.
      float *rb = red + (size_t)(npass & 1) * DV_WARPS * RV * 32;
      float f1[2], f3[2];   // this warp's finished values: tokens 2t, 2t+1 of its row
      int frow;
      bool fin;
      if constexpr (KS == 2) {
        const bool s0 = split == 0;
        // kept: this warp's row; given: the partner's row
        const float k10 = s0 ? acc1[0] : acc1[2], k11 = s0 ? acc1[1] : acc1[3];
        const float k30 = s0 ? acc3[0] : acc3[2], k31 = s0 ? acc3[1] : acc3[3];
        rb[(warp * RV + 0) * 32 + lane] = s0 ? acc1[2] : acc1[0];
        rb[(warp * RV + 1) * 32 + lane] = s0 ? acc1[3] : acc1[1];
        rb[(warp * RV + 2) * 32 + lane] = s0 ? acc3[2] : acc3[0];
        rb[(warp * RV + 3) * 32 + lane] = s0 ? acc3[3] : acc3[1];
        if (group_sync_or(grp, 32 * KS, !ok)) { ok = false; break; }
        const int pw_ = warp ^ 1;
        // warp order: split 0's sum first
        const float o10 = rb[(pw_ * RV + 0) * 32 + lane], o11 = rb[(pw_ * RV + 1) * 32 + lane];
        const float o30 = rb[(pw_ * RV + 2) * 32 + lane], o31 = rb[(pw_ * RV + 3) * 32 + lane];
        f1[0] = s0 ? k10 + o10 : o10 + k10;
        f1[1] = s0 ? k11 + o11 : o11 + k11;
        f3[0] = s0 ? k30 + o30 : o30 + k30;
        f3[1] = s0 ? k31 + o31 : o31 + k31;
        frow = s0 ? g : g + 8;
        fin = active;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          rb[(warp * RV + q) * 32 + lane] = acc1[q];
          rb[(warp * RV + 4 + q) * 32 + lane] = acc3[q];
        }
        if (group_sync_or(grp, 32 * KS, !ok)) { ok = false; break; }
        // the first warp finishes row g, the second row g + 8
        fin = active && split < 2;
        const int q0 = split == 1 ? 2 : 0;
        f1[0] = f1[1] = f3[0] = f3[1] = 0.f;
        if (fin) {
#pragma unroll
          for (int w = 0; w < KS; ++w) {
            const int ww = grp * KS + w;
            f1[0] += rb[(ww * RV + q0) * 32 + lane];
            f1[1] += rb[(ww * RV + q0 + 1) * 32 + lane];
            f3[0] += rb[(ww * RV + 4 + q0) * 32 + lane];
            f3[1] += rb[(ww * RV + 4 + q0 + 1) * 32 + lane];
          }
        }
        frow = split == 1 ? g + 8 : g;
      }
      if (PAIRED && fin) {
        // rows r0 + frow (f1) and r0 + 16 + frow (f3)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tk = tg + 2 * t + q;
          if (tk < cnt) {
            a.out[(size_t)(beg + tk) * R + r0 + frow] = __float2bfloat16_rn(f1[q] * gs1);
            a.out[(size_t)(beg + tk) * R + r0 + 16 + frow] = __float2bfloat16_rn(f3[q] * gs3);
          }
        }
      } else if (fin) {
        const int row = r0 + frow;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float v;
          const float a1 = f1[q] * gs1, a3 = f3[q] * gs3;   // NVFP4 matrix scales (else 1)
          if constexpr (EPI == 2) v = a1 / (1.f + __expf(-a1)) * a3;
          else if constexpr (EPI == 1) v = fmaxf(a1, 0.f);
          else v = a1;
          const int tk = tg + 2 * t + q;
          if (tk < cnt && row < R) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(v);
            a.out[(size_t)(beg + tk) * R + row] = hb;
            if (a.out16)
              a.out16[(size_t)(beg + tk) * R + row] =
                  f16_bits_checked(__bfloat162float(hb), a.status, beg + tk);
          }
        }
      }
    }
    if (!ok) break;
  }
  if (!ok) {
    // let the copies this warp issued land before it exits
    if (lane == 0) {
      for (int j = consumed; j < P.issued; ++j)
        tc::mbar_wait_drain(&full[warp][j % DV_STAGES], (uint32_t)(j / DV_STAGES) & 1u,
                            100000000ull);
      if (raw_mine0 >= 0)
        tc::mbar_wait_drain(&sbar[0], (uint32_t)((raw_mine0 / NRAW) & 1), 100000000ull);
      if (raw_mine1 >= 0)
        tc::mbar_wait_drain(&sbar[1], (uint32_t)((raw_mine1 / NRAW) & 1), 100000000ull);
      set_status(a.status, MOE_ERR_TIMEOUT, blockIdx.x);
    }
  }
}

template <int EPI, int RG, bool POOL, int FMT>
cudaError_t launch_one(DecodeArgs a, const uint8_t *W, const uint8_t *W3, const uint8_t *PW,
                       const uint8_t *PW3, int num_experts, int slots, cudaStream_t s) {
  constexpr int NMAT = (EPI == 2 || EPI == 3) ? 2 : 1;
  constexpr int GROWS = (EPI == 3) ? 32 : 16;
  const size_t smem = 1024 + decode_plan(NMAT, a.K, RG, FMT).bytes;
  static size_t smem_set = 0;
  static int per_sm = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_mxfp4_kernel<EPI, RG, POOL, FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
    per_sm = 0;
  }
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mxfp4_kernel<EPI, RG, POOL, FMT>,
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
  if (EPI == 2) {
    if (!make_tensor_map(&m3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, W3, 2, dims, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    m3 = m1;
  }
  // the pool's codes, [n_slots * R] rows of the same layout
  CUtensorMap p1 = m1, p3 = m3;
  if (POOL) {
    const uint64_t pdims[2] = {(uint64_t)a.K / 2, (uint64_t)a.n_slots * a.R};
    if (!make_tensor_map(&p1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, PW, 2, pdims, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (EPI == 2 && !make_tensor_map(&p3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, PW3, 2, pdims, box,
                                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // units: at most `slots` experts x row blocks; no more CTAs than units
  const long units = (long)slots * ((a.R + GROWS * RG - 1) / (GROWS * RG));
  long grid = (long)per_sm * num_sms();
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  return launch_pdl(decode_mxfp4_kernel<EPI, RG, POOL, FMT>, dim3((unsigned)grid), dim3(32 * DV_WARPS),
                    smem, s, m1, m3, p1, p3, a);
}

// Rows per work unit: 64 (four 16-row groups, two reduction splits each)
// where that still gives every resident CTA a unit, else 32, else 16.
// Every configuration's shared memory stays within two CTAs per SM.  Longer
// units spread the per-unit costs (scale decoding, the partial-sum exchange,
// the epilogue) over more weight bytes.
template <int EPI, bool POOL, int FMT>
cudaError_t launch_rg(DecodeArgs a, const uint8_t *W, const uint8_t *W3, const uint8_t *PW,
                      const uint8_t *PW3, int num_experts, int slots, cudaStream_t s) {
  const long ctas = 2L * num_sms();
  constexpr int GROWS = (EPI == 3) ? 32 : 16;
  auto units = [&](int rg) { return (long)slots * ((a.R + GROWS * rg - 1) / (GROWS * rg)); };
  // (NVFP4 units stop at 32 rows: their scale bytes double, and 64-row units
  // would not fit two CTAs per SM)
  if constexpr (FMT == 0)
    if (units(4) >= ctas)
      return launch_one<EPI, 4, POOL, FMT>(a, W, W3, PW, PW3, num_experts, slots, s);
  if (units(2) >= ctas)
    return launch_one<EPI, 2, POOL, FMT>(a, W, W3, PW, PW3, num_experts, slots, s);
  return launch_one<EPI, 1, POOL, FMT>(a, W, W3, PW, PW3, num_experts, slots, s);
}

// Both projections of the small-batch FFN (see launch_decode_ffn); POOL: the
// kernels read resident experts from pool's slots.
template <bool POOL, int FMT>
cudaError_t run_decode_ffn(const moe_config &c, int part, const void *act, const int32_t *perm,
                           const int32_t *offsets, const moe_weights &w, void *h, void *y_perm,
                           void *act16, int *status, cudaStream_t s, const moe_expert_pool *pool) {
  const int P = c.n * c.top_k;
  const int slots = P < c.n_experts ? P : c.n_experts;
  uint16_t *x16 = static_cast<uint16_t *>(act16);
  uint16_t *h16 = x16 + (size_t)P * c.d;
  DecodeArgs a{};
  a.offsets = offsets;
  a.num_experts = c.n_experts;
  a.P = P;
  a.status = status;
  a.top_k = c.top_k;
  if (POOL) {
    a.slot_of = pool->slot_of;
    a.n_slots = pool->n_slots;
  }
  if (part == 0) {
    if (act != nullptr) {
      cudaError_t e = launch_rows_to_f16(act, perm, c.top_k, P, c.d, x16, status, s);
      if (e != cudaSuccess) return e;
    } else {
      a.perm = perm;   // x16 holds the x rows in token order
    }
    a.act16 = x16;
    a.S = w.S1;
    a.S3 = w.S3;
    a.PS = pool ? pool->S1 : nullptr;
    a.PS3 = pool ? pool->S3 : nullptr;
    a.G = w.G1;
    a.G3 = w.G3;
    a.R = c.d_ff;
    a.K = c.d;
    a.out = static_cast<__nv_bfloat16 *>(h);
    a.out16 = h16;
    const uint8_t *W1 = static_cast<const uint8_t *>(w.W1), *W3 = static_cast<const uint8_t *>(w.W3);
    const uint8_t *P1 = pool ? static_cast<const uint8_t *>(pool->W1) : nullptr;
    const uint8_t *P3 = pool ? static_cast<const uint8_t *>(pool->W3) : nullptr;
    return c.act == MOE_ACT_SWIGLU ? launch_rg<2, POOL, FMT>(a, W1, W3, P1, P3, c.n_experts, slots, s)
                                   : launch_rg<1, POOL, FMT>(a, W1, nullptr, P1, nullptr, c.n_experts, slots, s);
  }
  a.act16 = h16;
  a.S = w.S2;
  a.S3 = nullptr;
  a.PS = pool ? pool->S2 : nullptr;
  a.PS3 = nullptr;
  a.G = w.G2;
  a.G3 = nullptr;
  a.R = c.d;
  a.K = c.d_ff;
  a.out = static_cast<__nv_bfloat16 *>(y_perm);
  a.out16 = nullptr;
  // The down projection's rows (d) are a multiple of 32.  Paired 32-row
  // groups load each activation fragment once for two rows' MMAs; they pay
  // off once there are at least two 128-row units per resident CTA (measured
  // on the gpt-oss shape: n = 64 128 -> 113 us, n = 16 65 -> 59 us; at n = 4
  // the coarser units balance worse and single groups stay ahead).
  const uint8_t *W2 = static_cast<const uint8_t *>(w.W2);
  const uint8_t *P2 = pool ? static_cast<const uint8_t *>(pool->W2) : nullptr;
  const long paired_units = (long)slots * ((a.R + 127) / 128);
  if (paired_units >= 4L * num_sms())
    return launch_rg<3, POOL, FMT>(a, W2, nullptr, P2, nullptr, c.n_experts, slots, s);
  return launch_rg<0, POOL, FMT>(a, W2, nullptr, P2, nullptr, c.n_experts, slots, s);
}

}  // namespace
}  // namespace moe
