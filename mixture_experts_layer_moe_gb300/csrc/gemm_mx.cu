// MXFP4 grouped GEMM on the 5th-generation tensor cores, weights as the A
// operand in tensor memory.
//
// "How Mixture of Experts Scales Model Parameters": each expert's FFN runs on
// the rows routed to it (sections "Sparse models" and "The forward pass:
// dispatch, then combine"); weights are MXFP4 (feed post "What is MXFP4?": 4-bit
// elements in blocks of 32 sharing one scale; E2M1 / E8M0 bits per the OCP MX
// v1.0 format).
//
// A tile computes D[w][t] = sum_k W[w][k] * X[t][k] for 128 weight rows w (MMA
// M, the TMEM lanes) and up to 128 tokens t of one expert's segment (MMA N),
// i.e. the transposed output tile.  N is the segment's remaining token count
// rounded up to 16, so a small expert costs a small MMA instead of a padded
// one.  The token rows (f16 copies of the activations) come by TMA into a
// 128-byte-swizzled shared-memory tile, the B operand.  The weights never
// touch shared memory in f16: four transform warps read the packed codes (TMA,
// 32-byte swizzle), convert each row's 64 codes of a k-block with
// cvt.rn.f16x2.e2m1x2, multiply by the block's E8M0 scale as an f16 pair
// (exact for scale bytes 113..142; others are reported as MOE_ERR_RANGE) and
// write them with tcgen05.st into an A stage in tensor memory (lane = weight
// row, 32-bit column c = k-elements 2c and 2c + 1).
//
// Two CTAs share each SM, each with half of its tensor memory: a 128-column
// accumulator and GS A stages.  One CTA's ring (TMA -> transform -> MMA ->
// release) is latency-bound; the other CTA's MMAs fill the tensor pipe while
// it waits (measured on the Zipf-routed prefill, n = 8192: down projection
// 0.50 ms, against 0.77 ms for one CTA per SM with a double-buffered
// accumulator and 0.53 ms for one CTA per SM with 256-token tiles).  The single accumulator is drained into registers
// (bf16 pairs) and released to the next tile's MMAs before the epilogue
// writes to global memory.
//
// Epilogues: 0 y = X W^T; 1 h = relu(X W^T); 2 SwiGLU over 64 output columns,
// h = silu(X W1^T) * (X W3^T): in each 32-lane quarter of the tile, lanes
// 0..15 hold 16 rows of W1 and lanes 16..31 the same 16 rows of W3, so one
// shuffle between the half-warps brings each gate value next to its up value
// (each half then finishes half of the tokens).
//
// Warp roles (persistent, two CTAs per SM): 0 TMA producer, 1 MMA issuer and
// TMEM owner, 2-5 epilogue (one per TMEM lane quarter), 6-9 transform.  TMEM
// (256 columns per CTA): the accumulator, then GS stages of 32 columns of A.
#include "common.cuh"
#include "launch.h"
#include "mx_common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace mx;

constexpr int GM = 128;                         // weight rows per tile (MMA M)
constexpr int GN = 128;                         // tokens per tile at most (MMA N)
constexpr int GK = 64;                          // k-block
constexpr int GS = 4;                           // pipeline stages
constexpr int G_B_BYTES = GN * GK * 2;          // token tile: 16 KB
constexpr int G_C_BYTES = GM * GK / 2;          // codes of the k-block: 4 KB
constexpr int G_STAGE = G_B_BYTES + G_C_BYTES;  // 20 KB
constexpr int G_XFORM = 4;                      // transform warps
constexpr int G_EPI = 4;                        // epilogue warps
constexpr int G_THREADS = 32 * (2 + G_EPI + G_XFORM);
constexpr uint32_t G_TMEM_COLS = 256;           // two CTAs per SM
constexpr uint32_t G_A_COL0 = GN;               // A stages after the accumulator
constexpr int G_MAX_E = 256;
constexpr int G_BAR_XFORM = 3;                  // named barrier: transform agreement
static_assert(G_A_COL0 + GS * (GK / 2) <= G_TMEM_COLS, "tensor memory columns");
static_assert(G_STAGE % 1024 == 0, "stage alignment");

struct GShared {
  uint64_t full[GS], empty[GS], aready[GS];
  uint64_t tfull, tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort, failed_on_entry, num_tiles;
  int offs[G_MAX_E + 1];
  int tile_start[G_MAX_E];
};

struct GArgs {
  const int32_t *offsets;
  int num_experts, rows, K, N;
  const uint8_t *S;          // E8M0 scales [E][N][K/32] (W1's for SwiGLU)
  const uint8_t *S3;         // SwiGLU: W3's scales (else S)
  __nv_bfloat16 *out;        // [rows][N]
  uint16_t *out16;           // f16 copy of out, or nullptr
  int *status;
};

struct GTile {
  int e, row0, seg_end, n_idx;
};

__device__ __forceinline__ GTile g_decode(const GShared &sh, int E, int t) {
  int lo = 0, hi = E;   // largest e with tile_start[e] <= t (skips empty experts)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  GTile tl;
  tl.e = lo;
  const int beg = sh.offs[lo], end = sh.offs[lo + 1];
  const int m_tiles = (end - beg + GN - 1) / GN;
  const int local = t - sh.tile_start[lo];
  tl.n_idx = local / m_tiles;                  // token blocks fastest: neighbours share weights
  tl.row0 = beg + (local - tl.n_idx * m_tiles) * GN;
  tl.seg_end = end;
  return tl;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (f16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__host__ __device__ inline size_t g_scale_pitch(int K) {
  return ((size_t)GM * (K / 32) + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t g_scale_off() { return (size_t)GS * G_STAGE; }
size_t g_dyn_smem(int K) { return 1024 + g_scale_off() + 2 * g_scale_pitch(K); }

template <int EPI>
__global__ void __launch_bounds__(G_THREADS, 2)
gemm_mx_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ CUtensorMap tmW3, GArgs args) {
  constexpr int N_OUT = (EPI == 2) ? GM / 2 : GM;   // output columns per tile
  extern __shared__ uint8_t dyn_smem[];
  __shared__ GShared sh;
  uint8_t *smem = dyn_smem + ((1024 - (tc::smem_u32(dyn_smem) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.num_experts;
  const int n_tiles = (args.N + N_OUT - 1) / N_OUT;
  const int KB = args.K / GK;
  const int KBLK = args.K / 32;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    // the tensor maps are kernel parameters: fetch them while the previous
    // kernel finishes
    tc::prefetch_tmap(&tmX);
    tc::prefetch_tmap(&tmW);
    if (EPI == 2) tc::prefetch_tmap(&tmW3);
  }
  pdl_wait();
  if (threadIdx.x == 0) {
    sh.failed_on_entry = status_failed(args.status) ? 1 : 0;
    sh.abort = sh.failed_on_entry;
  }
  for (int i = threadIdx.x; i <= E; i += G_THREADS) sh.offs[i] = args.offsets[i];
  if (warp == 1) tc::tmem_alloc(&sh.tmem_base, G_TMEM_COLS);
  if (threadIdx.x == 32) {
    for (int s = 0; s < GS; ++s) {
      tc::mbar_init(&sh.full[s], 1);
      tc::mbar_init(&sh.empty[s], 1 + G_XFORM);   // the MMAs (token tile), the transform (codes)
      tc::mbar_init(&sh.aready[s], G_XFORM);
    }
    tc::mbar_init(&sh.tfull, 1);
    tc::mbar_init(&sh.tempty, G_EPI);
    tc::mbar_init(&sh.drain, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    // tile prefix over experts: lane l owns experts 8l .. 8l+7
    int cnt[8];
    int sum = 0, bad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      cnt[i] = 0;
      if (e < E) {
        const int b = sh.offs[e], en = sh.offs[e + 1];
        if (b < 0 || en < b || en > args.rows) bad = 1;
        else cnt[i] = ((en - b + GN - 1) / GN) * n_tiles;
      }
      sum += cnt[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) sh.tile_start[e] = run;
      run += cnt[i];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      sh.num_tiles = bad ? 0 : total;
      if (bad) set_status(args.status, MOE_ERR_BAD_INDEX, -1);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = sh.tmem_base;
  const int num_tiles = sh.num_tiles;
  volatile int *abort = &sh.abort;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: the tile's token boxes + the k-block's
      // codes of weight rows 0..63 and 64..127 (W1 and W3 rows for SwiGLU)
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[GS];
#pragma unroll
      for (int s = 0; s < GS; ++s) last_phase[s] = -1;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const GTile tl = g_decode(sh, E, t);
        const int r_lo = tl.n_idx * N_OUT;
        const int r_hi = (EPI == 2) ? r_lo : r_lo + GM / 2;
        const bool hi_ok = EPI == 2 && r_hi < args.N;  // SwiGLU: the W3 box
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&sh.empty[stage], phase ^ 1u, abort)) break;
          uint8_t *sb = smem + stage * G_STAGE;
          uint8_t *sc = sb + G_B_BYTES;
          tc::mbar_arrive_expect_tx(&sh.full[stage], (uint32_t)(G_B_BYTES + G_C_BYTES));
          tc::tma_load_2d(&tmX, &sh.full[stage], sb, kb * GK, tl.row0);
          tc::tma_load_3d(&tmW, &sh.full[stage], sc, kb * (GK / 2), r_lo, tl.e);
          if (hi_ok)
            tc::tma_load_3d(EPI == 2 ? &tmW3 : &tmW, &sh.full[stage], sc + G_C_BYTES / 2,
                            kb * (GK / 2), r_hi, tl.e);
          last_phase[stage] = (int)phase;
          if (++stage == GS) { stage = 0; phase ^= 1u; }
        }
      }
      if (*abort) {
        for (int s = 0; s < GS; ++s)
          if (last_phase[s] >= 0)
            tc::mbar_wait_drain(&sh.full[s], (uint32_t)last_phase[s], 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: D = A(TMEM, weights) x B(smem, tokens)^T
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok && !*abort; t += gridDim.x, ++local) {
        const GTile tl = g_decode(sh, E, t);
        const int ntok = min(GN, tl.seg_end - tl.row0);
        const uint32_t idesc = tc::idesc_f16_f32(GM, (ntok + 15) & ~15);
        if (!tc::mbar_wait(&sh.tempty, (local & 1) ^ 1u, abort)) { ok = false; break; }
        tc::tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          // one wait per k-block: every transform thread waited for the
          // stage's full barrier (its token box and codes land together)
          // before arriving on aready, so aready's phase implies the tokens
          if (!tc::mbar_wait(&sh.aready[stage], phase, abort)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t sb = tc::smem_u32(smem + stage * G_STAGE);
          const uint32_t a_tmem = tmem_base + G_A_COL0 + (uint32_t)(stage * (GK / 2));
#pragma unroll
          for (int k = 0; k < GK / 16; ++k)
            mma_ta(tmem_base, a_tmem + k * 8, tc::smem_desc_sw128(sb + k * 32), idesc,
                   (kb != 0 || k != 0) ? 1u : 0u);
          tc::mma_commit(&sh.empty[stage]);
          if (++stage == GS) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc::mma_commit(&sh.tfull);
      }
      if (*abort) {
        tc::mma_commit(&sh.drain);
        tc::mbar_wait_drain(&sh.drain, 0, 100000000ull);
      }
    }
  } else if (warp < 2 + G_EPI) {
    // ---------------- epilogue: warp w drains TMEM lanes 32*(w%4) .. +31, 32
    // tokens per chunk, into bf16 pairs held in registers; the accumulator is
    // then released and each thread writes its output column for its tokens
    // (a warp's stores of one token are 64 contiguous bytes, 2 x 32 for SwiGLU)
    const int quarter = warp & 3;
    const bool low = lane < 16;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const GTile tl = g_decode(sh, E, t);
      const int ntok = min(GN, tl.seg_end - tl.row0);
      const bool ok = tc::mbar_wait(&sh.tfull, local & 1, abort);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::tc_fence_after();
      // bf16 pairs: packed[c][q] = tokens 2q, 2q+1 of chunk c (SwiGLU: of the
      // lane's 16 tokens of the chunk, q < 8)
      uint32_t packed[4][EPI == 2 ? 8 : 16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col0 = c * 32;
        if (col0 < ntok) {
          if constexpr (EPI == 2) {
            uint32_t a[32];
            tc::tmem_ld32(lane_base + (uint32_t)col0, a);
            tc::tmem_ld_wait();
            // low lane: gate values g[0..31] of its row; high lane: up values
            // u[0..31] of the same row.  The low lane takes tokens 0..15, the
            // high lane tokens 16..31.
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const uint32_t s0 = __shfl_xor_sync(0xffffffffu, low ? a[16 + i] : a[i], 16);
              const uint32_t s1 = __shfl_xor_sync(0xffffffffu, low ? a[17 + i] : a[i + 1], 16);
              const float g0 = __uint_as_float(low ? a[i] : s0);
              const float u0 = __uint_as_float(low ? s0 : a[16 + i]);
              const float g1 = __uint_as_float(low ? a[i + 1] : s1);
              const float u1 = __uint_as_float(low ? s1 : a[17 + i]);
              packed[c][i >> 1] = pack_bf16x2(silu_mul(g0, u0), silu_mul(g1, u1));
            }
          } else {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t a[16];
              tmem_ld16(lane_base + (uint32_t)(col0 + 16 * hh), a);
              tc::tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                float v0 = __uint_as_float(a[2 * i]), v1 = __uint_as_float(a[2 * i + 1]);
                if constexpr (EPI == 1) {
                  v0 = fmaxf(v0, 0.f);
                  v1 = fmaxf(v1, 0.f);
                }
                packed[c][8 * hh + i] = pack_bf16x2(v0, v1);
              }
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sh.tempty);
      constexpr int PER = (EPI == 2) ? 16 : 32;         // tokens per thread per chunk
      const int col = (EPI == 2) ? tl.n_idx * N_OUT + quarter * 16 + (lane & 15)
                                 : tl.n_idx * N_OUT + quarter * 32 + lane;
      const int tsub = (EPI == 2 && !low) ? 16 : 0;
      if (col < args.N) {
        uint16_t *o = reinterpret_cast<uint16_t *>(args.out);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c * 32 < ntok) {
            const int tok0 = tl.row0 + c * 32 + tsub;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
              const int tok = tok0 + i;
              if (tok < tl.seg_end) {
                const uint32_t hb = (i & 1) ? (packed[c][i >> 1] >> 16)
                                            : (packed[c][i >> 1] & 0xffffu);
                o[(size_t)tok * args.N + col] = (uint16_t)hb;
                if (args.out16)
                  args.out16[(size_t)tok * args.N + col] =
                      f16_bits_checked(__uint_as_float(hb << 16), args.status, tok);
              }
            }
          }
        }
      }
    }
  } else {
    // ---------------- transform: warp w writes TMEM lanes 32*(w%4) .. +31, one
    // weight row per thread.  A tile's scales are copied (cp.async) into one
    // of two buffers while the previous tile runs.  The codes arrive with a
    // 32-byte swizzle: 16-byte half c of row r sits at c ^ ((r >> 2) & 1).
    const int quarter = warp & 3;
    // this thread's TMEM lane and the row of the codes / scales tile feeding it
    // (SwiGLU: lanes 16..31 of a quarter take W3 rows, held in tile rows 64..127)
    const int r = quarter * 32 + lane;
    const int crow = (EPI == 2) ? (lane < 16 ? quarter * 16 + lane : GM / 2 + quarter * 16 + lane - 16)
                                : r;
    const int tt = threadIdx.x - 32 * (2 + G_EPI);     // 0 .. 127
    constexpr int XT = 32 * G_XFORM;
    const size_t spitch = g_scale_pitch(args.K);
    uint8_t *scale_buf[2] = {smem + g_scale_off(), smem + g_scale_off() + spitch};
    // scales of tile rows 0..63 and 64..127 (rows past N are left unset: their
    // codes are zero-filled by TMA and their columns are never stored)
    auto fetch_scales = [&](int t, int b) {
      const GTile tl = g_decode(sh, E, t);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int wrow = (EPI == 2) ? tl.n_idx * N_OUT : tl.n_idx * N_OUT + h * (GM / 2);
        const uint8_t *S = (EPI == 2 && h == 1) ? args.S3 : args.S;
        const int rows = max(0, min(GM / 2, args.N - wrow));
        const size_t bytes = (size_t)rows * KBLK;       // a multiple of 16
        const uint8_t *src = S + ((size_t)tl.e * args.N + wrow) * KBLK;
        uint8_t *dst = scale_buf[b] + (size_t)h * (GM / 2) * KBLK;
        for (size_t o = (size_t)tt * 16; o < bytes; o += XT * 16) cp_async16(dst + o, src + o);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    bool bad_scale = false;
    const int sw = ((crow >> 2) & 1) << 4;
    const uint32_t a_lane = tmem_base + ((uint32_t)(quarter * 32) << 16) + G_A_COL0;
    if (blockIdx.x < num_tiles) fetch_scales(blockIdx.x, 0);
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, buf ^= 1) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
      // this tile's scales are in; the transform warps also agree here on
      // stopping (a warp whose wait ran out has raised *abort)
      if (tc::bar_or(G_BAR_XFORM, XT, *abort != 0)) break;
      if (t + (int)gridDim.x < num_tiles) fetch_scales(t + gridDim.x, buf ^ 1);
      const uint8_t *srow = scale_buf[buf] + (size_t)crow * KBLK;
      const GTile tl = g_decode(sh, E, t);
      const int wrow = tl.n_idx * N_OUT + (crow & (GM / 2 - 1)) + (EPI == 2 ? 0 : (crow & (GM / 2)));
      const bool row_ok = wrow < args.N;              // else: zero row
      for (int kb = 0; kb < KB; ++kb) {
        const bool ok = tc::mbar_wait(&sh.full[stage], phase, abort);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint8_t *codes = smem + stage * G_STAGE + G_B_BYTES + crow * 32;
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        if (row_ok) {
          c0 = *reinterpret_cast<const uint4 *>(codes + sw);
          c1 = *reinterpret_cast<const uint4 *>(codes + (sw ^ 16));
        }
        // the codes are in registers: this warp is done with the stage's codes
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh.empty[stage]);
        uint32_t v[32];
        if (row_ok) {
          const uint32_t f0 = scale_f16x2(srow[2 * kb], bad_scale);
          const uint32_t f1 = scale_f16x2(srow[2 * kb + 1], bad_scale);
          const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const uint32_t f = w < 4 ? f0 : f1;
            const uint4 q = e2m1x8_to_f16x2x4(words[w]);
            v[4 * w] = hmul2(q.x, f);
            v[4 * w + 1] = hmul2(q.y, f);
            v[4 * w + 2] = hmul2(q.z, f);
            v[4 * w + 3] = hmul2(q.w, f);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        // the stage's A columns are free: the MMAs that read them completed
        // before the producer refilled this stage
        tmem_st32(a_lane + (uint32_t)(stage * (GK / 2)), v);
        tmem_st_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sh.aready[stage]);
        if (++stage == GS) { stage = 0; phase ^= 1u; }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (bad_scale) set_status(args.status, MOE_ERR_RANGE, 0);
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, G_TMEM_COLS);
  }
  if (threadIdx.x == 0 && sh.abort && !sh.failed_on_entry)
    set_status(args.status, MOE_ERR_TIMEOUT, blockIdx.x);
}

template <int EPI>
cudaError_t launch_mx(const GemmStage &g, int *status, cudaStream_t s) {
  const size_t smem = g_dyn_smem(g.K);
  static size_t smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_mx_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  CUtensorMap mX, mW, mW3;
  const uint64_t dX[2] = {(uint64_t)g.K, (uint64_t)g.rows};
  const uint32_t bX[2] = {GK, GN};
  if (!make_tensor_map(&mX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.A, 2, dX, bX,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // packed codes: [E][N][K/2] bytes, boxes of 32 bytes (one k-block) x 64 rows
  const uint64_t dC[3] = {(uint64_t)g.K / 2, (uint64_t)g.N, (uint64_t)g.num_experts};
  const uint32_t bC[3] = {GK / 2, (uint32_t)(EPI == 2 ? GM / 2 : GM), 1};
  if (!make_tensor_map(&mW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.B, 3, dC, bC,
                       CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  if (EPI == 2) {
    if (!make_tensor_map(&mW3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.B3, 3, dC, bC,
                         CU_TENSOR_MAP_SWIZZLE_32B))
      return cudaErrorInvalidValue;
  } else {
    mW3 = mW;
  }
  GArgs a{};
  a.offsets = g.offsets;
  a.num_experts = g.num_experts;
  a.rows = g.rows;
  a.K = g.K;
  a.N = g.N;
  a.S = g.SB;
  a.S3 = (EPI == 2) ? g.SB3 : g.SB;
  a.out = static_cast<__nv_bfloat16 *>(g.out);
  a.out16 = static_cast<uint16_t *>(g.out16);
  a.status = status;
  return launch_pdl(gemm_mx_kernel<EPI>, dim3(2 * num_sms()), dim3(G_THREADS), smem, s, mX, mW, mW3,
                    a);
}

}  // namespace

// Shapes only: the callers pass 16-byte-aligned code and scale arrays.
bool gemm_mx_supported(const GemmStage &g) {
  return g.rows > 0 && tensor_maps_available() && g.b_dtype == MOE_MXFP4 && g.a_dtype == kF16 &&
         g.out_dtype == MOE_BF16 && (g.epi == 0 || g.epi == 1 || g.epi == 2) &&
         g.offsets != nullptr && g.num_experts <= G_MAX_E && g.K % GK == 0 && g.N % 32 == 0 &&
         g_dyn_smem(g.K) + sizeof(GShared) <= 113 * 1024;   // two CTAs per SM
}

cudaError_t launch_gemm_mx(const GemmStage &g, int *status, cudaStream_t s) {
  switch (g.epi) {
    case 1: return launch_mx<1>(g, status, s);
    case 2: return launch_mx<2>(g, status, s);
    default: return launch_mx<0>(g, status, s);
  }
}

}  // namespace moe
