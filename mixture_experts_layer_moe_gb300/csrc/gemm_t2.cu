// Grouped expert GEMM on a pair of SMs (tcgen05.mma.cta_group::2), weights on
// the MMA's M side and tokens on its N side.
//
// Each expert runs its FFN projection on its own dispatched segment ("How
// Mixture of Experts Scales Model Parameters", sections "Dense models" and
// "The forward pass: dispatch, then combine"):
//   out[q][j] = epi( sum_i A[q][i] * W_e[j][i] )   for q in segment e,
// computed as the transposed tile D[j][q] = sum_i W_e[j][i] * A[q][i]: 256
// weight rows j (MMA M, 128 in each CTA of a two-CTA cluster, one per TMEM
// lane) by up to 256 tokens q of the segment (MMA N: a segment splits into
// blocks of nearly equal size, rounded up to 16, so that a ragged segment
// costs MMAs as wide as its tokens and no tile is a thin remainder).  SwiGLU
// fuses h = silu(A W1^T) * (A W3^T) in the epilogue.
//
// Why a CTA pair: with M = 256 split over two SMs and the token tile split
// along N (each CTA stages half of the token rows, the MMA reads both halves),
// each SM stages 16 KB of weights and 16 KB of tokens per 64-wide k-block for
// a 128 x 256 x 64 share of the product, against 48 KB for the same share on
// one SM with a 128 x 256 tile: a third less shared-memory and L2 traffic per
// MMA cycle.
//
// Roles (persistent, one CTA per SM, clusters of two):
//   warp 0     TMA producer in both CTAs: this CTA's 128 weight rows and its
//              half of the token rows per stage (128-byte swizzle, 6 stages);
//              every copy signals the stage barrier of the pair's first CTA
//              (cp.async.bulk.tensor .cta_group::2), whose producer expects the
//              bytes of both.
//   warp 1     allocates 512 TMEM columns in both CTAs (cta_group::2); in the
//              first CTA one thread issues the MMAs (M 256, N <= 256, K 16) into
//              two accumulators of 256 columns and commits to the barriers of
//              both CTAs at once (multicast arrive).
//   warps 2-5  epilogue in both CTAs: each drains its own TMEM lanes, applies
//              the activation, rounds to bf16 and stores the rows masked to the
//              segment, then arrives (remotely, for the second CTA) on the
//              first CTA's accumulator-empty barrier.
// For SwiGLU, a CTA's 128 weight rows are 64 rows of W1 (TMEM lanes 0..63)
// and the same 64 rows of W3 (lanes 64..127), each one 64-row TMA box (eight
// 16-row boxes interleaving them per lane quarter measured 29 % slower: the
// copy engine's cost grows with the number of boxes).  The epilogue warp of
// lane quarter q (W1) and that of quarter q + 2 (W3) then trade half of each
// 32-token chunk through shared memory, so each finishes 16 tokens with the
// gate value and the up value side by side; a tile has 128 output columns (64
// per CTA), otherwise 256 (128 per CTA).
//
// Tiles are ordered expert-major, then weight block, then token block, so the
// clusters running together share one expert's weight block and segment in
// L2 (token block, then weight block, when a segment outweighs its weights).
// Pair p takes tiles p, p + pairs, ...  (An atomic tile counter, which kept
// the pairs sharing a weight block in step and cut the fine-grained up
// projection's DRAM reads from 22.4 to 18.0 GB, measured 5-7 % slower.)  The
// tile list comes from the segment offsets on the device; empty segments give
// no tiles.
#include "common.cuh"
#include "launch.h"
#include "pair_common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace pair;

constexpr int PM = 128;                         // weight rows per CTA (MMA M = 256 per pair)
constexpr int PN = 256;                         // tokens per tile at most (MMA N)
constexpr int PK = 64;                          // k-block
constexpr int PS = 6;                           // pipeline stages
constexpr int P_B_BYTES = (PN / 2) * PK * 2;    // this CTA's half of the token tile: 16 KB
constexpr int P_A_BYTES = PM * PK * 2;          // this CTA's weight rows: 16 KB
constexpr int P_STAGE = P_B_BYTES + P_A_BYTES;  // 32 KB (tokens first, then weights)
constexpr int P_EPI = 4;                        // epilogue warps
constexpr int P_THREADS = 32 * (2 + P_EPI);
constexpr uint32_t P_TMEM_COLS = 512;           // two accumulators of PN columns
constexpr int P_MAX_E = 256;
// SwiGLU exchange: per warp pair, two chunk buffers (alternating), each with
// 16 values per lane going each way; rows of 17 floats avoid bank conflicts
constexpr int P_XROW = 17;
constexpr int P_XBUF = 32 * P_XROW;              // floats of one direction of one chunk
constexpr size_t P_XBYTES = (size_t)2 * 2 * 2 * P_XBUF * 4;   // pairs x chunks x directions
constexpr size_t P_DYN_SMEM = 1024 + (size_t)PS * P_STAGE + P_XBYTES;
static_assert(P_STAGE % 1024 == 0, "stage alignment");

struct PShared {
  uint64_t full[PS];    // first CTA: tokens + weights of both CTAs landed
  uint64_t empty[PS];   // both CTAs: the MMAs that read the stage completed
  uint64_t tfull[2];    // both CTAs: the accumulator's MMAs completed
  uint64_t tempty[2];   // first CTA: both CTAs' epilogues drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort, failed_on_entry, num_tiles;
  int offs[P_MAX_E + 1];
  int tile_start[P_MAX_E];
};

struct PArgs {
  const int32_t *offsets;  // nullptr: one segment [0, rows) of expert 0
  int num_experts;
  int rows;                // token rows of A (and of out)
  int K;
  int N;                   // output columns (weight rows of W, and of W3 for SwiGLU)
  __nv_bfloat16 *out;      // [rows][N]
  int *status;
  int tok_major;           // 1: token block outer, weight block fastest
};

struct PTile {
  int e, tok0, ntok, seg_end, wb;
};

// Tokens per block of a segment of c tokens: the segment splits into
// ceil(c / PN) blocks of nearly equal size, rounded up to 16 (the MMA's N
// step), so that no block is a thin remainder.  A tile's weight copies cost
// the same whatever its N, and a thin block's MMAs are too short to hide them.
__device__ __forceinline__ int block_tokens(int c) {
  const int nb = max(1, (c + PN - 1) / PN);
  return ((c + nb - 1) / nb + 15) & ~15;
}
__device__ __forceinline__ int token_blocks(int c) {
  return c > 0 ? (c + block_tokens(c) - 1) / block_tokens(c) : 0;
}

__device__ __forceinline__ PTile p_decode(const PShared &sh, int E, int t, int n_wb,
                                          bool tok_major) {
  int lo = 0, hi = E;   // largest e with tile_start[e] <= t (skips empty experts)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  PTile tl;
  tl.e = lo;
  const int beg = sh.offs[lo], end = sh.offs[lo + 1];
  const int bt = block_tokens(end - beg);
  const int m_tiles = token_blocks(end - beg);
  const int local = t - sh.tile_start[lo];
  // weight-major: token blocks fastest, so pairs running side by side share a
  // weight block; token-major (a segment larger than its weights, e.g. the
  // shared expert's 16k tokens): weight blocks fastest, so the weights stay
  // in L2 and each token block comes from DRAM once
  int tb;
  if (tok_major) {
    tb = local / n_wb;
    tl.wb = local - tb * n_wb;
  } else {
    tl.wb = local / m_tiles;
    tb = local - tl.wb * m_tiles;
  }
  tl.tok0 = beg + tb * bt;
  tl.ntok = min(bt, end - tl.tok0);
  tl.seg_end = min(end, tl.tok0 + bt);
  return tl;
}

__device__ __forceinline__ float silu_mul(float a, float b) {
  return __fdividef(a, 1.f + __expf(-a)) * b;
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t *>(&h);
}

// EPI: 0 plain, 1 relu, 2 swiglu (W = W1 rows, W3 = W3 rows).
template <int EPI>
__global__ void __launch_bounds__(P_THREADS, 1)
gemm_t2_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ CUtensorMap tmW3, PArgs args) {
  constexpr int OUT_CTA = (EPI == 2) ? PM / 2 : PM;   // output columns per CTA per tile
  constexpr int OUT_TILE = 2 * OUT_CTA;
  constexpr uint32_t TX_BYTES = 2u * P_STAGE;          // both CTAs' copies of one stage
  extern __shared__ uint8_t dyn_smem[];
  __shared__ PShared sh;
  uint8_t *smem = dyn_smem + ((1024 - (tc::smem_u32(dyn_smem) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int E = args.offsets ? args.num_experts : 1;
  const int n_wb = (args.N + OUT_TILE - 1) / OUT_TILE;
  const int KB = (args.K + PK - 1) / PK;

  if (threadIdx.x == 0) {
    tc::prefetch_tmap(&tmX);
    tc::prefetch_tmap(&tmW);
    if (EPI == 2) tc::prefetch_tmap(&tmW3);
    sh.failed_on_entry = status_failed(args.status) ? 1 : 0;
    sh.abort = sh.failed_on_entry;
  }
  for (int i = threadIdx.x; i <= E; i += P_THREADS)
    sh.offs[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows);
  if (warp == 1) tmem_alloc2(&sh.tmem_base, P_TMEM_COLS);
  if (threadIdx.x == 32) {
    for (int s = 0; s < PS; ++s) {
      tc::mbar_init(&sh.full[s], 1);
      tc::mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sh.tfull[a], 1);
      tc::mbar_init(&sh.tempty[a], 2 * P_EPI);   // one arrival per epilogue warp of each CTA
    }
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
        else cnt[i] = token_blocks(en - b) * n_wb;
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
      if (bad && rank == 0) set_status(args.status, MOE_ERR_BAD_INDEX, -1);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either CTA touches the other's
  cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem_base = sh.tmem_base;
  const int num_tiles = sh.num_tiles;
  volatile int *abort = &sh.abort;
  const bool tok_major = args.tok_major != 0;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[PS];
#pragma unroll
      for (int s = 0; s < PS; ++s) last_phase[s] = -1;
      for (int t = pair; t < num_tiles && !*abort; t += n_pairs) {
        const PTile tl = p_decode(sh, E, t, n_wb, tok_major);
        const int ntok = tl.ntok;
        const int half = ((ntok + 15) & ~15) >> 1;   // tokens staged by each CTA
        const int brow = tl.tok0 + (int)rank * half;
        const int wrow = tl.wb * OUT_TILE + (int)rank * OUT_CTA;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&sh.empty[stage], phase ^ 1u, abort)) break;
          uint8_t *sb = smem + stage * P_STAGE;
          uint8_t *sa = sb + P_B_BYTES;
          const uint32_t bar = map_to_rank(tc::smem_u32(&sh.full[stage]), 0);
          if (rank == 0) tc::mbar_arrive_expect_tx(&sh.full[stage], TX_BYTES);
          tma2_load_2d(&tmX, bar, sb, kb * PK, brow);
          if constexpr (EPI == 2) {
            tma2_load_3d(&tmW, bar, sa, kb * PK, wrow, tl.e);               // rows 0..63
            tma2_load_3d(&tmW3, bar, sa + P_A_BYTES / 2, kb * PK, wrow, tl.e);  // rows 64..127
          } else {
            tma2_load_3d(&tmW, bar, sa, kb * PK, wrow, tl.e);
          }
          last_phase[stage] = (int)phase;
          if (++stage == PS) { stage = 0; phase ^= 1u; }
        }
      }
      if (*abort && rank == 0) {
        // let the copies in flight land before the pair exits (the second
        // CTA's copies count on these barriers too)
        for (int s = 0; s < PS; ++s)
          if (last_phase[s] >= 0)
            tc::mbar_wait_drain(&sh.full[s], (uint32_t)last_phase[s], 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (first CTA of the pair)
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok && !*abort; t += n_pairs, ++local) {
        const PTile tl = p_decode(sh, E, t, n_wb, tok_major);
        const int ntok = tl.ntok;
        const uint32_t idesc = tc::idesc_bf16_f32(2 * PM, (ntok + 15) & ~15);
        const int acc = local & 1;
        if (!mbar_wait_cluster(&sh.tempty[acc], ((local >> 1) & 1) ^ 1u, abort)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc::mbar_wait(&sh.full[stage], phase, abort)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t sb = tc::smem_u32(smem + stage * P_STAGE);
          const uint32_t sa = sb + P_B_BYTES;
#pragma unroll
          for (int k = 0; k < PK / 16; ++k)
            mma2_bf16(d_tmem, tc::smem_desc_sw128(sa + k * 32), tc::smem_desc_sw128(sb + k * 32),
                      idesc, (kb != 0 || k != 0) ? 1u : 0u);
          mma2_commit_both(&sh.empty[stage]);
          if (++stage == PS) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma2_commit_both(&sh.tfull[acc]);
      }
      if (*abort) {
        mma2_commit_self(&sh.drain);
        tc::mbar_wait_drain(&sh.drain, 0, 100000000ull);
      }
    }
  } else {
    // ---------------- epilogue (both CTAs): warp w drains TMEM lanes 32*(w%4) .. +31
    const int quarter = warp & 3;
    const int pq = quarter & 1;                  // SwiGLU: W1 quarter pq pairs with W3 quarter pq + 2
    const bool w3 = quarter >= 2;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tempty_first = map_to_rank(tc::smem_u32(&sh.tempty[0]), 0);
    float *xbuf = reinterpret_cast<float *>(smem + (size_t)PS * P_STAGE);
    int local = 0;
    for (int t = pair; t < num_tiles; t += n_pairs, ++local) {
      const PTile tl = p_decode(sh, E, t, n_wb, tok_major);
      const int ntok = tl.ntok;
      const int acc = local & 1;
      const bool ok = tc::mbar_wait(&sh.tfull[acc], (local >> 1) & 1, abort);
      if constexpr (EPI == 2) {
        // the two warps of a pair meet on named barriers below: they agree on
        // going on first (a warp whose wait ran out has raised *abort)
        if (tc::bar_or(1 + pq, 64, !ok)) break;
      } else {
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      tc::tc_fence_after();
      const uint32_t tb = lane_base + (uint32_t)(acc * PN);
      // this thread's output column
      const int col = (EPI == 2) ? tl.wb * OUT_TILE + (int)rank * OUT_CTA + pq * 32 + lane
                                 : tl.wb * OUT_TILE + (int)rank * OUT_CTA + quarter * 32 + lane;
      const bool col_ok = col < args.N;
      uint16_t *o = reinterpret_cast<uint16_t *>(args.out) + col;
#pragma unroll 1
      for (int c = 0; c * 32 < ntok; ++c) {
        uint32_t a[32];
        tc::tmem_ld32(tb + (uint32_t)(c * 32), a);
        tc::tmem_ld_wait();
        const int tok0 = tl.tok0 + c * 32;
        if constexpr (EPI == 2) {
          // the W1 warp (gate values) finishes tokens 0..15 of the chunk, the
          // W3 warp (up values) tokens 16..31; each hands the other its half
          float *to_w3 = xbuf + (size_t)((pq * 2 + (c & 1)) * 2) * P_XBUF;   // gates 16..31
          float *to_w1 = to_w3 + P_XBUF;                                    // ups 0..15
          float *mine = w3 ? to_w1 : to_w3;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mine[lane * P_XROW + i] = __uint_as_float(w3 ? a[i] : a[16 + i]);
          asm volatile("bar.sync %0, 64;" ::"r"(3 + pq) : "memory");
          const float *theirs = w3 ? to_w3 : to_w1;
          uint16_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float other = theirs[lane * P_XROW + i];
            const float g = w3 ? other : __uint_as_float(a[i]);
            const float u = w3 ? __uint_as_float(a[16 + i]) : other;
            hv[i] = bf16_bits(silu_mul(g, u));
          }
          const int tsub = w3 ? 16 : 0;
          if (col_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int tok = tok0 + tsub + i;
              if (tok < tl.seg_end) o[(size_t)tok * args.N] = hv[i];
            }
          }
        } else {
          if (col_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float v = __uint_as_float(a[i]);
              if constexpr (EPI == 1) v = fmaxf(v, 0.f);
              const int tok = tok0 + i;
              if (tok < tl.seg_end) o[(size_t)tok * args.N] = bf16_bits(v);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_first + (uint32_t)(acc * sizeof(uint64_t)));
    }
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  // neither CTA leaves (or frees its tensor memory) while the other may still
  // read its shared memory, signal its barriers or write its tensor memory
  cluster_sync();
  if (warp == 1) {
    tc::tc_fence_after();
    tmem_dealloc2(tmem_base, P_TMEM_COLS);
  }
  if (threadIdx.x == 0 && sh.abort && !sh.failed_on_entry)
    set_status(args.status, MOE_ERR_TIMEOUT, blockIdx.x);
}

int pairs_resident(const void *kernel, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (num_sms() / 2));
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = num_sms() / 2;
  }
  return n;
}

template <int EPI>
cudaError_t launch_t2(const GemmStage &g, int *status, cudaStream_t s) {
  static int pairs = 0;
  if (pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_t2_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)P_DYN_SMEM);
    if (e != cudaSuccess) return e;
    pairs = pairs_resident(reinterpret_cast<const void *>(gemm_t2_kernel<EPI>), P_DYN_SMEM);
  }
  const int E = g.offsets ? g.num_experts : 1;
  CUtensorMap mX, mW, mW3;
  const uint64_t dX[2] = {(uint64_t)g.K, (uint64_t)g.rows};
  const uint32_t bX[2] = {PK, PN / 2};
  if (!make_tensor_map(&mX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.A, 2, dX, bX,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t dW[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)E};
  const uint32_t bW[3] = {PK, (uint32_t)(EPI == 2 ? PM / 2 : PM), 1};
  if (!make_tensor_map(&mW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.B, 3, dW, bW,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (EPI == 2) {
    if (!make_tensor_map(&mW3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.B3, 3, dW, bW,
                         CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    mW3 = mW;
  }
  PArgs a{};
  a.offsets = g.offsets;
  a.num_experts = g.num_experts;
  a.rows = g.rows;
  a.K = g.K;
  a.N = g.N;
  a.out = static_cast<__nv_bfloat16 *>(g.out);
  a.status = status;
  // token blocks outer when an average segment holds more rows than the
  // weights it meets (the shared expert's one segment of all n tokens)
  const long seg_rows = (long)g.rows / (E > 0 ? E : 1);
  a.tok_major = seg_rows > (long)g.N * (EPI == 2 ? 2 : 1) ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(P_THREADS);
  cfg.dynamicSmemBytes = P_DYN_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_t2_kernel<EPI>, mX, mW, mW3, a);
}

}  // namespace

bool gemm_t2_supported(const GemmStage &g) {
  return g.rows > 0 && tensor_maps_available() && g.a_dtype == MOE_BF16 &&
         g.b_dtype == MOE_BF16 && g.out_dtype == MOE_BF16 &&
         (g.epi == 0 || g.epi == 1 || g.epi == 2) && g.num_experts <= P_MAX_E &&
         g.K % 8 == 0 && g.N % 8 == 0 && num_sms() >= 2;
}

cudaError_t launch_gemm_t2(const GemmStage &g, int *status, cudaStream_t s) {
  switch (g.epi) {
    case 1: return launch_t2<1>(g, status, s);
    case 2: return launch_t2<2>(g, status, s);
    default: return launch_t2<0>(g, status, s);
  }
}

}  // namespace moe
