// The router's linear layer on the 5th-generation tensor cores (tcgen05 +
// TMEM + TMA): logits = x Wg^T (+ b) in fp32 ("How Mixture of Experts Scales
// Model Parameters", section "Routing: a router scores the experts, and the
// top one runs": the router is one linear layer whose scores go through a
// softmax).  The expert projections run elsewhere: bf16 on SM pairs
// (gemm_t2.cu), MXFP4 with the weights dequantised into tensor memory
// (gemm_mx.cu); launch_gemm_tc sends them there.
//
// One CTA per SM, persistent:
//   warp 0      TMA producer: x tile 128 x 64 (rows) and Wg tile 128 x 64 (EPI
//               3, up to 128 experts per tile, 6-stage ring) or 32 x 64 (EPI
//               4, at most 32 experts, 10 stages), 128-byte swizzle.
//   warp 1      allocates 512 TMEM columns; one thread issues
//               tcgen05.mma.kind::f16 M=128 N=128 or 32, K=16 (fp32).
//   warps 2..   epilogue: tcgen05.ld of each partial, fp32 sums in registers.
// Each 64-wide k-block is summed into a fresh TMEM partial (four 128-column
// or eight 32-column partials in flight) and the partials are added in fp32
// registers.  Tiles run row block first, then expert block, so the CTAs that
// read one block of x rows for different experts run together and the rows
// come from DRAM once.  When the row tiles alone leave most SMs idle, a
// tile's k-blocks are split over up to four CTAs that write fp32 partial
// planes; the selection (the selection kernel, or for at most 32 experts the
// CTA that completes the row tile) adds them in plane order.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int MAX_STAGES = 10;

// Ring depth per variant: with 32 experts the B tile is narrower, so the same
// shared memory holds more k-blocks of the x stream in flight.
__host__ __device__ constexpr int stage_bytes(int epi) {
  return A_BYTES + (epi == 4 ? 32 : 128) * BK * 2;
}
__host__ __device__ constexpr int num_stages(int epi) { return epi == 4 ? MAX_STAGES : 6; }
__host__ __device__ constexpr int dyn_smem_bytes(int epi) {
  return num_stages(epi) * stage_bytes(epi) + 1024;
}
// Epilogue warps: the 128-expert router drains a 128-column partial every
// k-block, so two warps share each TMEM lane quarter (64 columns each).
__host__ __device__ constexpr int epi_warps(int epi) { return epi == 3 ? 8 : 4; }
__host__ __device__ constexpr int threads_of(int epi) { return 64 + 32 * epi_warps(epi); }
constexpr int MAX_E = 256;
constexpr uint32_t TMEM_COLS = 512;

struct TcArgs {
  const int32_t *offsets;  // nullptr: one segment [0, rows) of expert 0
  int num_experts;
  int rows;
  int K;
  int N;           // output columns
  void *out;       // fp32 [rows][N] logits, or [ksplit][rows][N] partial planes
  const float *bias;
  int *status;
  int ksplit;      // router: k ranges per row tile (> 1: partial sums, no bias)
  // EPI 4 with sel_idx set: the router's selection runs in the epilogue.  With
  // ksplit > 1 the CTA that completes a row tile's count (tile_count, zeroed
  // before the launch) adds the partial planes in out and selects.
  int *tile_count;
  float *logits;   // [rows][N] logits (bias included)
  int32_t *sel_idx;
  float *sel_gate;
  float *probs;    // [rows][N] softmax, or nullptr
  int top_k, gate_mode;
};

struct TcShared {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[8];    // partial ring: 4 (EPI 3) or 8 (EPI 4)
  uint64_t tempty[8];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int failed_on_entry;
  int num_tiles;
  int last;       // fused router selection: this CTA completed the row tile
  int offs[MAX_E + 1];
  int tile_start[MAX_E];
};

struct Tile {
  int e, row0, seg_end, n_idx;
};

// Tile t of the list: row block, then column block (the router's experts),
// so the CTAs that read one block of rows for different experts run together
// and the rows come from DRAM once.
__device__ __forceinline__ Tile decode_tile(const TcShared &sh, int E, int t, int n_tiles) {
  int lo = 0, hi = E;   // largest e with tile_start[e] <= t (skips empty experts)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  Tile tl;
  tl.e = lo;
  const int beg = sh.offs[lo], end = sh.offs[lo + 1];
  const int local = t - sh.tile_start[lo];
  const int m = local / n_tiles;
  tl.n_idx = local - m * n_tiles;
  tl.row0 = beg + m * BM;
  tl.seg_end = end;
  return tl;
}

// Selection of one router row by one thread (E <= 32 logits in registers),
// the same choice and gates as the warp-wide selection of the router's
// selection kernel ("How Mixture of Experts Scales Model Parameters",
// sections "Routing: a router scores the experts, and the top one runs" and
// "Top-K: several experts, added up by weight"): larger logit first, lower
// index on equal values, NaN ranks below everything; softmax with the
// maximum subtracted; top_prob gates divide by the full sum, renorm gates by
// the sum over the chosen k (added in rank order).
__device__ __forceinline__ void select_row(const float (&l)[32], int E, int k, int gate_mode,
                                           int32_t *idx, float *gate, float *probs) {
  float t[32];
  float mx = -INFINITY;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    t[e] = (e < E && !isnan(l[e])) ? l[e] : -INFINITY;
    mx = fmaxf(mx, t[e]);
  }
  float sum = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    if (e < E) {
      const float ex = expf(t[e] - mx);
      sum += ex;
      if (probs) probs[e] = ex;
    }
  }
  if (probs)
    for (int e = 0; e < E; ++e) probs[e] = probs[e] / sum;
  uint32_t taken = 0;
  float sel_sum = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      if (e < E && !((taken >> e) & 1u) && (t[e] > bv || (t[e] == bv && e < bi))) {
        bv = t[e];
        bi = e;
      }
    }
    taken |= 1u << bi;
    const float exj = expf(bv - mx);
    sel_sum += exj;
    idx[j] = bi;
    gate[j] = exj;
  }
  const float denom = (gate_mode == MOE_GATE_RENORM) ? sel_sum : sum;
  for (int j = 0; j < k; ++j) gate[j] = gate[j] / denom;
}

// EPI 3: fp32 logits + per-column bias, up to 128 experts per tile; EPI 4:
// the same for at most 32 experts (and optionally the selection).
//
// Both keep the router's logits accurate to fp32 rounding: the tensor
// core sums each 64-wide k-block into a fresh TMEM partial (N = 128 or 32
// columns, four or eight partials in flight), and the epilogue warps add the
// partials in fp32 registers with round-to-nearest.  Accumulating the whole
// reduction in TMEM instead drifted by ~2e-5 on d = 4096 rows, too close to
// the 1e-5 near-tie margin of the routing decision.
template <int EPI>
__global__ void __launch_bounds__(threads_of(EPI), 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               TcArgs args) {
  static_assert(EPI == 3 || EPI == 4, "router variants");
  // MMA N = B rows per stage: 128 experts per tile, or 32 (EPI 4) when there
  // are at most 32, so a layer with 8 experts does not drain 128 accumulator
  // columns per k-block
  constexpr int BNT = EPI == 4 ? 32 : 128;
  // partials in flight, so the MMAs run ahead of the epilogue's drains
  constexpr int NACC = EPI == 4 ? 8 : 4;
  constexpr int ACC_COLS = BNT;
  constexpr int EPI_WARPS = epi_warps(EPI);
  constexpr int N_OUT = BNT;   // output columns per tile
  constexpr int NSTAGE = num_stages(EPI);
  constexpr int SBYTES = stage_bytes(EPI);
  constexpr int NTHREADS = threads_of(EPI);
  constexpr uint32_t TX_BYTES = A_BYTES + BNT * BK * 2;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ TcShared sh;
  uint8_t *smem = dyn_smem + ((1024 - (tc::smem_u32(dyn_smem) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.offsets ? args.num_experts : 1;
  const int n_tiles = (args.N + N_OUT - 1) / N_OUT;
  const int KB = (args.K + BK - 1) / BK;
  // work unit t: row/column tile t / KS over k-blocks [k_begin, k_end)
  const int KS = args.ksplit;
  auto k_begin = [&](int t) { return (int)((int64_t)(t % KS) * KB / KS); };
  auto k_end = [&](int t) { return (int)((int64_t)(t % KS + 1) * KB / KS); };

  if (threadIdx.x == 0) {
    // descriptor fetches overlap the setup below instead of the first copy
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmB);
    sh.failed_on_entry = status_failed(args.status) ? 1 : 0;
    sh.abort = sh.failed_on_entry;
  }
  for (int i = threadIdx.x; i <= E; i += NTHREADS)
    sh.offs[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows);
  if (warp == 1) tc::tmem_alloc(&sh.tmem_base, TMEM_COLS);
  if (threadIdx.x == 32) {
    for (int s = 0; s < NSTAGE; ++s) {
      tc::mbar_init(&sh.full[s], 1);
      tc::mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      tc::mbar_init(&sh.tfull[a], 1);
      tc::mbar_init(&sh.tempty[a], 32 * EPI_WARPS);
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
        else cnt[i] = ((en - b + BM - 1) / BM) * n_tiles;
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
      sh.num_tiles = bad ? 0 : total * args.ksplit;
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
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int last_phase[NSTAGE];
#pragma unroll
      for (int s = 0; s < NSTAGE; ++s) last_phase[s] = -1;
      for (int t = blockIdx.x; t < num_tiles && !*abort; t += gridDim.x) {
        const Tile tl = decode_tile(sh, E, t / KS, n_tiles);
        const int wrow = tl.n_idx * N_OUT;
        const int kb1 = k_end(t);
        for (int kb = k_begin(t); kb < kb1; ++kb) {
          if (!tc::mbar_wait(&sh.empty[stage], phase ^ 1u, abort)) break;
          uint8_t *sa = smem + stage * SBYTES;
          uint8_t *sb = sa + A_BYTES;
          tc::mbar_arrive_expect_tx(&sh.full[stage], TX_BYTES);
          tc::tma_load_2d(&tmA, &sh.full[stage], sa, kb * BK, tl.row0);
          tc::tma_load_3d(&tmB, &sh.full[stage], sb, kb * BK, wrow, tl.e);
          last_phase[stage] = (int)phase;
          if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
        }
      }
      if (*abort) {
        // let the copies this thread issued land before the CTA exits
        for (int s = 0; s < NSTAGE; ++s)
          if (last_phase[s] >= 0)
            tc::mbar_wait_drain(&sh.full[s], (uint32_t)last_phase[s], 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, BNT);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;   // partials used so far (one per k-block)
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok && !*abort; t += gridDim.x) {
        const int kb1 = k_end(t);
        for (int kb = k_begin(t); kb < kb1; ++kb) {
          const int acc = local % NACC;
          const uint32_t acc_phase = (local / NACC) & 1;
          if (!tc::mbar_wait(&sh.tempty[acc], acc_phase ^ 1u, abort)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
          if (!tc::mbar_wait(&sh.full[stage], phase, abort)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t sa = tc::smem_u32(smem + stage * SBYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16(d_tmem, tc::smem_desc_sw128(sa + k * 32), tc::smem_desc_sw128(sb + k * 32),
                         idesc, k != 0 ? 1u : 0u);
          tc::mma_commit(&sh.empty[stage]);
          if (++stage == NSTAGE) { stage = 0; phase ^= 1u; }
          tc::mma_commit(&sh.tfull[acc]);
          ++local;
        }
      }
      if (*abort) {
        tc::mma_commit(&sh.drain);
        tc::mbar_wait_drain(&sh.drain, 0, 100000000ull);
      }
    }
  } else if (warp < 2 + EPI_WARPS) {
    // ---------------- epilogue: warps 2..; warp w reads TMEM lanes 32*(w%4)..
    const int quarter = warp & 3;
    const int r_local = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    int local = 0;
    {
      // the warps of one lane quarter split the columns: NCOL from col_off
      constexpr int NCOL = N_OUT / (EPI_WARPS / 4);
      const int col_off = ((warp - 2) >> 2) * NCOL;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        const Tile tl = decode_tile(sh, E, t / KS, n_tiles);
        float sum[NCOL];
#pragma unroll
        for (int i = 0; i < NCOL; ++i) sum[i] = 0.f;
        bool ok = true;
        const int kb1 = k_end(t);
        for (int kb = k_begin(t); kb < kb1; ++kb, ++local) {
          const int acc = local % NACC;
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&sh.tfull[acc], (local / NACC) & 1, abort));
          if (!ok) break;
          tc::tc_fence_after();
          uint32_t a[NCOL / 32][32];
#pragma unroll
          for (int c = 0; c < NCOL / 32; ++c)
            tc::tmem_ld32(lane_base + (uint32_t)(acc * ACC_COLS + col_off + c * 32), a[c]);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < NCOL / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) sum[c * 32 + i] += __uint_as_float(a[c][i]);
          tc::tc_fence_before();
          tc::mbar_arrive(&sh.tempty[acc]);
        }
        const int row = tl.row0 + r_local;
        const bool row_ok = row < tl.seg_end;
        if (EPI == 4 && args.sel_idx != nullptr) {
          // selection fused here.  The four epilogue warps first agree on
          // going on (a warp whose wait ran out has raised *abort), since
          // they meet on named barrier 1 below.
          if (tc::bar_or(1, 32 * EPI_WARPS, !ok || *abort != 0)) break;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = sum[i];
          bool last = true;
          if (KS > 1) {
            float *planes = static_cast<float *>(args.out);
            if (row_ok) {
              float *prow = planes + ((size_t)(t % KS) * args.rows + row) * args.N;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < args.N) prow[i] = sum[i];
            }
            // the planes this CTA wrote are visible before it counts itself
            __threadfence();
            tc::bar_or(1, 32 * EPI_WARPS, false);
            if (warp == 2 && lane == 0)
              sh.last = atomicAdd(&args.tile_count[t / KS], 1) == KS - 1 ? 1 : 0;
            tc::bar_or(1, 32 * EPI_WARPS, false);
            last = sh.last != 0;
            if (last && row_ok) {
              __threadfence();
              // the planes in order, as the selection kernel adds them
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
              for (int pp = 0; pp < KS; ++pp) {
                const float *prow = planes + ((size_t)pp * args.rows + row) * args.N;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (i < args.N) v[i] += __ldcg(prow + i);
              }
            }
          }
          if (last && row_ok) {
            float *lrow = args.logits + (size_t)row * args.N;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i < args.N) {
                v[i] = v[i] + (args.bias ? args.bias[i] : 0.f);
                lrow[i] = v[i];
              }
            }
            select_row(v, args.N, args.top_k, args.gate_mode,
                       args.sel_idx + (size_t)row * args.top_k,
                       args.sel_gate + (size_t)row * args.top_k,
                       args.probs ? args.probs + (size_t)row * args.N : nullptr);
          }
          __syncwarp();
          continue;
        }
        if (!ok) break;
        if (row_ok) {
          // k range p of a split writes its partial sums to plane p; the
          // reader adds the planes in order, then the bias
          const int p = t % KS;
          float *orow = static_cast<float *>(args.out) + ((size_t)p * args.rows + row) * args.N;
          const float *bias = KS > 1 ? nullptr : args.bias;
#pragma unroll
          for (int i = 0; i < NCOL; ++i) {
            const int col = tl.n_idx * N_OUT + col_off + i;
            if (col < args.N) orow[col] = sum[i] + (bias ? bias[col] : 0.f);
          }
        }
        __syncwarp();
      }
    }
  }

  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && sh.abort && !sh.failed_on_entry)
    set_status(args.status, MOE_ERR_TIMEOUT, blockIdx.x);
}

// ---------------------------------------------------------------- host side

template <int EPI>
cudaError_t launch_epi(const GemmStage &g, int *status, cudaStream_t s) {
  const size_t smem = (size_t)dyn_smem_bytes(EPI);
  static size_t smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
  }
  const int E = g.offsets ? g.num_experts : 1;
  CUtensorMap mA, mB;
  const uint64_t dA[2] = {(uint64_t)g.K, (uint64_t)g.rows};
  const uint32_t bA[2] = {BK, BM};
  const int wrows = EPI == 3 ? 128 : 32;
  if (!make_tensor_map(&mA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.A, 2, dA, bA,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const uint64_t dB[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)E};
  const uint32_t bB[3] = {BK, (uint32_t)wrows, 1};
  if (!make_tensor_map(&mB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.B, 3, dB, bB,
                       CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcArgs a{};
  a.offsets = g.offsets;
  a.num_experts = g.num_experts;
  a.rows = g.rows;
  a.K = g.K;
  a.N = g.N;
  a.out = g.out;
  a.bias = g.col_bias;
  a.status = status;
  a.ksplit = g.ksplit > 1 ? g.ksplit : 1;
  if (EPI == 4 && gemm_tc_router_fuses(g)) {
    a.sel_idx = g.sel_idx;
    a.sel_gate = g.sel_gate;
    a.probs = g.sel_probs;
    a.logits = g.logits;
    a.tile_count = g.tile_count;
    a.top_k = g.top_k;
    a.gate_mode = g.gate_mode;
  }
  gemm_tc_kernel<EPI><<<num_sms(), threads_of(EPI), smem, s>>>(mA, mB, a);
  return cudaGetLastError();
}

}  // namespace

bool gemm_tc_supported(const GemmStage &g) {
  if (g.rows <= 0 || !tensor_maps_available()) return false;
  // MXFP4: the weights-in-tensor-memory kernel of gemm_mx.cu
  if (g.b_dtype == MOE_MXFP4) return gemm_mx_supported(g);
  // bf16 expert projections: the SM-pair kernel of gemm_t2.cu
  if (g.epi <= 2) return gemm_t2_supported(g);
  // the router (epi 3; with N <= 32 the 32-column variant)
  return g.epi == 3 && g.a_dtype == MOE_BF16 && g.b_dtype == MOE_BF16 &&
         g.out_dtype == MOE_F32 && g.K % 8 == 0;
}

bool gemm_tc_router_fuses(const GemmStage &g) {
  return g.epi == 3 && g.N <= 32 && g.sel_idx != nullptr && g.sel_gate != nullptr &&
         g.logits != nullptr && g.top_k >= 1 && g.top_k <= g.N &&
         (g.ksplit <= 1 || g.tile_count != nullptr) && gemm_tc_supported(g);
}

int gemm_tc_router_ksplit(const GemmStage &g, size_t plane_room) {
  // row tiles x expert tiles of the router; when they cover less than half
  // the SMs, each tile's d range is split over up to four CTAs (at least
  // eight k-blocks each), as far as the partial planes fit in plane_room
  const int tiles = ((g.rows + BM - 1) / BM) * (g.N <= 32 ? 1 : (g.N + 127) / 128);
  const int kb = (g.K + BK - 1) / BK;
  int ks = num_sms() / tiles;
  ks = ks > 4 ? 4 : ks;
  ks = ks > kb / 8 ? kb / 8 : ks;
  while (ks > 1 && (size_t)ks * g.rows * g.N * sizeof(float) > plane_room) --ks;
  return ks < 2 ? 1 : ks;
}

cudaError_t launch_gemm_tc(const GemmStage &g, int *status, cudaStream_t s) {
  if (g.b_dtype == MOE_MXFP4) return launch_gemm_mx(g, status, s);
  if (g.epi <= 2) return launch_gemm_t2(g, status, s);
  return g.N <= 32 ? launch_epi<4>(g, status, s) : launch_epi<3>(g, status, s);
}

}  // namespace moe
