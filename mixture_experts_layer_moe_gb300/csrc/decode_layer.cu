// The small-batch MoE layer over MXFP4 or NVFP4 experts in one cooperative
// launch:
// router logits, top-k selection and gates, the stable dispatch, the selected
// experts' up (SwiGLU) and down projections, and the combine.
//
// "How Mixture of Experts Scales Model Parameters": the router is one linear
// layer followed by a softmax ("Routing: a router scores the experts, and the
// top one runs"); the K best experts run and their outputs are added by
// weight ("Top-K: several experts, added up by weight"); tokens are grouped
// per expert and put back in order ("The forward pass: dispatch, then
// combine").  Decode is bound by the weight bytes it reads ("Inference
// Optimization: The Bandwidth Wall, PagedAttention, and FlashAttention"), so
// the layer should take the time of one stream over the selected experts.  As
// five dependent kernels, each paying its launch, setup and drain, a one-token
// layer spends several times longer than that stream.
//
// One CTA per resident slot (two per SM), all resident together (cooperative
// launch), so CTAs may wait on one another:
//   1. router logits: one warp per (token, expert) pair, spread over the
//      grid, with the per-piece fp32 arithmetic of the small-batch router
//      kernel (bf16x8_dot, warp_sum_xor: the same logits); every CTA also
//      converts a share of the x rows to f16;
//   2. grid barrier;
//   3. every CTA selects for all n tokens and builds the stable dispatch
//      itself (the same code on the same logits in every CTA, hence the same
//      arrays); CTA 0 writes them out.  The first units' weights start
//      streaming as soon as the experts with tokens are known, before the
//      per-token positions are done;
//   4. work units -- 16 * RG rows of W1 and W3 of one selected expert ("up"),
//      or 32 * RG rows of its W2 ("down", two 16-row halves per group) -- are
//      claimed from a global counter in a fixed order: all up units, then all
//      down units, each expert by expert.  A unit streams its weight boxes as
//      the two-kernel FFN does (decode_kernel.cuh: the same MMA, split and
//      reduction order, so the same bits).  A down unit reads h rows, so it
//      first waits until every up unit of its expert has stored them (a
//      per-expert counter).  Each CTA runs its claims in order, so the
//      earliest unfinished unit never waits on a later one and the waits
//      always end; every wait is bounded besides (MOE_ERR_TIMEOUT);
//   5. grid barrier; combine: y[t] = sum_j g[t][j] * y_perm[inv_perm[t*k+j]]
//      in fp32, slot order, one rounding (as combine.cu).
// Data that this launch writes and then reads again (logits, selections,
// f16 x rows, h, y_perm) is never read through the read-only path: the
// reading warp first takes an acquire (a grid barrier, or the expert's
// counter), then loads with plain or L2-only loads.
#include "classify.cuh"
#include "decode_kernel.cuh"
#include "select.cuh"

namespace moe {
namespace {

constexpr int LY_THREADS = 32 * DV_WARPS;
constexpr int LY_NQ = 4;         // claimed units held per CTA (a ring)
constexpr int LY_NPEND = 32;     // up units a group may note before counting them
constexpr int LY_RW = 12;        // router: Wg pieces per lane
constexpr int LY_MAX_D = 32 * 8 * LY_RW;
// Batches up to this many tokens run as one launch.  Measured on the gpt-oss
// decode shape (d = d_ff = 2880, 128 experts, top-4; microseconds per layer,
// one launch against the chained kernels): n = 1 40 / 46, 4 72 / 82, 8 107 /
// 113, 16 171 / 169, 32 256 / 249, 64 348 / 332.  From about 32 tokens the
// one launch's serial head (router, selection, dispatch: 25 us at 64 tokens)
// costs more than the launches it saves, and the chain is faster.  (Within
// this range the chain's router is the small-batch kernel, so both paths
// compute the same logits.)
constexpr int LY_MAX_TOKENS = 16;
// NVFP4 experts, on the same shape (an E4M3 scale per 16 elements, so units
// of at most 32 rows: twice the MXFP4 units at 16 tokens): n = 1 42 / 47,
// 4 80 / 89, 8 125 / 125, 16 207 / 191.
constexpr int LY_MAX_TOKENS_NV = 8;

// Per-launch counters, zeroed before the launch: the two grid barriers, the
// unit queue, and per expert the up-unit groups whose h rows are stored.
enum { SY_BAR1 = 0, SY_BAR2 = 1, SY_QUEUE = 2, SY_UPDONE = 4 };

struct LayerArgs {
  const __nv_bfloat16 *x, *Wg;   // [n][d], [E][d]
  const float *bias;             // [E] or nullptr
  const uint8_t *S1, *S3, *S2;   // block scales of W1, W3 [E][d_ff][d/32 or d/16], W2 likewise
  const float *G1, *G3, *G2;     // NVFP4: one fp32 scale per expert matrix [E]
  int n, d, d_ff, E, k, gate_mode;
  float *logits;                 // [n][E]
  int32_t *topk_idx;             // [n][k]
  float *topk_gate;              // [n][k]
  int32_t *counts, *offsets, *perm, *inv_perm;
  uint16_t *x16;                 // [n][d] f16 x rows, token order
  __nv_bfloat16 *h;              // [P][d_ff]
  uint16_t *h16;                 // [P][d_ff] f16 copy of h
  __nv_bfloat16 *y_perm;         // [P][d]
  __nv_bfloat16 *y;              // [n][d]
  int *sync;                     // SY_UPDONE + 256 zeroed ints
  int *status;
  // resident pool (POOL): slot table, the slots' scales, classification outputs
  const int32_t *slot_of;
  int n_slots;
  const uint8_t *PS1, *PS3, *PS2;
  int32_t *state, *miss_list, *pool_counts;
};

// Shared memory of the fused kernel (bytes from the 1024-aligned base).  Before
// the first weight box lands in it, the ring also holds a lone router pair's
// rows (step 1) and the logits the CTA selects from (step 3).
struct LayerPlan {
  int KBu, KBd;      // MX blocks per row: up (K = d), down (K = d_ff)
  int bpsu, bpsd;    // blocks per reduction split
  int PP;            // decoded-scale row pitch (u32)
  int sc_pitch;      // raw scale bytes of one matrix of an up unit (half a down unit), padded
  int nraw;          // raw scale buffers (two for the short units of RG = 1)
  size_t raw_off, pairs_off, red_off, bytes;
};

__host__ __device__ inline int imax(int a, int b) { return a > b ? a : b; }

__host__ __device__ inline LayerPlan layer_plan(int d, int d_ff, int rg, int fmt) {
  LayerPlan p;
  const int ks = DV_WARPS / rg;
  p.KBu = d / 32;
  p.KBd = d_ff / 32;
  // an even split point keeps every warp's first raw scale byte 2-byte aligned
  p.bpsu = (((p.KBu + ks - 1) / ks) + 1) & ~1;
  p.bpsd = (((p.KBd + ks - 1) / ks) + 1) & ~1;
  p.PP = (imax(p.bpsu, p.bpsd) + 7) & ~7;
  if (p.PP % 32 == 0) p.PP += 8;   // rows g and g + 1 of a quarter-warp on other banks
  // (NVFP4: two E4M3 scale bytes per 16-byte chunk of 32 elements)
  p.sc_pitch = (16 * rg * imax(p.KBu, p.KBd) * (fmt == 1 ? 2 : 1) + 15) & ~15;
  p.nraw = rg == 1 ? 2 : 1;
  p.raw_off = (size_t)DV_WARPS * DV_STAGES * 2 * DV_BOX;
  p.pairs_off = p.raw_off + (size_t)p.nraw * 2 * p.sc_pitch;
  p.red_off = p.pairs_off + (size_t)DV_WARPS * 2 * 8 * p.PP * 4;
  const int red_vals = ks == 2 ? 4 : 8;
  // (at least the selection's scratch: 256 indices, 256 counts, 256 offsets)
  p.bytes = p.red_off + (size_t)2 * DV_WARPS * red_vals * 32 * 4;
  return p;
}

struct Unit {
  int kind;   // 0 up, 1 down
  int sl;     // index into the active-expert list
  int rb;     // row block
};

// Unit u of the claim order: every up unit (expert by expert), then every
// down unit in the same expert order (nbu up and nbd down row blocks per
// expert).  A down unit is claimed at least (A - 1) * nbd claims after the
// last up unit of its expert, so it rarely waits, and a CTA waiting on one
// never holds an up unit back.
__device__ __forceinline__ Unit unit_of(int u, int A, int nbu, int nbd) {
  if (u < A * nbu) return Unit{0, u / nbu, u - (u / nbu) * nbu};
  const int v = u - A * nbu;
  return Unit{1, v / nbd, v - (v / nbd) * nbd};
}

__device__ __forceinline__ uint4 ld_cg_u4(const void *p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_cg_u32(const void *p) {
  uint32_t r;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Barrier over the grid's CTAs on a zeroed per-launch counter.  A wait that
// runs out records MOE_ERR_TIMEOUT and lets the CTA go on (its results are
// then reported invalid).
__device__ void grid_barrier(int *ctr, int *status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1);
    const int target = (int)gridDim.x;
    if (ld_acquire(ctr) < target) {
      const uint64_t t0 = tc::globaltimer();
      while (ld_acquire(ctr) < target) {
        if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
          set_status(status, MOE_ERR_TIMEOUT, -1);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// FMT: 0 MXFP4 (E8M0 scale per 32 elements), 1 NVFP4 (E4M3 scale per 16, fp32
// scale per matrix), as in the two-kernel FFN.
template <int RG, bool POOL, int FMT>
__global__ void __launch_bounds__(LY_THREADS, 2)
decode_layer_kernel(const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm3,
                    const __grid_constant__ CUtensorMap tm2, const __grid_constant__ CUtensorMap tp1,
                    const __grid_constant__ CUtensorMap tp3, const __grid_constant__ CUtensorMap tp2,
                    LayerArgs a) {
  constexpr int KS = DV_WARPS / RG;
  constexpr int RV = KS == 2 ? 4 : 8;   // partial sums a warp hands over per lane
  constexpr int UROWS = 16 * RG;        // W1 (and W3) rows of an up unit
  constexpr int DROWS = 32 * RG;        // W2 rows of a down unit
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ uint64_t full[DV_WARPS][DV_STAGES];
  __shared__ uint64_t sbar[2];
  __shared__ int s_abort, s_nactive, s_nclaimed;
  __shared__ unsigned s_raw_done;
  __shared__ int s_claim[LY_NQ];
  // per active expert: id, segment start and length (< 2^15); per segment
  // position: the token; per pair: its segment position
  __shared__ int16_t s_active[256], s_beg[256], s_cnt[256];
  __shared__ int16_t s_row[kDecodeMaxPairs], s_inv[kDecodeMaxPairs];
  __shared__ float s_gate[kDecodeMaxPairs];
  __shared__ int16_t s_slot[POOL ? 256 : 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = a.n, d = a.d, d_ff = a.d_ff, E = a.E, k = a.k, P = n * k;
  uint8_t *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
  volatile int *abort = &s_abort;
  const LayerPlan plan = layer_plan(d, d_ff, RG, FMT);
  constexpr int SPC = FMT == 1 ? 2 : 1;   // scale bytes per 16-byte code chunk
  // until the units start, the reduction buffer holds the selection's
  // indices and the per-expert counts and offsets
  int32_t *s_idx = reinterpret_cast<int32_t *>(smem + plan.red_off);   // [kDecodeMaxPairs]
  int *s_ecnt = s_idx + kDecodeMaxPairs;                                // [256]
  int *s_eoff = s_ecnt + 256;                                           // [256]

  if (tid == 0) {
    tc::prefetch_tmap(&tm1);
    tc::prefetch_tmap(&tm3);
    tc::prefetch_tmap(&tm2);
    if constexpr (POOL) {
      tc::prefetch_tmap(&tp1);
      tc::prefetch_tmap(&tp3);
      tc::prefetch_tmap(&tp2);
    }
    s_abort = 0;
    s_raw_done = 0;
    s_nclaimed = 0;
    tc::mbar_init(&sbar[0], 1);
    tc::mbar_init(&sbar[1], 1);
  }
  if (lane == 0) {
    for (int st = 0; st < DV_STAGES; ++st) tc::mbar_init(&full[warp][st], 1);
    tc::fence_mbar_init();
  }

  // ---- 1. router logits and the f16 x rows.  Pair (token t, expert e) =
  // t * E + e goes to warp (pair mod the grid's warps), spread over the CTAs
  // first; a warp keeps its expert's router row in registers while the
  // expert stays the same.  With at most one pair per CTA, the CTA's threads
  // stage the pair's router row and x row in shared memory instead (one round
  // of loads rather than a warp's three), and warp 0 adds them up in the
  // same per-lane piece order: the same logits.
  {
    const int vpr = d / 8, nv = (vpr - lane + 31) / 32;   // lane's pieces: lane + 32 v
    const int nw = (int)gridDim.x * DV_WARPS;
    const bool staged = n * E <= (int)gridDim.x;
    if (staged && (int)blockIdx.x < n * E) {
      const int t = (int)blockIdx.x / E, e = (int)blockIdx.x - t * E;
      uint4 *sw = reinterpret_cast<uint4 *>(smem);   // [vpr] in the ring, unused until step 3
      uint4 *sx = sw + vpr;                          // [vpr]
      const uint4 *wrow = reinterpret_cast<const uint4 *>(a.Wg + (size_t)e * d);
      const uint4 *xrow = reinterpret_cast<const uint4 *>(a.x + (size_t)t * d);
      for (int i = tid; i < vpr; i += LY_THREADS) {
        sw[i] = __ldg(wrow + i);
        sx[i] = __ldg(xrow + i);
      }
      __syncthreads();
      if (warp == 0) {
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < LY_RW; ++v)
          if (v < nv) acc += bf16x8_dot(sw[lane + 32 * v], sx[lane + 32 * v]);
        acc = warp_sum_xor(acc);
        if (lane == 0) a.logits[(size_t)t * E + e] = acc + (a.bias ? a.bias[e] : 0.f);
      }
    }
    uint4 wv[LY_RW];
    int cur = -1;
    for (int pr = staged ? n * E : warp * (int)gridDim.x + (int)blockIdx.x; pr < n * E; pr += nw) {
      const int t = pr / E, e = pr - t * E;
      if (e != cur) {
        const uint4 *wrow = reinterpret_cast<const uint4 *>(a.Wg + (size_t)e * d);
#pragma unroll
        for (int v = 0; v < LY_RW; ++v)
          if (v < nv) wv[v] = __ldg(wrow + lane + 32 * v);
        cur = e;
      }
      // the x row's pieces in two halves (fewer live registers), added in
      // piece order
      const uint4 *xrow = reinterpret_cast<const uint4 *>(a.x + (size_t)t * d);
      float acc = 0.f;
#pragma unroll
      for (int h = 0; h < LY_RW; h += LY_RW / 2) {
        uint4 xa[LY_RW / 2];
#pragma unroll
        for (int v = 0; v < LY_RW / 2; ++v)
          if (h + v < nv) xa[v] = __ldg(xrow + lane + 32 * (h + v));
#pragma unroll
        for (int v = 0; v < LY_RW / 2; ++v)
          if (h + v < nv) acc += bf16x8_dot(wv[h + v], xa[v]);
      }
      acc = warp_sum_xor(acc);
      if (lane == 0) a.logits[(size_t)t * E + e] = acc + (a.bias ? a.bias[e] : 0.f);
    }
    const int nvec = n * vpr;
    const uint4 *xv = reinterpret_cast<const uint4 *>(a.x);
    uint4 *x16v = reinterpret_cast<uint4 *>(a.x16);
    for (int i = blockIdx.x * LY_THREADS + tid; i < nvec; i += gridDim.x * LY_THREADS)
      x16v[i] = bf16x8_to_f16x8_checked(__ldg(xv + i), a.status, i / vpr);
  }

  // ---- 2. every logit and f16 row is stored
  grid_barrier(&a.sync[SY_BAR1], a.status);

  // ---- 3. selection and the stable dispatch, in every CTA: the same code on
  // the same logits gives the same arrays in every CTA; CTA 0 writes them
  // out.  Warp w selects tokens w, w + 8 (at most 16 tokens) from the logits
  // staged in shared memory (the ring, before the first weight box).
  {
    float *lg = reinterpret_cast<float *>(smem);   // [n][E]
    {
      // all of a thread's logits in flight at once (n * E <= 16 * 256)
      constexpr int LB = LY_MAX_TOKENS * 256 / LY_THREADS;
      uint32_t r[LB];
#pragma unroll
      for (int j = 0; j < LB; ++j)
        if (tid + j * LY_THREADS < n * E) r[j] = ld_cg_u32(a.logits + tid + j * LY_THREADS);
#pragma unroll
      for (int j = 0; j < LB; ++j)
        if (tid + j * LY_THREADS < n * E) lg[tid + j * LY_THREADS] = __uint_as_float(r[j]);
    }
    for (int e = tid; e < 256; e += LY_THREADS) s_ecnt[e] = 0;
    __syncthreads();
    for (int t = warp; t < n; t += DV_WARPS)
      select_topk_warp(lg + (size_t)t * E, E, k, a.gate_mode, lane, s_idx + t * k, s_gate + t * k,
                       nullptr);
    __syncthreads();
    for (int p = tid; p < P; p += LY_THREADS) {
      const int e = s_idx[p];
      if (e >= 0 && e < E) atomicAdd(&s_ecnt[e], 1);
      else if (blockIdx.x == 0) set_status(a.status, MOE_ERR_BAD_INDEX, p);   // (never: selection)
      if (blockIdx.x == 0) {
        a.topk_idx[p] = e;
        a.topk_gate[p] = s_gate[p];
      }
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive prefix sum of the counts (lane l owns experts 8l .. 8l+7)
      int c[8], run = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = s_ecnt[8 * lane + j];
        run += c[j];
      }
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int base = incl - run;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = 8 * lane + j;
        s_eoff[e] = base;
        if (blockIdx.x == 0 && e < E) {
          a.counts[e] = c[j];
          a.offsets[e] = base;
        }
        base += c[j];
      }
      if (blockIdx.x == 0 && lane == 31) a.offsets[E] = incl;
      __syncwarp();
      // the experts with tokens, in order
      int seen = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int ce = e < E ? s_ecnt[e] : 0;
        const unsigned m = __ballot_sync(0xffffffffu, ce > 0);
        if (ce > 0) {
          const int q = seen + __popc(m & lanemask_lt());
          s_active[q] = (int16_t)e;
          s_beg[q] = (int16_t)s_eoff[e];
          s_cnt[q] = (int16_t)ce;
        }
        seen += __popc(m);
      }
      if (lane == 0) s_nactive = seen;
    }
    if constexpr (POOL) {
      if (warp == 1 && blockIdx.x == 0)
        classify_warp(s_ecnt, E, a.slot_of, a.n_slots, P, a.state, a.miss_list, a.pool_counts,
                      a.status);
    }
    __syncthreads();
    if constexpr (POOL) {
      // each active expert's pool slot (-1: read from the backing arrays); a
      // slot outside the pool is reported and the backing expert read
      for (int q = tid; q < s_nactive; q += LY_THREADS) {
        const int e = s_active[q], sl = a.slot_of[e];
        if (sl < -1 || sl >= a.n_slots) set_status(a.status, MOE_ERR_BAD_INDEX, e);
        s_slot[q] = (int16_t)((sl >= 0 && sl < a.n_slots) ? sl : -1);
      }
    }
    // the ring was read and written through the generic proxy; the TMA
    // engine writes it next
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
  }

  // ---- 4. the expert units
  const int A = s_nactive;
  const int nbu = (d_ff + UROWS - 1) / UROWS, nbd = (d + DROWS - 1) / DROWS;
  const int total = A * (nbu + nbd);
  const int NRAW = plan.nraw, PP = plan.PP, scp = plan.sc_pitch;
  const int grp = warp / KS, split = warp - grp * KS;
  // this warp's share of the reduction in either kind of unit
  const int bbu = min(plan.KBu, split * plan.bpsu), nblu = min(plan.KBu, bbu + plan.bpsu) - bbu;
  const int bbd = min(plan.KBd, split * plan.bpsd), nbld = min(plan.KBd, bbd + plan.bpsd) - bbd;
  const int nslu = (nblu + 7) / 8, nsld = (nbld + 7) / 8;
  uint8_t *ring = smem + (size_t)warp * DV_STAGES * 2 * DV_BOX;
  uint32_t *pw = reinterpret_cast<uint32_t *>(smem + plan.pairs_off) + (size_t)warp * 2 * 8 * PP;
  float *red = reinterpret_cast<float *>(smem + plan.red_off);   // [2][DV_WARPS][RV][32]
  const int g = lane >> 2, t = lane & 3;
  const uint32_t lane_off = (uint32_t)(g * DV_BOXB + (g << 4) + 4 * t);
  int *up_done = a.sync + SY_UPDONE;

  // claim j of this CTA is published once s_nclaimed > j
  auto wait_claim = [&](int j) -> bool {
    const volatile int *nc = &s_nclaimed;
    if (*nc > j) {
      __threadfence_block();
      return true;
    }
    const uint64_t t0 = tc::globaltimer();
    while (*nc <= j) {
      if (*abort) return false;
      if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
        *abort = 1;
        return false;
      }
    }
    __threadfence_block();
    return true;
  };

  // raw scale bytes of claim j (E8M0, or E4M3 pairs) into buffer j % NRAW (a
  // thread drains the copies it issued on abort)
  int raw_mine0 = -1, raw_mine1 = -1;
  auto fetch_raw = [&](int j) {
    const int u = s_claim[j % LY_NQ];
    if (u >= total) return;
    const Unit w = unit_of(u, A, nbu, nbd);
    const int e = s_active[w.sl];
    const int ps = POOL ? s_slot[w.sl] : -1;
    const int b = j % NRAW;
    uint8_t *dst = smem + plan.raw_off + (size_t)b * 2 * scp;
    if (w.kind == 0) {
      const int r0 = w.rb * UROWS, rows = min(UROWS, d_ff - r0);   // rows % 16 == 0
      const uint32_t bytes = (uint32_t)rows * plan.KBu * SPC;
      const size_t row = (size_t)(ps >= 0 ? ps : e) * d_ff + r0;
      const uint8_t *S1 = ps >= 0 ? a.PS1 : a.S1, *S3 = ps >= 0 ? a.PS3 : a.S3;
      tc::mbar_arrive_expect_tx(&sbar[b], 2 * bytes);
      bulk_load(dst, S1 + row * plan.KBu * SPC, bytes, &sbar[b]);
      bulk_load(dst + scp, S3 + row * plan.KBu * SPC, bytes, &sbar[b]);
    } else {
      const int r0 = w.rb * DROWS, rows = min(DROWS, d - r0);
      const uint32_t bytes = (uint32_t)rows * plan.KBd * SPC;
      const size_t row = (size_t)(ps >= 0 ? ps : e) * d + r0;
      tc::mbar_arrive_expect_tx(&sbar[b], bytes);
      bulk_load(dst, (ps >= 0 ? a.PS2 : a.S2) + row * plan.KBd * SPC, bytes, &sbar[b]);
    }
    if (b) raw_mine1 = j;
    else raw_mine0 = j;
  };

  // The producer (lane 0 of each warp) keeps up to DV_STAGES of the warp's
  // slots in flight: claim i, pass, slot c of the pass, the first weight row
  // of the warp's group, slots issued.  It never waits: a claim not yet
  // published is picked up on a later call (each consumed slot and each unit
  // start call fill), and units in which this warp has no MX blocks are skipped.
  struct {
    int i, pass, c, passes, wrow, issued, kind, nslot, bb;
    bool valid, done, active, pool;
  } Pr{};
  auto try_load = [&]() -> bool {
    for (;;) {
      if (*reinterpret_cast<volatile int *>(&s_nclaimed) <= Pr.i) return false;
      __threadfence_block();
      const int u = s_claim[Pr.i % LY_NQ];
      if (u >= total) {
        Pr.done = true;
        return false;
      }
      const Unit w = unit_of(u, A, nbu, nbd);
      Pr.nslot = w.kind ? nsld : nslu;
      if (Pr.nslot == 0) {
        ++Pr.i;
        continue;
      }
      const int R = w.kind ? d : d_ff;
      const int r = w.kind ? w.rb * DROWS + grp * 32 : w.rb * UROWS + grp * 16;
      const int ps = POOL ? s_slot[w.sl] : -1;
      Pr.valid = true;
      Pr.kind = w.kind;
      Pr.bb = w.kind ? bbd : bbu;
      Pr.active = r < R;
      Pr.pool = ps >= 0;
      Pr.wrow = (ps >= 0 ? ps : (int)s_active[w.sl]) * R + r;
      Pr.passes = (s_cnt[w.sl] + DV_TOK - 1) / DV_TOK;
      Pr.c = 0;
      Pr.pass = 0;
      return true;
    }
  };
  auto fill = [&](int consumed_slots) {
    while (!Pr.done && Pr.issued - consumed_slots < DV_STAGES) {
      if (!Pr.valid && !try_load()) return;
      const int sl = Pr.issued & (DV_STAGES - 1);
      if (Pr.active) {
        tc::mbar_arrive_expect_tx(&full[warp][sl], 2 * DV_BOX);
        uint8_t *dst = ring + (size_t)sl * 2 * DV_BOX;
        const int x = (Pr.bb + 8 * Pr.c) * 16;   // a multiple of 16 bytes
        const int y = Pr.wrow;
        // each copy names its tensor map directly (a kernel-parameter
        // address); a box past the end of the row reads zeros
        if (Pr.kind == 0) {
          if (POOL && Pr.pool) {
            tc::tma_load_2d(&tp1, &full[warp][sl], dst, x, y);
            tc::tma_load_2d(&tp3, &full[warp][sl], dst + DV_BOX, x, y);
          } else {
            tc::tma_load_2d(&tm1, &full[warp][sl], dst, x, y);
            tc::tma_load_2d(&tm3, &full[warp][sl], dst + DV_BOX, x, y);
          }
        } else if (POOL && Pr.pool) {
          tc::tma_load_2d(&tp2, &full[warp][sl], dst, x, y);
          tc::tma_load_2d(&tp2, &full[warp][sl], dst + DV_BOX, x, y + 16);
        } else {
          tc::tma_load_2d(&tm2, &full[warp][sl], dst, x, y);
          tc::tma_load_2d(&tm2, &full[warp][sl], dst + DV_BOX, x, y + 16);
        }
      } else {
        tc::mbar_arrive(&full[warp][sl]);   // a group past the last row: keep the phases in step
      }
      ++Pr.issued;
      if (++Pr.c == Pr.nslot) {
        Pr.c = 0;
        if (++Pr.pass == Pr.passes) {
          ++Pr.i;
          Pr.valid = false;
        }
      }
    }
  };

  // the first NRAW claims are static (units b, b + G, ...), the rest come
  // from the queue, which counts from NRAW * G: each CTA's claims still rise
  // in the claim order
  if (tid == 0) {
    for (int j = 0; j < NRAW; ++j) s_claim[j] = (int)blockIdx.x + j * (int)gridDim.x;
    s_nclaimed = NRAW;
  }
  __syncthreads();
  // the first units' weights start streaming while the last warp finishes
  // the dispatch: stable positions, a pair's rank among equal experts being
  // the number of earlier pairs with that expert
  if (tid == 0)
    for (int j = 0; j < NRAW; ++j) fetch_raw(j);
  if (lane == 0) fill(0);
  if (warp == DV_WARPS - 1) {   // (not warp 0, whose thread 0 issued the scale copies)
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      int e = p < P ? s_idx[p] : -1;
      if (e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int pos = s_eoff[e] + __popc(peers & lanemask_lt());
        s_row[pos] = (int16_t)(p / k);
        s_inv[p] = (int16_t)pos;
        if (blockIdx.x == 0) {
          a.perm[pos] = p;
          a.inv_perm[p] = pos;
        }
      } else if (p < P) {
        s_inv[p] = -1;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) s_eoff[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  int consumed = 0, npass = 0;
  int pending = -1;   // expert of an up unit whose h rows are stored but not yet counted
  int16_t pend[LY_NPEND];   // (the group's counting thread) experts noted, not yet counted
  int npend = 0;
  bool ok = true;

  for (int i = 0;; ++i) {
    // this unit's claim, then its scale bytes (wait for the raw copy); the
    // warps of a group leave together, so none waits on a barrier alone
    const bool okc = __all_sync(0xffffffffu, wait_claim(i));
    const int u = okc ? s_claim[i % LY_NQ] : total;
    bool oks = true;
    if (okc && u < total)
      oks = __all_sync(0xffffffffu,
                       tc::mbar_wait(&sbar[i % NRAW], (uint32_t)((i / NRAW) & 1), abort));
    ok = okc && oks;
    if (group_sync_or(grp, 32 * KS, !ok)) {
      ok = false;
      break;
    }
    // Counting the previous unit's h rows (up units).  Every warp of the
    // group stored its rows before this barrier, so a fence by one thread
    // orders them all before the expert's count.  The fence stalls that
    // thread until the stores have landed, so far from the first down unit
    // (more than two grid rounds before it in the claim order, where no down
    // unit can be waiting yet) the group's thread only notes the expert, and
    // counts its notes behind one fence at its first unit past that point
    // (or when its list is full, or when it leaves).
    if (split == 0 && lane == 0 && (pending >= 0 || npend > 0)) {
      const bool early = u < A * nbu - 2 * (int)gridDim.x;
      if (early && pending >= 0 && npend < LY_NPEND) {
        pend[npend++] = (int16_t)pending;
      } else if (!early || pending >= 0) {
        __threadfence();
        for (int j = 0; j < npend; ++j) atomicAdd(up_done + pend[j], 1);
        npend = 0;
        if (pending >= 0) atomicAdd(up_done + pending, 1);
      }
    }
    pending = -1;
    if (u >= total) break;
    const Unit w = unit_of(u, A, nbu, nbd);
    const int kind = w.kind;
    const int e = s_active[w.sl], beg = s_beg[w.sl], cnt = s_cnt[w.sl];
    const int KB = kind ? plan.KBd : plan.KBu;
    const int R = kind ? d : d_ff;
    const int bb = kind ? bbd : bbu, nbl = kind ? nbld : nblu, nslot = kind ? nsld : nslu;
    const int r0 = kind ? w.rb * DROWS + grp * 32 : w.rb * UROWS + grp * 16;
    const bool active = r0 < R;
    // the first slot's activation lines into L1 (x rows are final from the
    // start; h rows only once the expert's count is complete, further down)
    auto prefetch_first = [&]() {
      const int pft = min(lane >> 2, cnt - 1);
      const uint16_t *xp = (kind ? a.h16 + (size_t)(beg + pft) * d_ff
                                 : a.x16 + (size_t)s_row[beg + pft] * d) +
                           (size_t)bb * 32 + (lane & 3) * 64;
      if (active && (lane & 3) * 2 < nbl) asm volatile("prefetch.global.L1 [%0];" ::"l"(xp));
    };
    if (kind == 0) prefetch_first();

    // decode this warp's part of the scales (MXFP4: bf16 pairs row g | row
    // g + 8; NVFP4: byte pairs per block parity, as the two-kernel FFN); the
    // last warp done claims the unit that reuses the buffer and issues its copy
    {
      // matrix m of the warp's group: W1 / W3 (up), or rows 0..15 / 16..31 of
      // the group (down), at the warp's first block
      const uint8_t *buf = smem + plan.raw_off + (size_t)(i % NRAW) * 2 * scp;
      const int gg = lane >> 2, q = lane & 3;
      auto raw_row = [&](int m) -> const uint8_t * {
        return kind ? buf + ((size_t)(grp * 32 + 16 * m + gg) * KB + bb) * SPC
                    : buf + (size_t)m * scp + ((size_t)(grp * 16 + gg) * KB + bb) * SPC;
      };
      if constexpr (FMT == 1) {
        // lane (gg, q) takes chunks q, q + 4, ... of row pair gg; a chunk's two
        // scale bytes of row gg and of row gg + 8 become two byte pairs, one
        // per block parity, stored [matrix][row pair][parity][chunk]
        uint16_t *pw16 = reinterpret_cast<uint16_t *>(pw);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint8_t *src = raw_row(m);
          uint16_t *dst16 = pw16 + (size_t)(m * 8 + gg) * 2 * PP;
          for (int b = q; b < nbl; b += 4) {
            const uint32_t x = *reinterpret_cast<const uint16_t *>(src + 2 * b);
            const uint32_t y = *reinterpret_cast<const uint16_t *>(src + 2 * b + 16 * KB);
            dst16[b] = (uint16_t)__byte_perm(x, y, 0x0040);
            dst16[PP + b] = (uint16_t)__byte_perm(x, y, 0x0051);
          }
        }
      } else {
      const bool even = (KB & 1) == 0;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint8_t *src = raw_row(m);
        uint32_t *dstp = pw + (m * 8 + gg) * PP;
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
          if (two) *reinterpret_cast<uint2 *>(dstp + b) = make_uint2(p0, p1);
          else dstp[b] = p0;
        }
      }
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&s_raw_done, 1u) == (unsigned)((i + 1) * DV_WARPS - 1)) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int j = i + NRAW;
        const int prev = s_claim[(j - 1) % LY_NQ];
        s_claim[j % LY_NQ] =
            prev >= total ? prev : NRAW * (int)gridDim.x + atomicAdd(&a.sync[SY_QUEUE], 1);
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&s_nclaimed) = j + 1;
        fetch_raw(j);
      }
    }
    if (lane == 0) fill(consumed);   // this unit's claim is published: its slots can go out
    if (kind == 1) {
      // every up unit of this expert has stored its h rows
      const int need = nbu * RG;
      bool dok = true;
      if (ld_acquire(up_done + e) < need) {
        const uint64_t t0 = tc::globaltimer();
        while (ld_acquire(up_done + e) < need) {
          if (*abort) {
            dok = false;
            break;
          }
          if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
            *abort = 1;
            dok = false;
            break;
          }
        }
      }
      ok = __all_sync(0xffffffffu, dok);
      if (group_sync_or(grp, 32 * KS, !ok)) {
        ok = false;
        break;
      }
      prefetch_first();
    }
    const uint32_t *pr1 = pw + g * PP;
    const uint32_t *pr3 = pr1 + 8 * PP;
    // NVFP4: this lane's block parity (t / 2) row of byte pairs, and the
    // unit's matrix scales (W1 and W3, or W2 for both halves)
    const uint16_t *pn1 = reinterpret_cast<const uint16_t *>(pw) + (size_t)(g * 2 + (t >> 1)) * PP;
    const uint16_t *pn3 = pn1 + (size_t)8 * 2 * PP;
    float gs1 = 1.f, gs3 = 1.f;
    if constexpr (FMT == 1) {
      gs1 = kind ? a.G2[e] : a.G1[e];
      gs3 = kind ? gs1 : a.G3[e];
    }

    for (int tg = 0; tg < cnt; tg += DV_TOK, ++npass) {
      // token g of this pass, or the pass's last token where g is past it (its
      // results are not stored)
      const int tok = tg + min(g, cnt - tg - 1);
      const uint16_t *xbase = kind ? a.h16 : a.x16;
      const int xpitch = kind ? d_ff : d;
      const uint16_t *xrow = xbase + (size_t)(kind ? beg + tok : s_row[beg + tok]) * xpitch +
                             (size_t)bb * 32 + 8 * t;
      const int pft = tg + min(lane >> 2, cnt - tg - 1);   // prefetch: lane's token, 2-block line
      const uint16_t *xpf = xbase + (size_t)(kind ? beg + pft : s_row[beg + pft]) * xpitch +
                            (size_t)bb * 32 + (lane & 3) * 64;
      float acc1[4] = {0.f, 0.f, 0.f, 0.f}, acc3[4] = {0.f, 0.f, 0.f, 0.f};
      uint4 bx[8];
      // (plain, L1-cached loads: the rows were published to this warp by an
      // acquire -- the grid barrier for x, the expert's counter for h)
      auto load_bx = [&](int cb, int nb) {
        const uint16_t *xb = xrow + cb * 32;
#pragma unroll
        for (int bl = 0; bl < 8; ++bl)
          bx[bl] = (bl < nb) ? *reinterpret_cast<const uint4 *>(xb + bl * 32)
                             : make_uint4(0u, 0u, 0u, 0u);
      };
      // the 8-block group at local block cb: matrix 1 in box sw, matrix 3
      // (W3, or the group's rows 16..31) in the box after it
      auto compute8 = [&](const uint8_t *sw, int cb, int nb) {
        if constexpr (FMT == 1) {
          const uint4 n1 = *reinterpret_cast<const uint4 *>(pn1 + cb);
          const uint4 n3 = *reinterpret_cast<const uint4 *>(pn3 + cb);
          // the eight chunks' scale pairs {s_g, s_g+8} as f16x2
          const uint2 f1a = e4m3x4_to_f16x2x2(n1.x), f1b = e4m3x4_to_f16x2x2(n1.y),
                      f1c = e4m3x4_to_f16x2x2(n1.z), f1d = e4m3x4_to_f16x2x2(n1.w);
          const uint2 f3a = e4m3x4_to_f16x2x2(n3.x), f3b = e4m3x4_to_f16x2x2(n3.y),
                      f3c = e4m3x4_to_f16x2x2(n3.z), f3d = e4m3x4_to_f16x2x2(n3.w);
          const uint32_t f1[8] = {f1a.x, f1a.y, f1b.x, f1b.y, f1c.x, f1c.y, f1d.x, f1d.y};
          const uint32_t f3[8] = {f3a.x, f3a.y, f3b.x, f3b.y, f3c.x, f3c.y, f3d.x, f3d.y};
          auto block = [&](int bl) {
            const uint8_t *wp = sw + (lane_off ^ (uint32_t)(bl << 4));
            const uint32_t wg = *reinterpret_cast<const uint32_t *>(wp);
            const uint32_t wh = *reinterpret_cast<const uint32_t *>(wp + 8 * DV_BOXB);
            nv_block(acc1, wg, wh, f1[bl], bx[bl]);
            const uint32_t vg = *reinterpret_cast<const uint32_t *>(wp + DV_BOX);
            const uint32_t vh = *reinterpret_cast<const uint32_t *>(wp + DV_BOX + 8 * DV_BOXB);
            nv_block(acc3, vg, vh, f3[bl], bx[bl]);
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
        const uint4 s3a = *reinterpret_cast<const uint4 *>(pr3 + cb);
        const uint4 s3b = *reinterpret_cast<const uint4 *>(pr3 + cb + 4);
        const uint32_t sp1[8] = {s1a.x, s1a.y, s1a.z, s1a.w, s1b.x, s1b.y, s1b.z, s1b.w};
        const uint32_t sp3[8] = {s3a.x, s3a.y, s3a.z, s3a.w, s3b.x, s3b.y, s3b.z, s3b.w};
        auto block = [&](int bl) {
          const uint8_t *wp = sw + (lane_off ^ (uint32_t)(bl << 4));
          const uint32_t wg = *reinterpret_cast<const uint32_t *>(wp);
          const uint32_t wh = *reinterpret_cast<const uint32_t *>(wp + 8 * DV_BOXB);
          mx_block(acc1, wg, wh, __uint_as_float(sp1[bl] << 16),
                   __uint_as_float(sp1[bl] & 0xffff0000u), bx[bl]);
          const uint32_t vg = *reinterpret_cast<const uint32_t *>(wp + DV_BOX);
          const uint32_t vh = *reinterpret_cast<const uint32_t *>(wp + DV_BOX + 8 * DV_BOXB);
          mx_block(acc3, vg, vh, __uint_as_float(sp3[bl] << 16),
                   __uint_as_float(sp3[bl] & 0xffff0000u), bx[bl]);
        };
        if (nb == 8) {
#pragma unroll
          for (int bl = 0; bl < 8; ++bl) block(bl);
        } else {
#pragma unroll
          for (int bl = 0; bl < 8; ++bl)
            if (bl < nb) block(bl);
        }
      };
      for (int c = 0; c < nslot; ++c) {
        const int cb = c * 8;
        const int slot = consumed & (DV_STAGES - 1);
        const uint32_t parity = (uint32_t)(consumed / DV_STAGES) & 1u;
        ++consumed;
        if (active) {
          load_bx(cb, min(8, nbl - cb));
          // the next slot's activation lines: one 128-byte line (two blocks)
          // per lane
          if (c + 1 < nslot && (lane & 3) * 2 < nbl - (cb + 8))
            asm volatile("prefetch.global.L1 [%0];" ::"l"(xpf + (cb + 8) * 32));
        }
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&full[warp][slot], parity, abort));
        if (!ok) break;
        if (active) compute8(ring + (size_t)slot * 2 * DV_BOX, cb, min(8, nbl - cb));
        __syncwarp();
        if (lane == 0) {
          // the slot was read through the generic proxy; order those reads
          // before the TMA engine overwrites it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          fill(consumed);
        }
      }
      // partial sums of the group's warps, added in warp order (as the
      // two-kernel FFN: two splits hand each other a row, more splits give
      // both rows to the first two warps)
      float *rb = red + (size_t)(npass & 1) * DV_WARPS * RV * 32;
      float f1[2], f3[2];   // this warp's finished values: tokens 2t, 2t+1 of its row
      int frow;
      bool fin;
      if constexpr (KS == 2) {
        const bool s0 = split == 0;
        const float k10 = s0 ? acc1[0] : acc1[2], k11 = s0 ? acc1[1] : acc1[3];
        const float k30 = s0 ? acc3[0] : acc3[2], k31 = s0 ? acc3[1] : acc3[3];
        rb[(warp * RV + 0) * 32 + lane] = s0 ? acc1[2] : acc1[0];
        rb[(warp * RV + 1) * 32 + lane] = s0 ? acc1[3] : acc1[1];
        rb[(warp * RV + 2) * 32 + lane] = s0 ? acc3[2] : acc3[0];
        rb[(warp * RV + 3) * 32 + lane] = s0 ? acc3[3] : acc3[1];
        if (group_sync_or(grp, 32 * KS, !ok)) {
          ok = false;
          break;
        }
        const int pw_ = warp ^ 1;
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
        if (group_sync_or(grp, 32 * KS, !ok)) {
          ok = false;
          break;
        }
        fin = active && split < 2;
        const int q0 = split == 1 ? 2 : 0;
        f1[0] = f1[1] = f3[0] = f3[1] = 0.f;
        if (fin) {
#pragma unroll
          for (int w2 = 0; w2 < KS; ++w2) {
            const int ww = grp * KS + w2;
            f1[0] += rb[(ww * RV + q0) * 32 + lane];
            f1[1] += rb[(ww * RV + q0 + 1) * 32 + lane];
            f3[0] += rb[(ww * RV + 4 + q0) * 32 + lane];
            f3[1] += rb[(ww * RV + 4 + q0 + 1) * 32 + lane];
          }
        }
        frow = split == 1 ? g + 8 : g;
      }
      if (fin) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int tk = tg + 2 * t + q;
          if (tk >= cnt) continue;
          if (kind) {
            // rows r0 + frow (f1) and r0 + 16 + frow (f3) of y_perm
            a.y_perm[(size_t)(beg + tk) * d + r0 + frow] = __float2bfloat16_rn(f1[q] * gs1);
            a.y_perm[(size_t)(beg + tk) * d + r0 + 16 + frow] = __float2bfloat16_rn(f3[q] * gs3);
          } else {
            const int row = r0 + frow;
            const float a1 = f1[q] * gs1, a3 = f3[q] * gs3;   // NVFP4 matrix scales (else 1)
            const float v = a1 / (1.f + __expf(-a1)) * a3;
            if (row < R) {
              const __nv_bfloat16 hb = __float2bfloat16_rn(v);
              a.h[(size_t)(beg + tk) * d_ff + row] = hb;
              a.h16[(size_t)(beg + tk) * d_ff + row] =
                  f16_bits_checked(__bfloat162float(hb), a.status, beg + tk);
            }
          }
        }
      }
    }
    if (!ok) break;
    if (kind == 0) pending = e;   // counted at the next unit's first barrier
  }
  if (!ok) {
    // let the copies this warp issued land before it leaves the loop
    if (lane == 0) {
      for (int j = consumed; j < Pr.issued; ++j)
        tc::mbar_wait_drain(&full[warp][j % DV_STAGES], (uint32_t)(j / DV_STAGES) & 1u,
                            100000000ull);
      if (raw_mine0 >= 0)
        tc::mbar_wait_drain(&sbar[0], (uint32_t)((raw_mine0 / NRAW) & 1), 100000000ull);
      if (raw_mine1 >= 0)
        tc::mbar_wait_drain(&sbar[1], (uint32_t)((raw_mine1 / NRAW) & 1), 100000000ull);
      set_status(a.status, MOE_ERR_TIMEOUT, blockIdx.x);
    }
  }

  // ---- 5. every y_perm row is stored; combine
  grid_barrier(&a.sync[SY_BAR2], a.status);
  {
    const int vpr = d / 8;
    const uint4 *yp = reinterpret_cast<const uint4 *>(a.y_perm);
    uint4 *yo = reinterpret_cast<uint4 *>(a.y);
    for (int i = blockIdx.x * LY_THREADS + tid; i < n * vpr; i += gridDim.x * LY_THREADS) {
      const int tk = i / vpr, v = i - tk * vpr;
      float acc[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = 0.f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        int q[8];
        uint4 r[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = j0 + u < k ? (int)s_inv[tk * k + j0 + u] : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (q[u] >= 0) r[u] = ld_cg_u4(yp + (size_t)q[u] * vpr + v);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (q[u] < 0) continue;
          const float gt = s_gate[tk * k + j0 + u];
          const uint32_t ww[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[2 * c] = fmaf(gt, __uint_as_float(ww[c] << 16), acc[2 * c]);
            acc[2 * c + 1] = fmaf(gt, __uint_as_float(ww[c] & 0xffff0000u), acc[2 * c + 1]);
          }
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const __nv_bfloat162 hv = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
        o[c] = *reinterpret_cast<const uint32_t *>(&hv);
      }
      yo[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Rows per group step: RG = 4 (64 up rows, 128 down rows per unit) when that
// still gives every CTA two units on average, else 2 when every CTA gets one,
// else 1.  (The active experts are bounded by min(n k, E) here.)
int layer_rg(const moe_config &c, int ctas) {
  // NVFP4 units stay at 32 rows a side: their scale rows are twice as long
  const int max_rg = c.weight_dtype == MOE_NVFP4 ? 2 : 4;
  const long slots = (long)c.n * c.top_k < c.n_experts ? (long)c.n * c.top_k : c.n_experts;
  auto units = [&](int rg) {
    return slots * ((c.d_ff + 16 * rg - 1) / (16 * rg) + (c.d + 32 * rg - 1) / (32 * rg));
  };
  if (max_rg == 4 && units(4) >= 2L * ctas) return 4;
  if (units(2) >= ctas) return 2;
  return 1;
}

template <int RG, bool POOL, int FMT>
cudaError_t launch_layer(const LayerArgs &a, const CUtensorMap (&maps)[6], cudaStream_t s) {
  const size_t smem = 1024 + layer_plan(a.d, a.d_ff, RG, FMT).bytes;
  static size_t smem_set = 0;
  static int per_sm = 0;
  auto kern = decode_layer_kernel<RG, POOL, FMT>;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set = smem;
    per_sm = 0;
  }
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, LY_THREADS, smem) !=
            cudaSuccess ||
        per_sm < 1)
      return cudaErrorInvalidConfiguration;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(per_sm * num_sms()));
  cfg.blockDim = dim3(LY_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
}

}  // namespace

bool decode_layer_supported(const moe_config &c, bool pooled) {
  const bool fmt_ok = c.weight_dtype == MOE_MXFP4 || (c.weight_dtype == MOE_NVFP4 && !pooled);
  if (!decode_route_supported(c) || !fmt_ok || c.act != MOE_ACT_SWIGLU) return false;
  if (c.n > (c.weight_dtype == MOE_NVFP4 ? LY_MAX_TOKENS_NV : LY_MAX_TOKENS) || c.d > LY_MAX_D)
    return false;
  if (!tensor_maps_available()) return false;
  static int coop = -1;   // (per process, as the other launch settings)
  if (coop < 0) {
    int dev = 0, v = 0;
    coop = cudaGetDevice(&dev) == cudaSuccess &&
                   cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess
               ? (v != 0)
               : 0;
  }
  return coop != 0;
}

size_t decode_layer_sync_bytes() { return (size_t)(SY_UPDONE + 256) * sizeof(int); }

cudaError_t launch_decode_layer(const moe_config &c, const void *x, const moe_weights &w,
                                const moe_expert_pool *pool, const DecodeLayerBuffers &b,
                                cudaStream_t s) {
  LayerArgs a{};
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.Wg = static_cast<const __nv_bfloat16 *>(w.Wg);
  a.bias = w.router_bias;
  a.S1 = w.S1;
  a.S3 = w.S3;
  a.S2 = w.S2;
  a.G1 = w.G1;
  a.G3 = w.G3;
  a.G2 = w.G2;
  a.n = c.n;
  a.d = c.d;
  a.d_ff = c.d_ff;
  a.E = c.n_experts;
  a.k = c.top_k;
  a.gate_mode = (int)c.gate;
  a.logits = b.logits;
  a.topk_idx = b.topk_idx;
  a.topk_gate = b.topk_gate;
  a.counts = b.counts;
  a.offsets = b.offsets;
  a.perm = b.perm;
  a.inv_perm = b.inv_perm;
  a.x16 = static_cast<uint16_t *>(b.act16);
  a.h16 = a.x16 + (size_t)c.n * c.top_k * c.d;
  a.h = static_cast<__nv_bfloat16 *>(b.h);
  a.y_perm = static_cast<__nv_bfloat16 *>(b.y_perm);
  a.y = static_cast<__nv_bfloat16 *>(b.y);
  a.sync = b.sync;
  a.status = b.status;
  CUtensorMap maps[6];
  const uint32_t box[2] = {DV_BOXB, 16};
  const uint64_t dup[2] = {(uint64_t)c.d / 2, (uint64_t)c.n_experts * c.d_ff};
  const uint64_t ddn[2] = {(uint64_t)c.d_ff / 2, (uint64_t)c.n_experts * c.d};
  auto tmap = [&](CUtensorMap *m, const void *base, const uint64_t *dims) {
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, 2, dims, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
  };
  if (!tmap(&maps[0], w.W1, dup) || !tmap(&maps[1], w.W3, dup) || !tmap(&maps[2], w.W2, ddn))
    return cudaErrorInvalidValue;
  maps[3] = maps[0];
  maps[4] = maps[1];
  maps[5] = maps[2];
  if (pool) {
    const uint64_t pup[2] = {(uint64_t)c.d / 2, (uint64_t)pool->n_slots * c.d_ff};
    const uint64_t pdn[2] = {(uint64_t)c.d_ff / 2, (uint64_t)pool->n_slots * c.d};
    if (!tmap(&maps[3], pool->W1, pup) || !tmap(&maps[4], pool->W3, pup) ||
        !tmap(&maps[5], pool->W2, pdn))
      return cudaErrorInvalidValue;
    a.slot_of = pool->slot_of;
    a.n_slots = pool->n_slots;
    a.PS1 = pool->S1;
    a.PS3 = pool->S3;
    a.PS2 = pool->S2;
    a.state = b.state;
    a.miss_list = b.miss_list;
    a.pool_counts = b.pool_counts;
  }
  const int rg = layer_rg(c, 2 * num_sms());
  if (c.weight_dtype == MOE_NVFP4) {
    if (pool) return cudaErrorNotSupported;
    if (rg == 2) return launch_layer<2, false, 1>(a, maps, s);
    return launch_layer<1, false, 1>(a, maps, s);
  }
  if (pool) {
    if (rg == 4) return launch_layer<4, true, 0>(a, maps, s);
    if (rg == 2) return launch_layer<2, true, 0>(a, maps, s);
    return launch_layer<1, true, 0>(a, maps, s);
  }
  if (rg == 4) return launch_layer<4, false, 0>(a, maps, s);
  if (rg == 2) return launch_layer<2, false, 0>(a, maps, s);
  return launch_layer<1, false, 0>(a, maps, s);
}

}  // namespace moe
