/*
 * moe.h - C ABI of the GB300 (sm_103a) Mixture-of-Experts layer forward pass.
 *
 * The layer, as "How Mixture of Experts Scales Model Parameters" states it:
 *   X (n x d) -> router: one d x E linear layer, softmax per row
 *               ("Routing: a router scores the experts, and the top one runs")
 *             -> the K highest-scoring experts per token, their weights
 *                renormalised over the chosen K ("Top-K: several experts,
 *                added up by weight"), or, for top-1 Switch routing, the
 *                chosen expert's own probability ("Routing", 0.45 example)
 *             -> dispatch: tokens regrouped into one contiguous segment per
 *                expert, possibly empty ("The forward pass: dispatch, then
 *                combine")
 *             -> each expert's FFN d -> d_ff -> d on its segment ("Dense
 *                models: every parameter in the FFN does work for every token")
 *             -> combine: outputs scaled by their gate and put back in token
 *                order ("The forward pass: dispatch, then combine")
 *             -> Y (n x d).
 * MXFP4 expert weights (the feed post "What is MXFP4?": 4-bit floats in blocks
 * of 32 sharing a scale) use OCP MX v1.0 E2M1 elements and E8M0 scales.
 *
 * Conventions for every entry point
 *   - Pointers named x, W*, y, ws, ... are DEVICE pointers (cudaMalloc or any
 *     allocator of the same context); cfg and w point to HOST structs.
 *   - Ownership: the caller owns every buffer, the workspace included.  The
 *     library never allocates, frees or synchronises, except moe_status_check.
 *   - Execution: launches are asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL = legacy default stream).  Nothing reads device data on
 *     the host, so calls can be captured into a CUDA graph.
 *   - Errors: argument checks run on the host before any launch and return
 *     MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE with
 *     nothing launched.  A failed launch returns MOE_ERR_CUDA.  Faults found
 *     on the device (an expert index out of range, a permutation entry out of
 *     range, a pipeline wait that ran out) are written to a sticky status word
 *     at the start of the workspace; kernels then skip the offending access
 *     and later kernels of the same workspace return early.  Read it with
 *     moe_status_check.  No kernel traps.
 *   - Threads and devices: the library keeps per-process launch settings
 *     (each kernel's configured shared-memory size and occupancy, the SM
 *     count) from its first calls.  Call it from one host thread at a time,
 *     on one device per process (a data-parallel job runs one process per
 *     GPU).
 *   - Layouts are row-major.  Weights are stored out x in, so the reduction
 *     dimension is contiguous: W1, W3 [E][d_ff][d]; W2 [E][d][d_ff]; Wg [E][d]
 *     (the router's d x E matrix, transposed).  The page's X.W1 uses W1^T of
 *     this storage.
 *   - Alignment: every device pointer must be 16-byte aligned; the workspace
 *     256-byte aligned.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or enum */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d % 32 != 0 with MXFP4) */
  MOE_ERR_WORKSPACE = 3,    /* ws_bytes smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, attribute, ...) */
  MOE_ERR_BAD_INDEX = 5,    /* device: expert index >= E or < 0, or perm entry out of range */
  MOE_ERR_TIMEOUT = 6,      /* device: a bounded pipeline wait ran out */
  MOE_ERR_RANGE = 7,        /* device: an MXFP4 block scale outside the range the
                               tensor-core path applies exactly (E8M0 byte 113..142) */
  MOE_ERR_F16_RANGE = 8     /* device: an activation (x or h) of an MXFP4 layer outside
                               the f16 range its tensor-core operands use (|v| > 65504,
                               or NaN); the value was clamped and y is not valid */
} moe_status;

/* NVFP4: the feed post "What is MXFP4?" names it as the block-of-16 variant
 * (blocks of 16 with their own scale); the scale byte is FP8 E4M3 (OCP 8-bit
 * floating point specification) and each expert matrix carries one fp32
 * scale.  Expert weights only, small batches only (n * top_k <= 256, bf16
 * activations): other NVFP4 configurations return MOE_ERR_UNSUPPORTED. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_MXFP4 = 2, MOE_NVFP4 = 3 } moe_dtype;

/* Gate rule. TOP_PROB: g = p of the chosen expert, unrenormalised (Switch
 * top-1; "Routing", output x 0.45).  RENORM: g_j = p_j / sum of the chosen p
 * ("Top-K", 0.45/0.76 and 0.31/0.76). */
typedef enum { MOE_GATE_TOP_PROB = 0, MOE_GATE_RENORM = 1 } moe_gate;

/* Expert activation.  RELU: h = max(x W1^T, 0).  SWIGLU: h = silu(x W1^T) *
 * (x W3^T), silu(a) = a / (1 + e^-a).  The pages name only "a nonlinear
 * activation"; SwiGLU's branch roles follow the Mixtral convention. */
typedef enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;

/* Layer shape.  All enum fields are stored as int32_t. */
typedef struct {
  int32_t n;            /* tokens (rows of X), >= 1 */
  int32_t d;            /* model dim */
  int32_t d_ff;         /* expert intermediate dim */
  int32_t n_experts;    /* E, 1..256 */
  int32_t top_k;        /* K, 1..E */
  int32_t act_dtype;    /* MOE_F32 or MOE_BF16: x, Wg, y, shared-expert weights */
  int32_t weight_dtype; /* routed expert weights: MOE_F32 (needs act F32), MOE_BF16, MOE_MXFP4,
                           MOE_NVFP4 */
  int32_t gate;         /* moe_gate */
  int32_t act;          /* moe_act */
  int32_t d_ff_shared;  /* 0: none; else one always-on SwiGLU expert added unweighted */
} moe_config;

/* Layer weights (device pointers).  Unused entries must be NULL. */
typedef struct {
  const void *Wg;            /* [E][d], act_dtype */
  const float *router_bias;  /* [E] fp32 added to the router logits, or NULL */
  const void *W1;            /* [E][d_ff][d] (f32/bf16) or FP4 codes [E][d_ff][d/2] */
  const void *W3;            /* as W1; SwiGLU only, else NULL */
  const void *W2;            /* [E][d][d_ff] (f32/bf16) or FP4 codes [E][d][d_ff/2] */
  const uint8_t *S1;         /* block scales of W1: MXFP4 E8M0 [E][d_ff][d/32], NVFP4 E4M3
                                [E][d_ff][d/16]; else NULL */
  const uint8_t *S3;         /* block scales of W3, as S1; else NULL */
  const uint8_t *S2;         /* block scales of W2: [E][d][d_ff/32] or [E][d][d_ff/16] */
  const void *Ws1;           /* shared expert [d_ff_shared][d], act_dtype, or NULL */
  const void *Ws3;           /* shared expert [d_ff_shared][d] */
  const void *Ws2;           /* shared expert [d][d_ff_shared] */
  const float *G1;           /* NVFP4: fp32 scale of each expert's W1 [E], else NULL */
  const float *G3;           /* NVFP4: of W3 [E] (SwiGLU), else NULL */
  const float *G2;           /* NVFP4: of W2 [E], else NULL */
} moe_weights;
/* MXFP4 codes: element i of a row sits in byte i/2, low nibble when i is even.
 * Scale byte s gives the 32 consecutive elements of its block 2^(s-127);
 * s = 255 (NaN) is not accepted and decodes to NaN.  NVFP4 codes are packed the
 * same way; element i of row r of expert e is e2m1(code) * e4m3(S[e][r][i/16])
 * * G[e]. */

/* Offsets (bytes from the workspace start) of the intermediates that
 * moe_forward leaves in the workspace, for inspection after a call. */
typedef struct {
  size_t status;     /* int32 status word (moe_status), then int32 detail */
  size_t logits;     /* fp32 [n][E] router logits (bias included) */
  size_t topk_idx;   /* int32 [n][K] */
  size_t topk_gate;  /* fp32  [n][K] */
  size_t counts;     /* int32 [E] */
  size_t offsets;    /* int32 [E+1] */
  size_t perm;       /* int32 [n*K]: segment position -> pair t*K+j */
  size_t inv_perm;   /* int32 [n*K]: pair t*K+j -> segment position */
  size_t x_perm;     /* act_dtype [n*K][d] (not written for MXFP4 layers, which
                        stage f16 rows in act16 instead) */
  size_t h;          /* [n*K][d_ff]: bf16, or fp32 when act_dtype is F32 */
  size_t y_perm;     /* act_dtype [n*K][d], unweighted expert outputs */
  size_t y_shared;   /* act_dtype [n][d] shared-expert output, 0 if none */
  size_t h_shared;   /* [n][d_ff_shared] shared-expert intermediate, 0 if none */
  size_t act16;      /* MXFP4 layers: f16 copies of the expert-ordered activation
                        rows [n*K][d] then of h [n*K][d_ff]; 0 for other layers */
  size_t total;      /* = moe_workspace_size() */
} moe_workspace_layout;

/* Bytes of workspace that moe_forward needs for `cfg` (enough for every other
 * entry point too).  Host-only; no CUDA call. */
moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes);

/* Region offsets inside that workspace.  Host-only. */
moe_status moe_workspace_layout_of(const moe_config *cfg, moe_workspace_layout *out);

/* Router: logits = x Wg^T (+ bias) accumulated in fp32, softmax per row
 * ("Routing"; the maximum is subtracted first), the top_k experts per row in
 * rank order (score descending, lower expert index first on equal fp32
 * scores), and their gates (cfg->gate).
 *   x [n][d] act_dtype; topk_idx int32 [n][K]; topk_gate fp32 [n][K];
 *   probs fp32 [n][E] or NULL (full softmax rows, for inspection).
 *   ws: a workspace of at least moe_workspace_size(cfg) bytes (scratch for
 *   the logits and the status word). */
moe_status moe_route(const moe_config *cfg, const void *x, const moe_weights *w,
                     int32_t *topk_idx, float *topk_gate, float *probs,
                     void *ws, size_t ws_bytes, void *stream);

/* Routing statistics of one batch ("How Mixture of Experts Scales Model
 * Parameters", section "Load balancing: how collapse happens, and how it's
 * kept in check"):
 *   P[i]  = (1/n) sum_t probs[t][i]            mean router probability
 *   f[i]  = (1/n) #{t : topk_idx[t][0] == i}   share of tokens whose argmax is i
 *   aux[0] = alpha * E * sum_i f[i] * P[i]      auxiliary load-balancing loss
 * probs fp32 [n][E] and topk_idx int32 [n][K] as produced by moe_route
 * (rank 0 of each row is the argmax).  P, f fp32 [E]; aux fp32 [1].  Sums run
 * in a fixed order (deterministic).  A top-1 index outside [0, E) sets
 * MOE_ERR_BAD_INDEX in the workspace status word. */
moe_status moe_route_stats(const moe_config *cfg, const float *probs, const int32_t *topk_idx,
                           float alpha, float *P, float *f, float *aux, void *ws,
                           size_t ws_bytes, void *stream);

/* moe_route without a workspace, for callers that cannot allocate device
 * memory: code running during CUDA graph capture under an allocator that is
 * not capture-safe, plugins handed only their input and output buffers by a
 * host runtime that owns all device memory, fixed-arena embedded runtimes.
 * (An addition of this library; the pages have no counterpart.)
 * Arguments as moe_route, minus ws/ws_bytes; the same selection rules.  The
 * router's reduction is never split over extra CTAs here (that needs scratch
 * for the partial sums), so on shapes where moe_route splits it the fp32
 * logits, probs and gates may differ from moe_route's in the last bits, and a
 * token whose top-k margin is at rounding level may rank differently.
 * The logits live in one file-scope device array of 16 MiB, and device-side
 * faults (a pipeline wait that ran out) in a file-scope status word; every GPU
 * loading the library holds both until exit.  n * n_experts above 4,194,304
 * returns MOE_ERR_WORKSPACE.  The first call on a device (with it current) in
 * a CUDA context looks up the arrays' addresses; make that call before any
 * stream capture.  Each call clears the status word on its stream first.  All
 * calls share the arrays: calls that overlap on the GPU race and must be
 * serialised by the caller.  No allocation, no synchronisation. */
moe_status moe_route_noalloc(const moe_config *cfg, const void *x, const moe_weights *w,
                             int32_t *topk_idx, float *topk_gate, float *probs, void *stream);

/* Synchronises `stream`, then returns the device status word of the last
 * moe_route_noalloc on the current device (MOE_OK, or MOE_ERR_TIMEOUT when a
 * wait of its router ran out and its outputs are not valid).  detail, if not
 * NULL, receives the detail word.  Allocates nothing. */
moe_status moe_route_noalloc_status(void *stream, int32_t *detail);

/* Dispatch ("The forward pass: dispatch, then combine"): a stable counting
 * sort of the n*K (token, slot) pairs by expert.  Bit-exact.
 *   topk_idx int32 [n][K] (any values; out-of-range ones set MOE_ERR_BAD_INDEX
 *   and are skipped); counts int32 [E]; offsets int32 [E+1] (exclusive prefix
 *   sum, offsets[E] = n*K); perm int32 [n*K] (position -> pair t*K+j, pairs of
 *   one expert in increasing pair order); inv_perm int32 [n*K] (its inverse);
 *   x_perm act_dtype [n*K][d] = x[perm[q] / K], or NULL to skip the gather.
 * From 16,384 pairs on the sort runs over one CTA per SM in two launches,
 * with its per-CTA counts in the workspace's h region (free at this point of
 * the forward); the arrays are the same either way. */
moe_status moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                        int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                        void *x_perm, void *ws, size_t ws_bytes, void *stream);

/* Expert FFNs over the dispatched segments: for each expert e and each
 * position q in [offsets[e], offsets[e+1]), y_perm[q] = FFN_e(x_perm[q])
 * (no gate applied).  The intermediate h is rounded to bf16 (fp32 when
 * act_dtype is F32) and kept in the workspace.  MXFP4 weights are decoded on
 * the fly.  x_perm, y_perm act_dtype [n*K][d]. */
moe_status moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets,
                          const moe_weights *w, void *y_perm,
                          void *ws, size_t ws_bytes, void *stream);

/* Combine ("The forward pass: dispatch, then combine"):
 *   y[t] = sum_{j=0..K-1} topk_gate[t][j] * y_perm[inv_perm[t*K+j]]  (+ y_shared[t])
 * summed in fp32 in slot order, rounded once to act_dtype.
 *   y_shared act_dtype [n][d] or NULL.  An inv_perm entry outside [0, n*K)
 *   sets MOE_ERR_BAD_INDEX (status word in ws) and that term is skipped. */
moe_status moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *inv_perm,
                       const float *topk_gate, const void *y_shared, void *y,
                       void *ws, size_t ws_bytes, void *stream);

/* The whole layer: route, dispatch, expert FFNs (+ shared expert), combine.
 * x [n][d] act_dtype in, y [n][d] act_dtype out.  Intermediates stay in the
 * workspace at moe_workspace_layout_of() offsets.  Clears the status word
 * first. */
moe_status moe_forward(const moe_config *cfg, const void *x, const moe_weights *w, void *y,
                       void *ws, size_t ws_bytes, void *stream);

/* Stages of moe_forward, in launch order. */
typedef enum {
  MOE_STAGE_ROUTE = 0,     /* router logits, softmax, top-k, gates */
  MOE_STAGE_DISPATCH = 1,  /* counting sort + gather of x rows (for MXFP4 prefill, their
                              f16 copies) */
  MOE_STAGE_FFN_UP = 2,    /* grouped GEMM x_perm -> h (activation fused) */
  MOE_STAGE_FFN_DOWN = 3,  /* grouped GEMM h -> y_perm */
  MOE_STAGE_SHARED = 4,    /* shared expert (only when d_ff_shared > 0) */
  MOE_STAGE_COMBINE = 5,   /* gate scaling + un-permute */
  MOE_STAGE_END = 6,       /* after the last launch */
  MOE_STAGE_FUSED = 7      /* the whole layer in one launch (small-batch SwiGLU layers with
                              d <= 3072: MXFP4 with n <= 16, NVFP4 without a pool with
                              n <= 8): in place of stages 0..5 */
} moe_stage;

/* Host callback run by moe_forward_staged on the calling thread just before
 * the launches of `stage` are enqueued (and once with MOE_STAGE_END after the
 * last one).  kernels_so_far counts the kernels this call has launched.  Work
 * the callback enqueues on the same stream (e.g. a CUDA event record) lands
 * between the stages. */
typedef void (*moe_stage_hook)(int32_t stage, int32_t kernels_so_far, void *user);

/* moe_forward with a stage hook (hook may be NULL: identical to moe_forward). */
moe_status moe_forward_staged(const moe_config *cfg, const void *x, const moe_weights *w, void *y,
                              void *ws, size_t ws_bytes, void *stream, moe_stage_hook hook,
                              void *user);

/* ------------------------------------------------------------------------
 * Expert-slot indirection for the small-batch path.  FreeToken paper summary
 * post on the minseoc03.com feed, section "3. Decode: Exploit Expert
 * Locality" (a selected expert held in GPU memory is a hit and runs from
 * there; one that is not is a miss) and section "10. Dynamic Scheduling
 * Without Giving Up CUDA Graphs" (hit/miss classification and the rewrite of
 * logical expert ids to physical slots happen on the GPU, no host round
 * trip).  A pool of n_slots physical slots holds copies of some experts'
 * MXFP4 weights; slot_of maps each logical expert to its slot or to -1.
 * ------------------------------------------------------------------------ */
typedef struct {
  const int32_t *slot_of;      /* [E] device: slot of expert e in [0, n_slots), or -1 */
  int32_t n_slots;             /* >= 1 */
  const void *W1, *W3, *W2;    /* MXFP4 codes [n_slots][d_ff][d/2], [n_slots][d_ff][d/2]
                                  (W3: SwiGLU only, else NULL), [n_slots][d][d_ff/2] */
  const uint8_t *S1, *S3, *S2; /* E8M0 scales [n_slots][d_ff][d/32], ..., [n_slots][d][d_ff/32] */
} moe_expert_pool;

/* Indices of the counts written by moe_classify_experts / moe_forward_pooled. */
enum {
  MOE_POOL_SELECTED = 0,  /* distinct experts selected by the batch */
  MOE_POOL_RESIDENT = 1,  /* of those, resident (hits) */
  MOE_POOL_LOOKUPS = 2,   /* (token, slot) selections: n * K */
  MOE_POOL_SERVED = 3     /* of those, selections of a resident expert */
};

/* Hit/miss classification of a batch's expert selections (device, async):
 *   topk_idx int32 [n][K] as moe_route writes it; slot_of int32 [E] device.
 *   state int32 [E]: -1 expert not selected, 1 selected and resident (hit),
 *     0 selected and not resident (miss).
 *   miss_list int32 [E]: the missed experts in ascending order, then -1.
 *   counts int32 [4], indexed by MOE_POOL_*.
 * Bit-exact.  A topk_idx value outside [0, E) or a slot_of value outside
 * [-1, n_slots) sets MOE_ERR_BAD_INDEX in the status word (detail: the pair
 * index or the expert; a bad slot counts as a miss). */
moe_status moe_classify_experts(const moe_config *cfg, const int32_t *topk_idx,
                                const int32_t *slot_of, int32_t n_slots, int32_t *state,
                                int32_t *miss_list, int32_t *counts, void *ws, size_t ws_bytes,
                                void *stream);

/* moe_forward for a small batch (MXFP4 experts, bf16 activations, n*K <= 256,
 * no shared expert; else MOE_ERR_UNSUPPORTED) whose expert FFNs read each
 * selected expert from its pool slot when it is resident and from w (which
 * holds all E experts and the router) when it is not.  The result equals
 * moe_forward's bit for bit whatever the resident set, as long as the pool's
 * slots hold byte copies of their experts.  state, miss_list and counts
 * (each nullable) receive the classification of moe_classify_experts.  A
 * slot outside [-1, n_slots) sets MOE_ERR_BAD_INDEX; as after any device-side
 * error, the layer's later kernels then do nothing and y is undefined.
 * Graph-capturable: replays follow the slot table's contents at replay time. */
moe_status moe_forward_pooled(const moe_config *cfg, const void *x, const moe_weights *w,
                              const moe_expert_pool *pool, void *y, int32_t *state,
                              int32_t *miss_list, int32_t *counts, void *ws, size_t ws_bytes,
                              void *stream);

/* moe_forward_pooled with a stage hook (as moe_forward_staged; hook may be NULL). */
moe_status moe_forward_pooled_staged(const moe_config *cfg, const void *x, const moe_weights *w,
                                     const moe_expert_pool *pool, void *y, int32_t *state,
                                     int32_t *miss_list, int32_t *counts, void *ws,
                                     size_t ws_bytes, void *stream, moe_stage_hook hook,
                                     void *user);

/* Synchronises `stream`, then returns the workspace's device status word
 * (MOE_OK if no device-side fault was recorded).  detail, if not NULL,
 * receives the detail word (e.g. the offending pair index). */
moe_status moe_status_check(const void *ws, void *stream, int32_t *detail);

/* Clears the workspace status word (asynchronous on stream). */
moe_status moe_status_clear(void *ws, void *stream);

/* Static string for a status code. */
const char *moe_status_string(moe_status s);

/* Diagnostics for the device-side failure path.  Launches one warp that waits,
 * with the same bounded wait the pipeline kernels use, on a barrier nothing
 * arrives on; after limit_ns (1 .. 1e9) the wait gives up and the kernel sets
 * MOE_ERR_TIMEOUT in the status word and exits, leaving the context usable.
 * ws: a layer workspace (256-byte aligned; read the result with
 * moe_status_check), or NULL for the status word of moe_route_noalloc on the
 * current device (read it with moe_route_noalloc_status).  Asynchronous on
 * stream.  MOE_ERR_INVALID_ARG for a misaligned ws or a bad limit. */
moe_status moe_selftest_wait_timeout(void *ws, uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
