"""fp64 CPU oracle of the Mixture-of-Experts layer forward pass.

TEST INFRASTRUCTURE ONLY.  This module defines what "correct" means for the
GPU library; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The product path (the C-ABI library and its
Python binding) never calls it, and it shares no code with that path: it reads
the same seeded input tensors (from ``moe_synth``) and nothing else.

Everything is computed in float64 with plain PyTorch CPU ops.  A matrix
product, a stable sort and a cumulative sum from the library serve as single
steps; there is no blocking, fusion or reordering beyond what the method
states.  Sources (page titles and sections):

* [MoE] "How Mixture of Experts Scales Model Parameters"
  - "Dense models: every parameter in the FFN does work for every token":
    the FFN X(n x d) . W1 (d x d_ff) -> activation -> . W2 (d_ff x d).
  - "Sparse models: four experts, and each token uses one": experts are copies
    of the FFN; a token runs through only the chosen ones.
  - "Routing: a router scores the experts, and the top one runs": the router is
    one d x E linear layer followed by a row softmax; top-1 output is the
    chosen expert's output times its probability (0.45 example).
  - "The forward pass: dispatch, then combine": tokens regrouped per expert
    (an expert may receive none), expert FFN per group, rows scaled by their
    routing probability, combine restores token order.
  - "Top-K: several experts, added up by weight": the K highest-scoring
    experts, weights renormalised over the chosen K (0.45/0.76, 0.31/0.76).
* [Lesson] "Inference Optimization: The Bandwidth Wall, PagedAttention, and
  FlashAttention", online-softmax section: softmax with the row maximum
  subtracted (worked example [2, 4, 1, 5], denominator 1.4360).
* [Feed] minseoc03.com feed, post "What is MXFP4?": 4-bit floats in blocks of
  32 values sharing one scale.  The bit-level element (E2M1) and scale (E8M0)
  definitions are those of the OCP Microscaling Formats specification v1.0.
  The same post names NVFP4 (blocks of 16); its scale byte is FP8 E4M3 as the
  OCP 8-bit floating point specification defines it, with one fp32 scale per
  matrix (the reading taken where the post gives only the block size).

Readings where the pages leave a step open:
selection ties go to the lower expert index; the Switch (top-1) gate is the
unrenormalised probability; SwiGLU applies silu to the W1 branch and
multiplies by the linear W3 branch; the router bias (when present) is part of
the router's linear layer, so it moves both selection and gates; MXFP4 blocks
run along the reduction dimension, low nibble first.

Every function here is pinned by ``tests/test_oracle_pins.py`` against page
values, closed forms, library routines or brute force; no function is
"parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import torch

F64 = torch.float64


# ---------------------------------------------------------------------------
# Element decoding
# ---------------------------------------------------------------------------

def to_f64(t: torch.Tensor) -> torch.Tensor:
    """fp32 or bf16 tensor -> exact float64 values.

    bf16 is decoded from its definition: the 16 stored bits are the upper half
    of an IEEE binary32 word whose lower half is zero.
    """
    if t.dtype == torch.float32:
        return t.to(F64)
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).to(torch.int32) << 16
        return bits.view(torch.float32).to(F64)
    raise TypeError(f"unsupported dtype {t.dtype}")


def e2m1_value(code: torch.Tensor) -> torch.Tensor:
    """FP4 E2M1 (OCP MX v1.0): 1 sign, 2 exponent (bias 1), 1 mantissa bit.

    exponent field 0 is subnormal: (-1)^s * 2^0 * (m/2); otherwise
    (-1)^s * 2^(e-1) * (1 + m/2).  No infinities or NaNs.
    """
    c = code.to(torch.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = (c & 1).to(F64)
    sub = m * 0.5
    nrm = torch.pow(2.0, (e - 1).to(F64)) * (1.0 + m * 0.5)
    mag = torch.where(e == 0, sub, nrm)
    return torch.where(s == 1, -mag, mag)


def e8m0_value(s: torch.Tensor) -> torch.Tensor:
    """E8M0 scale (OCP MX v1.0): 2^(s-127); s = 255 encodes NaN."""
    s64 = s.to(torch.int64)
    v = torch.pow(2.0, (s64 - 127).to(F64))
    return torch.where(s64 == 255, torch.full_like(v, math.nan), v)


def mxfp4_decode(packed: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Rows of MXFP4 data -> float64 [..., K].

    packed [..., K/2] uint8 holds element 2j in the low nibble of byte j and
    element 2j+1 in the high nibble; scales [..., K/32] uint8 gives one E8M0
    scale to each block of 32 consecutive elements.
    """
    lo = packed & 0x0F
    hi = packed >> 4
    codes = torch.stack((lo, hi), dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    # the 16 code values from the closed form, then looked up per element
    vals = e2m1_value(torch.arange(16, dtype=torch.uint8))[codes.to(torch.int64)]
    K = vals.shape[-1]
    scale = e8m0_value(scales)
    assert scale.shape[-1] * 32 == K
    return (vals.reshape(*vals.shape[:-1], K // 32, 32) * scale.unsqueeze(-1)).reshape(vals.shape)


def e4m3_value(s: torch.Tensor) -> torch.Tensor:
    """FP8 E4M3 (OCP 8-bit Floating Point Specification, the "FN" variant):
    1 sign, 4 exponent (bias 7), 3 mantissa bits.  Exponent field 0 is
    subnormal: (-1)^s * 2^-6 * (m/8); otherwise (-1)^s * 2^(e-7) * (1 + m/8).
    Exponent 15 with mantissa 7 (0x7F, 0xFF) is NaN; there are no infinities.
    """
    c = s.to(torch.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 15
    m = (c & 7).to(F64)
    sub = torch.pow(2.0, torch.full_like(m, -6.0)) * (m / 8.0)
    nrm = torch.pow(2.0, (e - 7).to(F64)) * (1.0 + m / 8.0)
    mag = torch.where(e == 0, sub, nrm)
    v = torch.where(sign == 1, -mag, mag)
    return torch.where((e == 15) & ((c & 7) == 7), torch.full_like(v, math.nan), v)


def nvfp4_decode(packed: torch.Tensor, scales: torch.Tensor, gscale: float) -> torch.Tensor:
    """Rows of NVFP4 data -> float64 [..., K].

    Feed post "What is MXFP4?": the NVFP4 variant gives each block of 16
    values its own scale.  Elements are E2M1 packed as in ``mxfp4_decode``;
    scales [..., K/16] uint8 hold one FP8 E4M3 scale per block of 16
    consecutive elements, and the whole matrix carries one fp32 scale gscale:
    value = e2m1(code) * e4m3(block scale) * gscale.
    """
    lo = packed & 0x0F
    hi = packed >> 4
    codes = torch.stack((lo, hi), dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = e2m1_value(torch.arange(16, dtype=torch.uint8))[codes.to(torch.int64)]
    K = vals.shape[-1]
    scale = e4m3_value(scales)
    assert scale.shape[-1] * 16 == K
    out = vals.reshape(*vals.shape[:-1], K // 16, 16) * scale.unsqueeze(-1)
    return out.reshape(vals.shape) * float(gscale)


# ---------------------------------------------------------------------------
# Router: linear layer, softmax, top-k, gates   [MoE] "Routing", "Top-K"
# ---------------------------------------------------------------------------

def router_logits(x64: torch.Tensor, Wg64: torch.Tensor,
                  bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """logits[t, e] = sum_i x[t, i] * Wg[e, i] (+ b[e]); Wg stored [E, d]."""
    l = x64 @ Wg64.T
    if bias is not None:
        l = l + bias.to(F64)
    return l


def softmax_rows(logits: torch.Tensor) -> torch.Tensor:
    """Row softmax with the row maximum subtracted first ([Lesson] safe softmax)."""
    m = logits.max(dim=-1, keepdim=True).values
    ex = torch.exp(logits - m)
    return ex / ex.sum(dim=-1, keepdim=True)


def topk_select(logits: torch.Tensor, k: int) -> torch.Tensor:
    """The k highest-scoring experts per row, in rank order.

    Rank order is logit descending; equal logits rank the lower expert index
    first (a stable sort of the negated scores keeps index order among ties).
    Softmax is monotone, so ranking logits ranks probabilities.
    """
    order = torch.sort(-logits, dim=-1, stable=True).indices
    return order[:, :k].contiguous()


def topk_margin(logits: torch.Tensor, k: int) -> torch.Tensor:
    """Smallest gap between consecutive sorted scores among ranks 1..k+1.

    margin[t] = min_{j<k, j+1<E} (l_(j) - l_(j+1)) with l_(0) >= l_(1) >= ...
    the row sorted descending.  Covers ties inside the chosen set (rank order)
    and at the selection boundary.  A row with E == 1 has margin +inf.
    """
    s = torch.sort(logits, dim=-1, descending=True).values
    E = s.shape[-1]
    upto = min(k, E - 1)
    if upto <= 0:
        return torch.full((s.shape[0],), math.inf, dtype=F64)
    gaps = s[:, :upto] - s[:, 1:upto + 1]
    return gaps.min(dim=-1).values


def gate_weights(probs: torch.Tensor, idx: torch.Tensor, mode: str) -> torch.Tensor:
    """Per-slot gate weights.

    "top_prob": the chosen expert's own probability (the Switch example
    multiplies expert 1's output by 0.45).  "renorm": the chosen probabilities
    divided by their sum (0.45/0.76 and 0.31/0.76 in the top-2 example).
    """
    p = probs.gather(1, idx.to(torch.int64))
    if mode == "top_prob":
        return p
    if mode == "renorm":
        return p / p.sum(dim=-1, keepdim=True)
    raise ValueError(mode)


# ---------------------------------------------------------------------------
# Dispatch arrays   [MoE] "The forward pass: dispatch, then combine"
# ---------------------------------------------------------------------------

def dispatch_arrays(idx: torch.Tensor, E: int) -> dict:
    """Per-expert segments of the (token, slot) pairs, by plain definition.

    Pair p = t*k + j routes token t to expert idx[t, j].
    counts[e]  = number of pairs routed to e (may be 0),
    offsets    = exclusive prefix sum of counts, offsets[E] = n*k,
    perm[q]    = the pair at segment position q: pairs sorted by expert,
                 and by pair index (token order) within an expert,
    inv_perm[p] = segment position of pair p (inv_perm[perm[q]] = q).
    """
    flat = idx.reshape(-1).to(torch.int64)
    P = flat.numel()
    counts = torch.bincount(flat, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    perm = torch.sort(flat, stable=True).indices
    inv_perm = torch.empty(P, dtype=torch.int64)
    inv_perm[perm] = torch.arange(P, dtype=torch.int64)
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv_perm)


def combine(y_perm64: torch.Tensor, inv_perm: torch.Tensor, gates64: torch.Tensor,
            y_shared64: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y[t] = sum_j gates[t, j] * y_perm[inv_perm[t*k + j]] (+ y_shared[t])."""
    n, k = gates64.shape
    rows = y_perm64[inv_perm.to(torch.int64)].reshape(n, k, -1)
    y = torch.zeros(n, y_perm64.shape[-1], dtype=F64)
    for j in range(k):
        y += gates64[:, j:j + 1] * rows[:, j, :]
    if y_shared64 is not None:
        y = y + y_shared64
    return y


# ---------------------------------------------------------------------------
# Expert FFN   [MoE] "Dense models"; SwiGLU reading in the module docstring
# ---------------------------------------------------------------------------

def silu(a: torch.Tensor) -> torch.Tensor:
    return a / (1.0 + torch.exp(-a))


def expert_ffn(X: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, act: str,
               W3: Optional[torch.Tensor] = None) -> torch.Tensor:
    """FFN of one expert on rows X [m, d]; weights stored out x in.

    relu:   H = max(X W1^T, 0)
    swiglu: H = silu(X W1^T) * (X W3^T)
    out   = H W2^T                                  -> [m, d]
    """
    A = X @ W1.T
    if act == "relu":
        H = torch.clamp(A, min=0.0)
    elif act == "swiglu":
        H = silu(A) * (X @ W3.T)
    else:
        raise ValueError(act)
    return H @ W2.T


def expert_weights(inputs: dict, cfg, e: int):
    """Expert e's (W1, W3, W2) decoded to float64 (W3 None for ReLU)."""
    if cfg.weight_dtype == "mxfp4":
        W1 = mxfp4_decode(inputs["W1q"][e], inputs["S1"][e])
        W3 = mxfp4_decode(inputs["W3q"][e], inputs["S3"][e]) if cfg.act == "swiglu" else None
        W2 = mxfp4_decode(inputs["W2q"][e], inputs["S2"][e])
    elif cfg.weight_dtype == "nvfp4":
        g = lambda key: float(inputs[key][e])
        W1 = nvfp4_decode(inputs["W1q"][e], inputs["S1"][e], g("G1"))
        W3 = (nvfp4_decode(inputs["W3q"][e], inputs["S3"][e], g("G3"))
              if cfg.act == "swiglu" else None)
        W2 = nvfp4_decode(inputs["W2q"][e], inputs["S2"][e], g("G2"))
    else:
        W1 = to_f64(inputs["W1"][e])
        W3 = to_f64(inputs["W3"][e]) if cfg.act == "swiglu" else None
        W2 = to_f64(inputs["W2"][e])
    return W1, W3, W2


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

def route(cfg, inputs: dict) -> dict:
    """Router linear + softmax + top-k + gates for every token."""
    x64 = to_f64(inputs["x"])
    logits = router_logits(x64, to_f64(inputs["Wg"]), inputs.get("bias"))
    probs = softmax_rows(logits)
    idx = topk_select(logits, cfg.k)
    gates = gate_weights(probs, idx, cfg.gate)
    return dict(logits=logits, probs=probs, topk_idx=idx, topk_gate=gates,
                margin=topk_margin(logits, cfg.k))


def forward(cfg, inputs: dict, tokens: Optional[torch.Tensor] = None,
            routing: Optional[dict] = None) -> dict:
    """y_t = sum_j g_{t,j} FFN_{e_{t,j}}(x_t) (+ shared FFN(x_t)) for the given tokens.

    Follows the pages' order: route every token, group the requested tokens'
    (token, slot) pairs by expert, run each expert's FFN on its group, scale
    each row by its gate and add the slots up in slot order j = 0..k-1.
    ``tokens`` (int64 indices) restricts the expert work to a sample of rows;
    routing is always computed for all rows.
    """
    r = routing if routing is not None else route(cfg, inputs)
    n, k = cfg.n, cfg.k
    if tokens is None:
        tokens = torch.arange(n, dtype=torch.int64)
    tokens = tokens.to(torch.int64)
    x64 = to_f64(inputs["x"][tokens])
    idx = r["topk_idx"][tokens]
    out = torch.zeros(tokens.numel(), k, cfg.d, dtype=F64)
    for e in torch.unique(idx).tolist():
        rows, slots = torch.nonzero(idx == e, as_tuple=True)
        W1, W3, W2 = expert_weights(inputs, cfg, e)
        out[rows, slots] = expert_ffn(x64[rows], W1, W2, cfg.act, W3)
    g = r["topk_gate"][tokens]
    y = torch.zeros(tokens.numel(), cfg.d, dtype=F64)
    for j in range(k):
        y += g[:, j:j + 1] * out[:, j, :]
    y_shared = None
    if cfg.d_ff_shared:
        y_shared = expert_ffn(x64, to_f64(inputs["Ws1"]), to_f64(inputs["Ws2"]), "swiglu",
                              to_f64(inputs["Ws3"]))
        y = y + y_shared
    return dict(y=y, y_shared=y_shared, tokens=tokens, routing=r)


# ---------------------------------------------------------------------------
# Routing statistics   [MoE] "Load balancing: how collapse happens, and how
# it's kept in check"
# ---------------------------------------------------------------------------

def routing_statistics(probs: torch.Tensor, top1: torch.Tensor, alpha: float) -> dict:
    """P_i, f_i and the auxiliary loss of one batch.

    P_i = (1/n) sum over tokens of p_i(x)        (mean router probability)
    f_i = (1/n) #{tokens whose argmax expert is i} (traffic share)
    aux = alpha * E * sum_i f_i * P_i
    ``top1`` is each token's argmax expert (rank 0 of the selection, so ties
    go to the lower index as in ``topk_select``).
    """
    n, E = probs.shape
    P = probs.sum(dim=0) / n
    f = torch.bincount(top1.reshape(-1).to(torch.int64), minlength=E).to(F64) / n
    aux = alpha * E * float((f * P).sum())
    return dict(P=P, f=f, aux=aux)


def near_ties(routing: dict, threshold: float = 1e-5) -> torch.Tensor:
    """Tokens whose top-k margin is below ``threshold`` (listed, not excused)."""
    return torch.nonzero(routing["margin"] < threshold, as_tuple=True)[0]


# ---------------------------------------------------------------------------
# Expert-slot indirection   [Feed] FreeToken paper summary post, section
# "3. Decode: Exploit Expert Locality" (a selected expert that is resident in
# GPU memory is a hit and runs from there; one that is not is a miss) and
# section "10. Dynamic Scheduling Without Giving Up CUDA Graphs" (hit/miss
# classification and the rewrite of logical expert ids to physical cache
# slots happen on the GPU).  The benchmark post's section "5. Why llama.cpp
# Still Hits a Ceiling" counts lookups served by the resident experts.
# ---------------------------------------------------------------------------

def classify_experts(idx: torch.Tensor, E: int, slot_of: torch.Tensor) -> dict:
    """Hit/miss classification of one batch's expert lookups.

    ``idx`` [n, k] holds the selected experts, ``slot_of`` [E] the physical
    slot of each resident expert and -1 for the others.

    * ``state[e]``: -1 if no token selected expert e, 1 if it was selected and
      is resident (hit), 0 if it was selected and is not (miss).
    * ``miss_list``: the missed experts in ascending order.
    * ``selected`` / ``resident``: distinct experts selected / of those, hits.
    * ``lookups`` / ``served``: (token, slot) selections n*k / of those, the
      ones whose expert is resident.
    """
    flat = idx.reshape(-1).to(torch.int64)
    slot_of = slot_of.reshape(-1).to(torch.int64)
    uses = torch.bincount(flat, minlength=E)
    chosen = uses > 0
    hit = slot_of >= 0
    state = torch.full((E,), -1, dtype=torch.int64)
    state[chosen & hit] = 1
    state[chosen & ~hit] = 0
    miss_list = torch.nonzero(chosen & ~hit, as_tuple=True)[0]
    return dict(state=state, miss_list=miss_list,
                selected=int(chosen.sum()), resident=int((chosen & hit).sum()),
                lookups=int(flat.numel()), served=int(uses[hit].sum()))

