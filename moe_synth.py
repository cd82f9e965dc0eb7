"""Seeded synthetic inputs for the MoE layer forward pass.

This module is the only code shared by the fp64 oracle (``oracle/``) and the
CUDA path (``mixture_experts_layer_moe_gb300``).  It draws random tensors and
lays them out in memory; it computes none of the layer's arithmetic (no
router, softmax, selection, dispatch, FFN, dequantisation or combine).

Workloads (shapes from the MoE layer as "How Mixture of Experts Scales Model
Parameters" states it: X is n x d, the router is one d x E linear layer, each
expert is a copy of the FFN d -> d_ff -> d):

* ``tiny_switch_fp32``       Switch-style top-1, ReLU, fp32, n=256 d=128 F=512 E=4
* ``mixtral_bf16``           top-2 renormalised, SwiGLU, bf16, n=4096 d=4096 F=14336 E=8
* ``gptoss_decode_mxfp4``    top-4, SwiGLU, MXFP4 experts, n in {1,4,16,64}, d=F=2880, E=128
* ``gptoss_prefill_zipf_mxfp4``  as above, n=8192, router bias giving Zipf(1.2) loads
* ``gptoss_decode_nvfp4``    the decode workload with NVFP4 experts (blocks of 16)
* ``finegrained_shared_bf16``    top-8 of 256, SwiGLU F=2048, d=7168, one shared expert, n=16384

Storage conventions (all row-major, weights stored out x in so the reduction
dimension is contiguous):

* ``x``   [n, d]             fp32 or bf16
* ``Wg``  [E, d]             same dtype as x (the router's d x E matrix, transposed)
* ``bias``[E]                fp32 or None (added to the router logits)
* bf16 / fp32 experts: ``W1``, ``W3`` [E, F, d]; ``W2`` [E, d, F] (``W3`` None for ReLU)
* MXFP4 experts: ``W1q``/``W3q`` [E, F, d/2] uint8, element i of a row in byte i//2,
  low nibble when i is even; ``S1``/``S3`` [E, F, d/32] uint8 E8M0 block scales
  (one per 32 consecutive elements along d); ``W2q`` [E, d, F/2], ``S2`` [E, d, F/32].
* NVFP4 experts: codes as MXFP4; ``S1``/``S3`` [E, F, d/16], ``S2`` [E, d, F/16] uint8
  FP8 E4M3 block scales (one per 16 consecutive elements); ``G1``/``G3``/``G2`` [E] fp32,
  one scale per expert matrix.
* shared expert (bf16): ``Ws1``, ``Ws3`` [Fs, d]; ``Ws2`` [d, Fs].

Draw order for a seed: x, Wg, [expert ordering for the bias], then per expert
W1, W3, W2 (codes then scales for MXFP4), then the shared expert.  Normals are
drawn in fp32 and cast with round-to-nearest-even to the config's dtype.  The
generator is ``torch.Generator`` on the device the tensors are made on, so a
seed gives the same bytes every time on the same device type (the CPU and CUDA
streams differ from each other).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    n: int
    d: int
    d_ff: int
    E: int
    k: int
    act_dtype: str          # "f32" | "bf16"
    weight_dtype: str       # "f32" | "bf16" | "mxfp4" | "nvfp4"
    gate: str               # "top_prob" (Switch: g = p of the chosen expert) | "renorm"
    act: str                # "relu" | "swiglu"
    router_bias: str = "none"   # "none" | "zipf"
    zipf_s: float = 1.2
    d_ff_shared: int = 0        # 0: no shared expert
    x_std: float = 1.0
    w_std: float = 0.02

    def scaled(self, **kw) -> "MoEConfig":
        """Same workload structure at other sizes (for parity tests)."""
        return dataclasses.replace(self, **kw)

    @property
    def P(self) -> int:
        return self.n * self.k


CONFIGS = {
    "tiny_switch_fp32": MoEConfig(
        "tiny_switch_fp32", n=256, d=128, d_ff=512, E=4, k=1,
        act_dtype="f32", weight_dtype="f32", gate="top_prob", act="relu"),
    "mixtral_bf16": MoEConfig(
        "mixtral_bf16", n=4096, d=4096, d_ff=14336, E=8, k=2,
        act_dtype="bf16", weight_dtype="bf16", gate="renorm", act="swiglu"),
    "gptoss_decode_mxfp4": MoEConfig(
        "gptoss_decode_mxfp4", n=1, d=2880, d_ff=2880, E=128, k=4,
        act_dtype="bf16", weight_dtype="mxfp4", gate="renorm", act="swiglu"),
    "gptoss_prefill_zipf_mxfp4": MoEConfig(
        "gptoss_prefill_zipf_mxfp4", n=8192, d=2880, d_ff=2880, E=128, k=4,
        act_dtype="bf16", weight_dtype="mxfp4", gate="renorm", act="swiglu",
        router_bias="zipf"),
    "gptoss_decode_nvfp4": MoEConfig(
        "gptoss_decode_nvfp4", n=1, d=2880, d_ff=2880, E=128, k=4,
        act_dtype="bf16", weight_dtype="nvfp4", gate="renorm", act="swiglu"),
    "finegrained_shared_bf16": MoEConfig(
        "finegrained_shared_bf16", n=16384, d=7168, d_ff=2048, E=256, k=8,
        act_dtype="bf16", weight_dtype="bf16", gate="renorm", act="swiglu",
        d_ff_shared=2048),
}

DECODE_BATCHES = (1, 4, 16, 64)

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _normal(shape, std, dtype, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """Pack 4-bit codes along the last dim: byte j = codes[2j] | codes[2j+1] << 4."""
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).contiguous()


def _mxfp4_matrix(rows, cols, g, device):
    """Uniform E2M1 codes (all 16) and E8M0 scales uniform over 2^-8 .. 2^-4."""
    codes = torch.randint(0, 16, (rows, cols), generator=g, device=device, dtype=torch.uint8)
    scales = torch.randint(119, 124, (rows, cols // 32), generator=g, device=device,
                           dtype=torch.uint8)
    return _pack_nibbles(codes), scales


def _nvfp4_matrix(rows, cols, g, device):
    """Uniform E2M1 codes (all 16); E4M3 block scales with exponent field
    uniform over 4..10 (2^-3 .. 2^3) and uniform mantissa; one fp32 matrix
    scale uniform over [2^-8, 2^-7)."""
    codes = torch.randint(0, 16, (rows, cols), generator=g, device=device, dtype=torch.uint8)
    ex = torch.randint(4, 11, (rows, cols // 16), generator=g, device=device, dtype=torch.uint8)
    man = torch.randint(0, 8, (rows, cols // 16), generator=g, device=device, dtype=torch.uint8)
    gs = (1.0 + torch.rand((), generator=g, device=device, dtype=torch.float32)) / 256.0
    return _pack_nibbles(codes), (ex << 3) | man, gs


def zipf_router_bias(cfg: MoEConfig, order: torch.Tensor) -> torch.Tensor:
    """Router bias b_e = ln q_{rank(e)} with q_r proportional to r^-s.

    ``order`` is a seeded permutation; expert ``order[r-1]`` gets rank r.  This
    only shapes the synthetic router so that expected loads are Zipf-skewed.
    """
    E = cfg.E
    r = torch.arange(1, E + 1, dtype=torch.float64)
    q = r.pow(-cfg.zipf_s)
    q = q / q.sum()
    b = torch.empty(E, dtype=torch.float64)
    b[order.cpu().long()] = q.log()
    return b.to(torch.float32)


def make_inputs(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """All tensors of one MoE layer call for ``cfg`` (see module docstring)."""
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    adt = _TORCH_DTYPE[cfg.act_dtype]
    n, d, F, E = cfg.n, cfg.d, cfg.d_ff, cfg.E
    out: dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal((n, d), cfg.x_std, adt, g, device)
    out["Wg"] = _normal((E, d), cfg.w_std, adt, g, device)
    if cfg.router_bias == "zipf":
        order = torch.randperm(E, generator=g, device=device)
        out["bias"] = zipf_router_bias(cfg, order).to(device)
    else:
        out["bias"] = None

    swiglu = cfg.act == "swiglu"
    if cfg.weight_dtype == "mxfp4":
        assert d % 32 == 0 and F % 32 == 0
        W1q = torch.empty((E, F, d // 2), dtype=torch.uint8, device=device)
        S1 = torch.empty((E, F, d // 32), dtype=torch.uint8, device=device)
        W3q = torch.empty_like(W1q) if swiglu else None
        S3 = torch.empty_like(S1) if swiglu else None
        W2q = torch.empty((E, d, F // 2), dtype=torch.uint8, device=device)
        S2 = torch.empty((E, d, F // 32), dtype=torch.uint8, device=device)
        for e in range(E):
            W1q[e], S1[e] = _mxfp4_matrix(F, d, g, device)
            if swiglu:
                W3q[e], S3[e] = _mxfp4_matrix(F, d, g, device)
            W2q[e], S2[e] = _mxfp4_matrix(d, F, g, device)
        out.update(W1q=W1q, S1=S1, W3q=W3q, S3=S3, W2q=W2q, S2=S2,
                   W1=None, W3=None, W2=None)
    elif cfg.weight_dtype == "nvfp4":
        assert d % 32 == 0 and F % 32 == 0
        W1q = torch.empty((E, F, d // 2), dtype=torch.uint8, device=device)
        S1 = torch.empty((E, F, d // 16), dtype=torch.uint8, device=device)
        W3q = torch.empty_like(W1q) if swiglu else None
        S3 = torch.empty_like(S1) if swiglu else None
        W2q = torch.empty((E, d, F // 2), dtype=torch.uint8, device=device)
        S2 = torch.empty((E, d, F // 16), dtype=torch.uint8, device=device)
        G1 = torch.empty(E, dtype=torch.float32, device=device)
        G3 = torch.empty(E, dtype=torch.float32, device=device) if swiglu else None
        G2 = torch.empty(E, dtype=torch.float32, device=device)
        for e in range(E):
            W1q[e], S1[e], G1[e] = _nvfp4_matrix(F, d, g, device)
            if swiglu:
                W3q[e], S3[e], G3[e] = _nvfp4_matrix(F, d, g, device)
            W2q[e], S2[e], G2[e] = _nvfp4_matrix(d, F, g, device)
        out.update(W1q=W1q, S1=S1, W3q=W3q, S3=S3, W2q=W2q, S2=S2, G1=G1, G3=G3, G2=G2,
                   W1=None, W3=None, W2=None)
    else:
        wdt = _TORCH_DTYPE[cfg.weight_dtype]
        W1 = torch.empty((E, F, d), dtype=wdt, device=device)
        W3 = torch.empty((E, F, d), dtype=wdt, device=device) if swiglu else None
        W2 = torch.empty((E, d, F), dtype=wdt, device=device)
        for e in range(E):
            W1[e] = _normal((F, d), cfg.w_std, wdt, g, device)
            if swiglu:
                W3[e] = _normal((F, d), cfg.w_std, wdt, g, device)
            W2[e] = _normal((d, F), cfg.w_std, wdt, g, device)
        out.update(W1=W1, W3=W3, W2=W2, W1q=None, S1=None, W3q=None, S3=None,
                   W2q=None, S2=None)

    if cfg.d_ff_shared:
        Fs = cfg.d_ff_shared
        out["Ws1"] = _normal((Fs, d), cfg.w_std, adt, g, device)
        out["Ws3"] = _normal((Fs, d), cfg.w_std, adt, g, device)
        out["Ws2"] = _normal((d, Fs), cfg.w_std, adt, g, device)
    else:
        out["Ws1"] = out["Ws3"] = out["Ws2"] = None
    return out


def make_stack_inputs(cfg: MoEConfig, layer: int, seed: int = 0, device="cpu",
                      in_log2: int = 0) -> dict:
    """Inputs of layer `layer` of a stack of MoE layers: layer 0 is
    make_inputs(seed); layer l > 0 draws its own weights from seed + 101 l.

    A stack feeds each layer's output to the next, and SwiGLU experts are
    quadratic in their input, so without a normalisation between the layers
    the activations leave every finite range within a few layers (the
    synthetic gpt-oss layer turns rms 1 into rms ~38).  A real model
    normalises each MoE layer's input; here the matrices that read the input
    (the router Wg and the experts' W1 and W3) are scaled by 2^-in_log2
    instead, in_log2 being the log2 of the previous layer's output rms
    (rounded), so every layer sees its input at the scale of the first
    layer's.  The scale is an exact power of two: Wg times 2^-in_log2, MXFP4
    E8M0 bytes of W1 and W3 lowered by in_log2, NVFP4 matrix scales G1 and G3
    times 2^-in_log2; bf16 and fp32 experts scale W1 and W3 themselves."""
    if layer == 0:
        return make_inputs(cfg, seed=seed, device=device)
    out = make_inputs(cfg, seed=seed + 101 * layer, device=device)
    k = int(in_log2)
    if k == 0:
        return out
    out["Wg"] = (out["Wg"].float() * 2.0 ** -k).to(out["Wg"].dtype)
    if cfg.weight_dtype == "mxfp4":
        for key in ("S1", "S3"):
            if out.get(key) is not None:
                out[key] = (out[key].to(torch.int32) - k).clamp(0, 254).to(torch.uint8)
    elif cfg.weight_dtype == "nvfp4":
        for key in ("G1", "G3"):
            if out.get(key) is not None:
                out[key] = out[key] * 2.0 ** -k
    else:
        for key in ("W1", "W3"):
            if out.get(key) is not None:
                out[key] = (out[key].float() * 2.0 ** -k).to(out[key].dtype)
    return out


def stack_in_log2(y: torch.Tensor) -> int:
    """The input scale exponent for the layer after one whose output is y: the
    log2 of y's rms, rounded to an integer."""
    import math
    rms = float(y.float().pow(2).mean().sqrt())
    return int(round(math.log2(rms))) if rms > 0 else 0


def to_cpu(inputs: dict) -> dict:
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}


def weight_bytes_per_expert(cfg: MoEConfig) -> int:
    """Bytes of one routed expert's weights as stored (codes + scales for MXFP4)."""
    mats = 3 if cfg.act == "swiglu" else 2
    elems = cfg.d * cfg.d_ff
    if cfg.weight_dtype == "mxfp4":
        return mats * (elems // 2 + elems // 32)
    if cfg.weight_dtype == "nvfp4":
        return mats * (elems // 2 + elems // 16 + 4)
    return mats * elems * (4 if cfg.weight_dtype == "f32" else 2)


def expert_flops_per_pair(cfg: MoEConfig) -> int:
    """FLOPs of one (token, expert) FFN evaluation: 2*d*F per projection."""
    mats = 3 if cfg.act == "swiglu" else 2
    return 2 * mats * cfg.d * cfg.d_ff


def describe(cfg: MoEConfig) -> str:
    return (f"{cfg.name}: n={cfg.n} d={cfg.d} d_ff={cfg.d_ff} E={cfg.E} k={cfg.k} "
            f"{cfg.act_dtype}/{cfg.weight_dtype} {cfg.act} gate={cfg.gate}"
            + (f" shared d_ff={cfg.d_ff_shared}" if cfg.d_ff_shared else "")
            + (f" bias={cfg.router_bias}" if cfg.router_bias != "none" else ""))



# ---------------------------------------------------------------------------
# Resident expert pool (expert-slot indirection inputs)
# ---------------------------------------------------------------------------

def make_slot_table(E: int, n_slots: int, resident: int, seed: int = 0) -> torch.Tensor:
    """A seeded resident set: ``resident`` distinct experts, each mapped to a
    distinct slot in [0, n_slots) (both drawn at random); -1 elsewhere."""
    assert 0 <= resident <= min(E, n_slots)
    g = torch.Generator().manual_seed(seed)
    experts = torch.randperm(E, generator=g)[:resident]
    slots = torch.randperm(n_slots, generator=g)[:resident]
    table = torch.full((E,), -1, dtype=torch.int32)
    table[experts] = slots.to(torch.int32)
    return table


def make_pool(inputs: dict, slot_of: torch.Tensor, n_slots: int, device="cpu") -> dict:
    """The resident pool for ``slot_of``: slot s holds a byte-for-byte copy of
    the weights (MXFP4 codes and scales) of the expert mapped to it; unused
    slots are zero.  Keys as in ``make_inputs``."""
    out = {}
    for key in ("W1q", "W3q", "W2q", "S1", "S3", "S2"):
        src = inputs.get(key)
        if src is None:
            continue
        pool = torch.zeros((n_slots,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
        for e, s in enumerate(slot_of.tolist()):
            if s >= 0:
                pool[s].copy_(src[e])
        out[key] = pool.to(device)
    return out
