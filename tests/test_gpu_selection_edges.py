"""GPU: top-k selection on exact ties and -inf scores, on every selection path.

With the router weights zeroed, every logit is exactly its expert's bias, so
the scores can hold exact ties and -inf entries (a masked expert) that seeded
normal weights never produce.  The selection must then equal the plain
definition exactly: logit descending, the lower expert index first among
equal scores ("How Mixture of Experts Scales Model Parameters", sections
"Routing: a router scores the experts, and the top one runs" and "Top-K:
several experts, added up by weight"; the oracle's stable sort).  A -inf
expert gets probability 0, so renormalised gates divide by the finite
experts' sum alone.

Token counts pick the path: 1 and 8 tokens run the one-launch layer, 24 the
chained small-batch routing cluster, 300 the tensor-core router with its
selection kernel (E > 32) or its fused epilogue selection (E <= 32).
"""
import math

import pytest
import torch

import moe_synth
import parity
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

C = moe_synth.CONFIGS
DEC = C["gptoss_decode_mxfp4"]
PRE = C["mixtral_bf16"]


def _ties_mod5(E):
    return torch.tensor([float((7 * e) % 5) for e in range(E)])


def _masked(E):
    # three finite experts, the rest masked: the top-k runs into the -inf tier
    b = torch.full((E,), -math.inf)
    b[E - 1], b[E // 2], b[5] = 1.5, 1.5, -2.0
    return b


def _tiers(E):
    # experts of a residue class masked, the rest in tiers of 64 (ties within a tier)
    return torch.tensor([-math.inf if e % 3 else float(e // 64) for e in range(E)])


BIASES = {"ties_mod5": _ties_mod5, "masked": _masked, "tiers": _tiers}

CASES = {
    # (config, bias pattern)
    "fused_e128_k4_ties": (DEC.scaled(n=1, d=256, d_ff=256, E=128, k=4), "ties_mod5"),
    "fused_e128_k6_masked": (DEC.scaled(n=8, d=256, d_ff=256, E=128, k=6), "masked"),
    "fused_e200_k5_tiers": (DEC.scaled(n=8, d=256, d_ff=256, E=200, k=5), "tiers"),
    "fused_e256_k8_tiers_top_prob": (DEC.scaled(n=4, d=256, d_ff=256, E=256, k=8,
                                                gate="top_prob"), "tiers"),
    "chain_e128_k4_ties": (DEC.scaled(n=24, d=256, d_ff=256, E=128, k=4), "ties_mod5"),
    "chain_e200_k6_masked": (DEC.scaled(n=24, d=256, d_ff=256, E=200, k=6), "masked"),
    "prefill_e128_k4_ties": (PRE.scaled(n=300, d=256, d_ff=256, E=128, k=4), "ties_mod5"),
    "prefill_e200_k6_masked": (PRE.scaled(n=300, d=256, d_ff=256, E=200, k=6), "masked"),
    "prefill_e32_k2_ties": (PRE.scaled(n=300, d=256, d_ff=256, E=32, k=2), "ties_mod5"),
    "prefill_e32_k3_masked": (PRE.scaled(n=300, d=256, d_ff=256, E=32, k=3), "masked"),
}


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    assert torch.cuda.is_available()
    return moe


@pytest.mark.parametrize("name", list(CASES))
def test_selection_edges(lib, name):
    cfg, pattern = CASES[name]
    inputs = moe_synth.make_inputs(cfg, seed=11, device="cuda")
    inputs["Wg"] = torch.zeros_like(inputs["Wg"])
    inputs["bias"] = BIASES[pattern](cfg.E).to(torch.float32).cuda()
    y, ws, L, inter = parity.run_forward(lib, cfg, inputs)
    r = O.route(cfg, parity.oracle_inputs(inputs))
    # the logits are the bias exactly, on the GPU and in the oracle
    assert torch.equal(inter["logits"].double(), r["logits"])
    assert torch.equal(inter["topk_idx"], r["topk_idx"].to(torch.int32)), (
        inter["topk_idx"][0].tolist(), r["topk_idx"][0].tolist())
    gdiff = (inter["topk_gate"].double() - r["topk_gate"]).abs().max().item()
    assert gdiff <= parity.GATE_ATOL, gdiff
    parity.check_dispatch(cfg, inter["topk_idx"], inter)
    assert torch.isfinite(y.float()).all()
