"""GPU: the small-batch MoE layer as one cooperative launch.

moe_forward runs SwiGLU layers with d <= 3072 as a single launch when they have
MXFP4 experts and at most 16 tokens, or NVFP4 experts and at most 8 tokens (router, selection, dispatch, both expert projections and the
combine; csrc/decode_layer.cu).  These tests pin which layers take that launch
(through the stage hook) and check it against the fp64 oracle at the edges of
its range and in shapes that exercise its scheduling:
- reduction splits that own no MX block;
- one expert holding every token, every token choosing every expert;
- k = 1 with the Zipf router bias, and top-prob gates;
- 256 experts with 256 pairs, most experts holding one;
- NVFP4 weights (E4M3 scales per 16 elements, a scale per matrix) at the same
  edges.
The work units are claimed at run time, so the result must also be the same
bits from run to run, and a workspace reused across calls must give the same
result as a fresh one.  Routing follows the pages: "How Mixture of Experts
Scales Model Parameters", sections "Routing: a router scores the experts, and
the top one runs", "Top-K: several experts, added up by weight" and "The
forward pass: dispatch, then combine".
"""
import pytest
import torch

import moe_synth
import parity

pytestmark = pytest.mark.gpu

C = moe_synth.CONFIGS
D = C["gptoss_decode_mxfp4"]
NV = C["gptoss_decode_nvfp4"]

CHAIN = ["route", "dispatch", "ffn_up", "ffn_down", "combine", "end"]
PATH_CASES = {
    "gptoss_n1": (D.scaled(n=1), True),
    "gptoss_n16": (D.scaled(n=16), True),
    "gptoss_n64": (D.scaled(n=64), False),
    "tokens_16": (D.scaled(n=16, k=2, d=256, d_ff=256, E=16), True),
    "tokens_17": (D.scaled(n=17, k=2, d=256, d_ff=256, E=16), False),
    "d_3072": (D.scaled(n=4, d=3072, d_ff=256, E=16), True),
    "d_3104": (D.scaled(n=4, d=3104, d_ff=256, E=16), False),
    "relu": (D.scaled(n=4, d=256, d_ff=256, E=16, act="relu"), False),
    "nvfp4_n4": (NV.scaled(n=4), True),
    "nvfp4_n8": (NV.scaled(n=8), True),
    "nvfp4_n9": (NV.scaled(n=9), False),
    "nvfp4_relu": (NV.scaled(n=4, d=256, d_ff=256, E=16, act="relu"), False),
}

PARITY_CASES = {
    # the range's edges together: 16 tokens, d = 3072 (12 router pieces a lane)
    "edge_n16_d3072": D.scaled(n=16, k=2, d=3072, d_ff=512, E=32),
    # every token chooses all four experts; rows of 8 and 10 MX blocks leave
    # half of the eight reduction splits without a block
    "every_expert_every_token": D.scaled(n=8, d=256, d_ff=320, E=4, k=4),
    "k1_zipf_bias": D.scaled(n=16, d=512, d_ff=384, E=64, k=1, router_bias="zipf"),
    "top_prob_gates": D.scaled(n=16, d=256, d_ff=256, E=16, k=2, gate="top_prob"),
    # 256 experts, 256 pairs (most experts with one token)
    "e256_k16": D.scaled(n=16, d=128, d_ff=128, E=256, k=16),
    # NVFP4: 8 tokens at d = 3072; odd chunk counts (3 and 5 a row) that
    # leave most reduction splits empty; 128 pairs over 256 experts
    "nvfp4_edge_n8_d3072": NV.scaled(n=8, k=2, d=3072, d_ff=512, E=32),
    "nvfp4_odd_chunks": NV.scaled(n=8, d=96, d_ff=160, E=4, k=4),
    "nvfp4_e256_k16": NV.scaled(n=8, d=128, d_ff=128, E=256, k=16),
}


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    assert torch.cuda.is_available()
    return moe


def _stages(lib, cfg, seed=0):
    inputs = moe_synth.make_inputs(cfg, seed=seed, device="cuda")
    ws = lib.alloc_workspace(cfg)
    y = torch.empty(cfg.n, cfg.d, dtype=torch.bfloat16, device="cuda")
    seen = []
    lib.moe_forward_staged(cfg, inputs["x"], lib.make_weights(inputs), y, ws,
                           lambda st, k: seen.append((lib.STAGES[st], k)))
    st, detail = lib.moe_status_check(ws)
    assert st == 0, (lib.status_string(st), detail)
    return seen


@pytest.mark.parametrize("name", list(PATH_CASES))
def test_path_taken(lib, name):
    cfg, fused = PATH_CASES[name]
    seen = _stages(lib, cfg)
    names = [s for s, _ in seen]
    if fused:
        assert names == ["fused", "end"] and seen[-1][1] == 1
    else:
        assert names == CHAIN and seen[-1][1] == 5


@pytest.mark.parametrize("name", list(PARITY_CASES))
def test_fused_matches_oracle(lib, name):
    cfg = PARITY_CASES[name]
    assert [s for s, _ in _stages(lib, cfg)] == ["fused", "end"]
    res = parity.full_parity(lib, cfg, seed=5)
    assert res["logit_err"] < 5e-6, res["logit_err"]
    print(f"{name}: err={res['err']:.3e} near_ties={res['near_ties']}")


def test_fused_same_bits_every_run(lib):
    """The units go to whichever CTA claims them first; each unit's arithmetic
    is fixed, so two runs give the same bits."""
    cfg = D.scaled(n=16)
    inputs = moe_synth.make_inputs(cfg, seed=3, device="cuda")
    y1, _, _, i1 = parity.run_forward(lib, cfg, inputs)
    y2, _, _, i2 = parity.run_forward(lib, cfg, inputs)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for k in i1:
        assert torch.equal(i1[k], i2[k]), k


def test_fused_workspace_reuse(lib):
    """Back-to-back layers on one workspace (the per-launch counters are
    cleared by each call) equal the same layers on fresh workspaces."""
    cfg = D.scaled(n=4)
    ws = lib.alloc_workspace(cfg)
    for seed in (1, 2, 1):
        inputs = moe_synth.make_inputs(cfg, seed=seed, device="cuda")
        y = torch.empty(cfg.n, cfg.d, dtype=torch.bfloat16, device="cuda")
        lib.moe_forward(cfg, inputs["x"], lib.make_weights(inputs), y, ws)
        assert lib.moe_status_check(ws)[0] == 0
        y_ref, _, _, _ = parity.run_forward(lib, cfg, inputs)
        assert torch.equal(y, y_ref)


@pytest.mark.parametrize("name,cfg", [
    ("n1_staged_router", D.scaled(n=1)),
    ("n2_staged_router", D.scaled(n=2, router_bias="zipf")),
    ("n3_warp_router", D.scaled(n=3)),
    ("n16", D.scaled(n=16, router_bias="zipf")),
    ("nvfp4_n4", NV.scaled(n=4)),
])
def test_fused_logits_equal_route(lib, name, cfg):
    """The one launch's router gives the route-only entry point's logits bit for
    bit (the same per-lane piece order and butterfly sum, whether a CTA stages
    a lone pair's rows in shared memory or a warp loads them itself), and so
    the same selection and gates."""
    inputs = moe_synth.make_inputs(cfg, seed=9, device="cuda")
    w = lib.make_weights(inputs)
    assert [s for s, _ in _stages(lib, cfg, seed=9)] == ["fused", "end"]
    _, ws_f, L, inter = parity.run_forward(lib, cfg, inputs)
    ws_r = lib.alloc_workspace(cfg)
    idx = torch.empty(cfg.n, cfg.k, dtype=torch.int32, device="cuda")
    gate = torch.empty(cfg.n, cfg.k, dtype=torch.float32, device="cuda")
    lib.moe_route(cfg, inputs["x"], w, idx, gate, None, ws_r)
    assert lib.moe_status_check(ws_r)[0] == 0
    logits_r = parity.ws_view(ws_r, L, "logits", torch.float32, cfg.n * cfg.E).view(cfg.n, cfg.E)
    assert torch.equal(inter["logits"].view(torch.int32), logits_r.cpu().view(torch.int32))
    assert torch.equal(inter["topk_idx"], idx.cpu())
    assert torch.equal(inter["topk_gate"].view(torch.int32), gate.cpu().view(torch.int32))
