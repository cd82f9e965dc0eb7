"""GPU: a stack of MoE layers replayed as one CUDA graph, as a decode step of a
model with many MoE layers runs them (the FreeToken benchmark post on the
minseoc03.com feed: gpt-oss-120b has 36 MoE layers, section "5. Why llama.cpp
Still Hits a Ceiling" and the setup section).

Three gpt-oss-shaped decode layers with independently seeded weights run back
to back in one captured graph, each reading the previous layer's bf16 output
(layers after the first scale their router and gate/up matrices to the
previous layer's output rms, as moe_synth.make_stack_inputs describes, in
place of the normalisation a real model applies before each MoE layer).
Each layer is compared with the fp64 oracle applied to the bf16 input that
layer received (the previous layer's output, as the GPU rounded it), under the
same rules as a single layer: routing and dispatch bit-exact (near ties
listed), output rows within 2e-2 of their max-abs.
"""
import pytest
import torch

import moe_synth
from oracle import moe_oracle as O
import parity

pytestmark = pytest.mark.gpu

LAYERS = 3


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    assert torch.cuda.is_available()
    return moe


@pytest.mark.parametrize("n", [4, 64])
def test_decode_stack_in_one_graph(lib, n):
    cfg = moe_synth.CONFIGS["gptoss_decode_mxfp4"].scaled(n=n)
    wss = [lib.alloc_workspace(cfg) for _ in range(LAYERS)]
    ys = [torch.empty(cfg.n, cfg.d, dtype=torch.bfloat16, device="cuda") for _ in range(LAYERS)]
    # each later layer's input-reading matrices scaled to the previous output
    layers = [moe_synth.make_stack_inputs(cfg, 0, seed=0, device="cuda")]
    weights = [lib.make_weights(layers[0])]
    x0 = layers[0]["x"]
    cur = x0
    for l in range(1, LAYERS):
        lib.moe_forward(cfg, cur, weights[l - 1], ys[l - 1], wss[l - 1])
        shift = moe_synth.stack_in_log2(ys[l - 1])
        layers.append(moe_synth.make_stack_inputs(cfg, l, seed=0, device="cuda", in_log2=shift))
        weights.append(lib.make_weights(layers[l]))
        cur = ys[l - 1]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()

    def stack():
        cur = x0
        for l in range(LAYERS):
            lib.moe_forward(cfg, cur, weights[l], ys[l], wss[l], stream=s)
            cur = ys[l]

    with torch.cuda.stream(s):
        stack()                                          # eager run (warm-up)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            stack()
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    L = lib.moe_workspace_layout_of(cfg)
    P = cfg.n * cfg.k
    x_in = x0
    for l in range(LAYERS):
        st, detail = lib.moe_status_check(wss[l])
        assert st == 0, (l, lib.status_string(st), detail)
        oin = parity.oracle_inputs(dict(layers[l], x=x_in))
        r = O.route(cfg, oin)
        idx = parity.ws_view(wss[l], L, "topk_idx", torch.int32, P).view(cfg.n, cfg.k).cpu()
        gate = parity.ws_view(wss[l], L, "topk_gate", torch.float32, P).view(cfg.n, cfg.k).cpu()
        listed = parity.check_routing(cfg, r, idx, gate)
        inter = {k: parity.ws_view(wss[l], L, k, torch.int32, cnt).cpu()
                 for k, cnt in (("counts", cfg.E), ("offsets", cfg.E + 1), ("perm", P),
                                ("inv_perm", P))}
        parity.check_dispatch(cfg, idx, inter)
        ref = O.forward(cfg, oin, routing=parity.routing_with_gpu_ties(cfg, r, idx, listed))
        err = parity.check_output(cfg, ys[l], ref["y"])
        print(f"layer {l}: err={err:.3e} near_ties={listed}")
        x_in = ys[l]
    # the replay equals the eager run of the same stack
    want = [y.clone() for y in ys]
    with torch.cuda.stream(s):
        stack()
    torch.cuda.synchronize()
    for a, b in zip(ys, want):
        assert torch.equal(a, b)
