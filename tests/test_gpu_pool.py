"""GPU: expert-slot indirection for the small-batch path, through the C ABI.

The hit/miss classification is integer work and must equal the oracle's
(``classify_experts``) bit for bit.  The pooled forward reads each resident
expert from its pool slot and the others from the backing arrays; since the
pool holds byte copies, its output must equal ``moe_forward``'s bit for bit
(and so inherits that path's oracle parity), for any resident set.
"""
import pytest
import torch

import moe_synth
from oracle import moe_oracle as O
import parity

pytestmark = pytest.mark.gpu

C = moe_synth.CONFIGS

CASES = {
    "decode_n1": C["gptoss_decode_mxfp4"].scaled(n=1),
    "decode_n16": C["gptoss_decode_mxfp4"].scaled(n=16),
    "decode_many_tokens_per_expert": C["gptoss_decode_mxfp4"].scaled(n=64, d=256, d_ff=320, E=4),
    "decode_relu_small": C["gptoss_decode_mxfp4"].scaled(n=16, d=128, d_ff=192, E=8, k=2,
                                                         act="relu"),
    "decode_odd_blocks": C["gptoss_decode_mxfp4"].scaled(n=4, d=96, d_ff=160, E=8, k=2),
}


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    assert torch.cuda.is_available()
    return moe


def _pool_outputs(cfg):
    return (torch.empty(cfg.E, dtype=torch.int32, device="cuda"),
            torch.empty(cfg.E, dtype=torch.int32, device="cuda"),
            torch.empty(4, dtype=torch.int32, device="cuda"))


def _check_classification(lib, cfg, topk_idx, slot_of, state, miss, counts):
    want = O.classify_experts(topk_idx.cpu(), cfg.E, slot_of.cpu())
    assert torch.equal(state.cpu().to(torch.int64), want["state"])
    m = want["miss_list"].numel()
    assert miss[:m].cpu().tolist() == want["miss_list"].tolist()
    assert (miss[m:].cpu() == -1).all()
    got = counts.cpu().tolist()
    assert got[lib.POOL_SELECTED] == want["selected"]
    assert got[lib.POOL_RESIDENT] == want["resident"]
    assert got[lib.POOL_LOOKUPS] == want["lookups"]
    assert got[lib.POOL_SERVED] == want["served"]


@pytest.mark.parametrize("name", ["decode_n16", "decode_relu_small"])
@pytest.mark.parametrize("resident_frac", [0.0, 0.3, 1.0])
def test_classify_matches_oracle(lib, name, resident_frac):
    cfg = CASES[name]
    inputs = moe_synth.make_inputs(cfg, seed=4, device="cuda")
    ws = lib.alloc_workspace(cfg)
    idx = torch.empty(cfg.n, cfg.k, dtype=torch.int32, device="cuda")
    gate = torch.empty(cfg.n, cfg.k, dtype=torch.float32, device="cuda")
    lib.moe_route(cfg, inputs["x"], lib.make_weights(inputs), idx, gate, None, ws)
    n_slots = max(1, cfg.E // 2)
    resident = min(n_slots, round(resident_frac * cfg.E))
    slot_of = moe_synth.make_slot_table(cfg.E, n_slots, resident, seed=11).cuda()
    state, miss, counts = _pool_outputs(cfg)
    lib.moe_classify_experts(cfg, idx, slot_of, n_slots, state, miss, counts, ws)
    assert lib.moe_status_check(ws)[0] == 0
    _check_classification(lib, cfg, idx, slot_of, state, miss, counts)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("resident_frac", [0.0, 0.5, 1.0])
def test_forward_pooled_equals_forward(lib, name, resident_frac):
    cfg = CASES[name]
    inputs = moe_synth.make_inputs(cfg, seed=6, device="cuda")
    y_ref, ws, L, inter = parity.run_forward(lib, cfg, inputs)
    n_slots = max(1, (cfg.E * 3) // 4)
    resident = min(n_slots, round(resident_frac * cfg.E))
    slot_of = moe_synth.make_slot_table(cfg.E, n_slots, resident, seed=12)
    pool = moe_synth.make_pool(inputs, slot_of, n_slots, device="cuda")
    slot_dev = slot_of.cuda()
    y = torch.empty_like(y_ref)
    state, miss, counts = _pool_outputs(cfg)
    ws2 = lib.alloc_workspace(cfg)
    lib.moe_forward_pooled(cfg, inputs["x"], lib.make_weights(inputs),
                           lib.make_pool(slot_dev, pool), y, state, miss, counts, ws2)
    st, detail = lib.moe_status_check(ws2)
    assert st == 0, (lib.status_string(st), detail)
    assert torch.equal(y, y_ref), (y.float() - y_ref.float()).abs().max().item()
    _check_classification(lib, cfg, inter["topk_idx"], slot_of, state, miss, counts)


def test_bad_slot_is_reported(lib):
    """A slot outside the pool sets MOE_ERR_BAD_INDEX (sticky: the layer's
    later kernels then do nothing); the classification counts it as a miss."""
    cfg = CASES["decode_relu_small"]
    inputs = moe_synth.make_inputs(cfg, seed=6, device="cuda")
    _, _, _, inter = parity.run_forward(lib, cfg, inputs)
    n_slots = 4
    slot_of = moe_synth.make_slot_table(cfg.E, n_slots, 2, seed=3)
    chosen = sorted(set(inter["topk_idx"].reshape(-1).tolist()))
    bad = next(e for e in chosen if int(slot_of[e]) < 0)
    slot_of[bad] = n_slots + 5                       # outside the pool
    valid = torch.where(slot_of < n_slots, slot_of, torch.full_like(slot_of, -1))
    pool = moe_synth.make_pool(inputs, valid, n_slots, device="cuda")
    y = torch.empty(cfg.n, cfg.d, dtype=torch.bfloat16, device="cuda")
    state, miss, counts = _pool_outputs(cfg)
    ws = lib.alloc_workspace(cfg)
    lib.moe_forward_pooled(cfg, inputs["x"], lib.make_weights(inputs),
                           lib.make_pool(slot_of.cuda(), pool), y, state, miss, counts, ws)
    st, detail = lib.moe_status_check(ws)
    assert (st, detail) == (5, bad)                  # MOE_ERR_BAD_INDEX, the expert
    _check_classification(lib, cfg, inter["topk_idx"], valid, state, miss, counts)


def test_forward_pooled_in_cuda_graph(lib):
    """The pooled forward captures into a CUDA graph; replays after the slot
    table changes on the device follow the new table (no host round trip)."""
    cfg = CASES["decode_odd_blocks"]
    inputs = moe_synth.make_inputs(cfg, seed=2, device="cuda")
    y_ref, _, _, _ = parity.run_forward(lib, cfg, inputs)
    n_slots = cfg.E
    full = torch.arange(cfg.E, dtype=torch.int32)
    pool = moe_synth.make_pool(inputs, full, n_slots, device="cuda")
    slot_dev = torch.full((cfg.E,), -1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(y_ref)
    state, miss, counts = _pool_outputs(cfg)
    ws = lib.alloc_workspace(cfg)
    w, p = lib.make_weights(inputs), lib.make_pool(slot_dev, pool)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lib.moe_forward_pooled(cfg, inputs["x"], w, p, y, state, miss, counts, ws, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            lib.moe_forward_pooled(cfg, inputs["x"], w, p, y, state, miss, counts, ws, stream=s)
    for table in (torch.full((cfg.E,), -1, dtype=torch.int32), full):
        slot_dev.copy_(table)
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        want_served = 0 if table[0] < 0 else cfg.n * cfg.k
        assert counts[lib.POOL_SERVED].item() == want_served


def test_forward_pooled_staged_hook(lib):
    """The staged variant runs the same launch, calling the hook before it (this
    MXFP4 SwiGLU layer runs as one fused launch) and after it."""
    cfg = CASES["decode_n16"]
    inputs = moe_synth.make_inputs(cfg, seed=8, device="cuda")
    y_ref, _, _, _ = parity.run_forward(lib, cfg, inputs)
    table = moe_synth.make_slot_table(cfg.E, 40, 40, seed=1)
    pool = moe_synth.make_pool(inputs, table, 40, device="cuda")
    table_dev = table.cuda()
    y = torch.empty_like(y_ref)
    seen = []
    ws = lib.alloc_workspace(cfg)
    lib.moe_forward_pooled_staged(cfg, inputs["x"], lib.make_weights(inputs),
                                  lib.make_pool(table_dev, pool), y, None, None, None, ws,
                                  lambda st, k: seen.append((st, k)))
    assert lib.moe_status_check(ws)[0] == 0
    assert torch.equal(y, y_ref)
    names = [lib.STAGES[st] for st, _ in seen]
    assert names == ["fused", "end"]
    assert seen[-1][1] == 1                          # kernels launched


@pytest.mark.parametrize("name", ["decode_n16", "decode_odd_blocks"])
def test_forward_pooled_matches_oracle(lib, name):
    """moe_forward_pooled against the fp64 oracle directly (every token), with
    half of the experts resident, on a seed of its own."""
    cfg = CASES[name]
    inputs = moe_synth.make_inputs(cfg, seed=9, device="cuda")
    n_slots = max(1, cfg.E // 2)
    slot_of = moe_synth.make_slot_table(cfg.E, n_slots, n_slots, seed=13)
    pool = moe_synth.make_pool(inputs, slot_of, n_slots, device="cuda")
    slot_dev = slot_of.cuda()
    y = torch.empty(cfg.n, cfg.d, dtype=torch.bfloat16, device="cuda")
    state, miss, counts = _pool_outputs(cfg)
    ws = lib.alloc_workspace(cfg)
    lib.moe_forward_pooled(cfg, inputs["x"], lib.make_weights(inputs),
                           lib.make_pool(slot_dev, pool), y, state, miss, counts, ws)
    st, detail = lib.moe_status_check(ws)
    assert st == 0, (lib.status_string(st), detail)
    L = lib.moe_workspace_layout_of(cfg)
    idx = parity.ws_view(ws, L, "topk_idx", torch.int32, cfg.n * cfg.k).view(cfg.n, cfg.k).cpu()
    gate = parity.ws_view(ws, L, "topk_gate", torch.float32, cfg.n * cfg.k).view(cfg.n, cfg.k).cpu()
    oin = parity.oracle_inputs(inputs)
    r = O.route(cfg, oin)
    listed = parity.check_routing(cfg, r, idx, gate)
    ref = O.forward(cfg, oin, routing=parity.routing_with_gpu_ties(cfg, r, idx, listed))
    parity.check_output(cfg, y, ref["y"])
    _check_classification(lib, cfg, idx, slot_of, state, miss, counts)
