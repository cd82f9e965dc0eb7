"""moe_route_noalloc: the router entry point for callers that cannot allocate
device memory (graph capture under a non-capture-safe allocator, plugins that
only receive their input/output buffers, fixed-arena runtimes).

It is called through the C ABI directly (ctypes, raw device pointers) and must
give the same routing as moe_route with a caller-owned workspace, on two calls
in a row (the static scratch array keeps the previous call's contents).  Its
router never splits the reduction over extra CTAs (moe_route may), so the
logits can differ in the last bits: indices are compared exactly on every
token whose oracle top-k margin is above the near-tie threshold, and the
near-tie tokens are checked as valid choices by parity.check_routing.  This
file is collected last so that a failure here never hides another test."""
import ctypes

import pytest
import torch

import moe_synth
import parity
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    assert torch.cuda.is_available()
    return moe


def _outputs(cfg):
    return (torch.full((cfg.n, cfg.k), -1, dtype=torch.int32, device="cuda"),
            torch.full((cfg.n, cfg.k), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((cfg.n, cfg.E), -1.0, dtype=torch.float32, device="cuda"))


def _noalloc_raw(lib, cfg, inputs, outs):
    c = lib.make_config(cfg)
    w = lib.make_weights(inputs)
    idx, g, pr = outs
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.raw_call("moe_route_noalloc", ctypes.byref(c), inputs["x"].data_ptr(), ctypes.byref(w),
                      idx.data_ptr(), g.data_ptr(), pr.data_ptr(), stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("name,seeds", [
    ("mixtral", (0, 1)),
    ("zipf", (2, 3)),
    ("finegrained", (4, 5)),
])
def test_noalloc_route_matches_workspace_route(lib, name, seeds):
    cfg = {"mixtral": moe_synth.CONFIGS["mixtral_bf16"].scaled(n=1000, d=512, d_ff=256),
           "zipf": moe_synth.CONFIGS["gptoss_prefill_zipf_mxfp4"].scaled(n=700, d=256, d_ff=64),
           "finegrained": moe_synth.CONFIGS["finegrained_shared_bf16"].scaled(
               n=16384, d=256, d_ff=64, d_ff_shared=0)}[name]
    for seed in seeds:                                  # two calls in a row
        inputs = moe_synth.make_inputs(cfg, seed=seed, device="cuda")
        ref = _outputs(cfg)
        ws = lib.alloc_workspace(cfg)
        lib.moe_route(cfg, inputs["x"], lib.make_weights(inputs), *ref, ws)
        assert lib.moe_status_check(ws)[0] == 0
        got = _outputs(cfg)
        assert _noalloc_raw(lib, cfg, inputs, got) == 0
        assert lib.moe_route_noalloc_status() == (0, 0)
        r = O.route(cfg, parity.oracle_inputs(inputs))
        clear = (r["margin"] >= parity.NEAR_TIE).cuda()
        assert torch.equal(got[0][clear], ref[0][clear])
        assert (got[1] - ref[1])[clear].abs().max().item() <= parity.GATE_ATOL
        assert (got[2] - ref[2]).abs().max().item() <= parity.GATE_ATOL
        # and against the oracle, under the same rules as the other routing tests
        parity.check_routing(cfg, r, got[0].cpu(), got[1].cpu())


def test_noalloc_status_reports_a_wait_that_ran_out(lib):
    """A bounded wait that nothing completes, reporting through the no-allocation
    router's status word, is visible through moe_route_noalloc_status; the next
    moe_route_noalloc call clears the word and succeeds."""
    cfg = moe_synth.CONFIGS["mixtral_bf16"].scaled(n=300, d=256, d_ff=64)
    inputs = moe_synth.make_inputs(cfg, seed=7, device="cuda")
    lib.moe_selftest_wait_timeout(None, 20_000_000)         # 20 ms, status word of this device
    st, _ = lib.moe_route_noalloc_status()
    assert st == 6, lib.status_string(st)                  # MOE_ERR_TIMEOUT
    got = _outputs(cfg)
    assert _noalloc_raw(lib, cfg, inputs, got) == 0
    assert lib.moe_route_noalloc_status() == (0, 0)
    r = O.route(cfg, parity.oracle_inputs(inputs))
    parity.check_routing(cfg, r, got[0].cpu(), got[1].cpu())


def test_noalloc_route_rejects_oversize(lib):
    cfg = moe_synth.CONFIGS["finegrained_shared_bf16"].scaled(n=16385, d=64, d_ff=64, d_ff_shared=0)
    c = lib.make_config(cfg)
    w = lib.moe_weights(1 << 20, None, None, None, None, None, None, None, None, None, None)
    st = lib.raw_call("moe_route_noalloc", ctypes.byref(c), 1 << 20, ctypes.byref(w), 1 << 20,
                      1 << 20, None, None)
    assert st == 3, lib.status_string(st)              # MOE_ERR_WORKSPACE, nothing launched
