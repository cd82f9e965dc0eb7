"""The C-ABI library loads, exports every symbol include/moe.h declares, and its
host-side argument checks and workspace layout behave as documented.  None of
these tests makes a CUDA call (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_moe_gb300 import build
    build.build()
    from mixture_experts_layer_moe_gb300 import moe
    return moe


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_workspace_size", "moe_status_check", "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from mixture_experts_layer_moe_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib.library(), n)


def _c(lib, **kw):
    base = dict(name="t", n=16, d=64, d_ff=128, E=8, k=2, act_dtype="bf16", weight_dtype="bf16",
                gate="renorm", act="swiglu")
    base.update(kw)
    return lib.make_config(moe_synth.MoEConfig(**base))


def _size(lib, c):
    out = ctypes.c_size_t(0)
    st = lib.raw_call("moe_workspace_size", ctypes.byref(c), ctypes.byref(out))
    return st, out.value


@pytest.mark.parametrize("kw,want", [
    (dict(n=0), 1), (dict(E=0), 1), (dict(E=257), 1), (dict(k=0), 1), (dict(k=9), 1),
    (dict(d=0), 1), (dict(d=60), 2), (dict(d_ff=100), 2),
    (dict(weight_dtype="mxfp4", d=80), 2), (dict(weight_dtype="f32"), 2),
    (dict(act_dtype="f32", weight_dtype="bf16"), 2), (dict(act_dtype="f32", weight_dtype="f32", d=4), 0),
    (dict(weight_dtype="mxfp4", d=64, d_ff=96), 0), (dict(E=256, k=256), 0), (dict(n=1, E=1, k=1), 0),
    (dict(weight_dtype="nvfp4", n=64, k=4), 0), (dict(weight_dtype="nvfp4", n=65, k=4), 2),
    (dict(weight_dtype="nvfp4", d=80), 2), (dict(act_dtype="f32", weight_dtype="nvfp4"), 2),
])
def test_config_checks(lib, kw, want):
    st, _ = _size(lib, _c(lib, **kw))
    assert st == want, lib.status_string(st)


def test_workspace_layout(lib):
    for name, cfg in moe_synth.CONFIGS.items():
        L = lib.moe_workspace_layout_of(cfg)
        assert L["total"] == lib.moe_workspace_size(cfg)
        P = cfg.n * cfg.k
        a = 2 if cfg.act_dtype == "bf16" else 4
        sizes = dict(status=8, logits=cfg.n * cfg.E * 4, topk_idx=P * 4, topk_gate=P * 4,
                     counts=cfg.E * 4, offsets=(cfg.E + 1) * 4, perm=P * 4, inv_perm=P * 4,
                     x_perm=P * cfg.d * a, h=P * cfg.d_ff * a, y_perm=P * cfg.d * a)
        if cfg.d_ff_shared:
            sizes.update(y_shared=cfg.n * cfg.d * a, h_shared=cfg.n * cfg.d_ff_shared * a)
        spans = sorted((L[k], L[k] + v) for k, v in sizes.items())
        for (s0, e0), (s1, _) in zip(spans, spans[1:]):
            assert e0 <= s1
        assert spans[-1][1] <= L["total"]
        assert all(L[k] % 256 == 0 for k in sizes)


FAKE = 1 << 20          # a 256-aligned non-null address; never dereferenced on the host


def test_forward_argument_checks_without_launch(lib):
    c = _c(lib)
    st, ws_bytes = _size(lib, c)
    w = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, None, None, None, None, None, None)
    call = lambda x, y, ws, n, w=w: lib.raw_call("moe_forward", ctypes.byref(c), x, ctypes.byref(w),
                                                  y, ws, n, None)
    assert call(None, FAKE, FAKE, ws_bytes) == 1                 # null x
    assert call(FAKE + 8, FAKE, FAKE, ws_bytes) == 1             # x not 16-byte aligned
    assert call(FAKE, FAKE, FAKE + 16, ws_bytes) == 1            # ws not 256-byte aligned
    assert call(FAKE, FAKE, FAKE, ws_bytes - 1) == 3             # workspace too small
    w_relu = lib.moe_weights(FAKE, None, FAKE, None, FAKE, None, None, None, None, None, None)
    assert call(FAKE, FAKE, FAKE, ws_bytes, w_relu) == 1         # SwiGLU without W3
    w_sc = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None)
    assert call(FAKE, FAKE, FAKE, ws_bytes, w_sc) == 1           # scales with bf16 weights
    w_sh = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, FAKE)
    assert call(FAKE, FAKE, FAKE, ws_bytes, w_sh) == 1           # shared weights, no shared expert


def test_entry_point_argument_checks(lib):
    c = _c(lib)
    _, n = _size(lib, c)
    w = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, None, None, None, None, None, None)
    cp, wp = ctypes.byref(c), ctypes.byref(w)
    assert lib.raw_call("moe_route", cp, FAKE, wp, None, FAKE, None, FAKE, n, None) == 1
    assert lib.raw_call("moe_route", cp, FAKE, wp, FAKE, FAKE, FAKE + 4, FAKE, n, None) == 1
    assert lib.raw_call("moe_dispatch", cp, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, n,
                        None) == 1                                 # x_perm wanted but no x
    assert lib.raw_call("moe_dispatch", cp, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 100,
                        None) == 3
    assert lib.raw_call("moe_expert_ffn", cp, FAKE, None, wp, FAKE, FAKE, n, None) == 1
    assert lib.raw_call("moe_combine", cp, FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, n, None) == 1
    assert lib.raw_call("moe_combine", None, FAKE, FAKE, FAKE, None, FAKE, FAKE, n, None) == 1
    assert lib.raw_call("moe_status_check", None, None, None) == 1
    assert lib.raw_call("moe_status_clear", FAKE + 1, None) == 1


def test_status_strings(lib):
    for code in range(7):
        s = lib.status_string(code)
        assert s.startswith("MOE_")
    assert "unknown" in lib.status_string(42)


def test_pool_entry_point_argument_checks(lib):
    """moe_forward_pooled / moe_classify_experts reject bad arguments before any launch."""
    c = _c(lib, n=4, weight_dtype="mxfp4")
    _, n = _size(lib, c)
    w = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None)
    pool = lib.moe_expert_pool(FAKE, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    fwd = lambda cfg, p, ws=FAKE, nb=n: lib.raw_call(
        "moe_forward_pooled", ctypes.byref(cfg), FAKE, ctypes.byref(w),
        None if p is None else ctypes.byref(p), FAKE, None, None, None, ws, nb, None)
    assert fwd(c, None) == 1                                       # no pool
    assert fwd(c, lib.moe_expert_pool(FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)) == 1
    assert fwd(c, lib.moe_expert_pool(None, 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)) == 1
    assert fwd(c, lib.moe_expert_pool(FAKE, 3, FAKE, None, FAKE, FAKE, FAKE, FAKE)) == 1  # no W3
    assert fwd(c, lib.moe_expert_pool(FAKE, 3, FAKE, FAKE, FAKE, FAKE + 4, FAKE, FAKE)) == 1
    assert fwd(c, pool, nb=n - 1) == 3                             # workspace too small
    bf16 = _c(lib, n=4)
    wb = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, None, None, None, None, None, None)
    assert lib.raw_call("moe_forward_pooled", ctypes.byref(bf16), FAKE, ctypes.byref(wb),
                        ctypes.byref(pool), FAKE, None, None, None, FAKE, n, None) == 2
    big = _c(lib, n=200, weight_dtype="mxfp4")                     # n*K above the small-batch limit
    _, nbig = _size(lib, big)
    assert lib.raw_call("moe_forward_pooled", ctypes.byref(big), FAKE, ctypes.byref(w),
                        ctypes.byref(pool), FAKE, None, None, None, FAKE, nbig, None) == 2
    cls = lambda slot, ns, st=FAKE: lib.raw_call("moe_classify_experts", ctypes.byref(c), FAKE,
                                                 slot, ns, st, FAKE, FAKE, FAKE, n, None)
    assert cls(None, 3) == 1
    assert cls(FAKE, 0) == 1
    assert cls(FAKE, 3, st=None) == 1


def test_nvfp4_weight_checks(lib):
    """NVFP4 weights need their per-matrix fp32 scales; other formats must not pass them."""
    c = _c(lib, n=4, weight_dtype="nvfp4")
    _, n = _size(lib, c)
    call = lambda cfg, w: lib.raw_call("moe_forward", ctypes.byref(cfg), FAKE, ctypes.byref(w),
                                       FAKE, FAKE, n, None)
    no_g = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None)
    assert call(c, no_g) == 1
    no_g3 = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                            FAKE, None, FAKE)
    assert call(c, no_g3) == 1
    mx = _c(lib, n=4, weight_dtype="mxfp4")
    with_g = lib.moe_weights(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                             FAKE, FAKE, FAKE)
    assert call(mx, with_g) == 1
