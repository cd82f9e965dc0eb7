"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each check ties an oracle function to a value printed on the pages (fixtures in
``tests/golden/`` carry the citation), a closed form, a library routine on a
special case, or brute force on tiny inputs.  The mutation tests at the end
plant plausible mistakes in the oracle and confirm that some pin catches each.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_synth
from oracle import moe_oracle as O

pytestmark = pytest.mark.filterwarnings("ignore")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _cfg(**kw):
    base = dict(name="t", n=8, d=64, d_ff=64, E=4, k=1, act_dtype="f32", weight_dtype="f32",
                gate="renorm", act="swiglu")
    base.update(kw)
    return moe_synth.MoEConfig(**base)


# ---------------------------------------------------------------- router pins

def check_router_example(golden_dir):
    g = _load(golden_dir, "router_example.json")
    p = torch.tensor([g["probs"]], dtype=torch.float64)
    logits = torch.log(p)
    probs = O.softmax_rows(logits)
    assert torch.allclose(probs, p, rtol=0, atol=1e-15)
    i1 = O.topk_select(logits, 1)
    assert i1.tolist() == [[g["top1"]["expert_1based"] - 1]]
    g1 = O.gate_weights(probs, i1, "top_prob")
    assert abs(g1.item() - g["top1"]["gate"]) < 1e-15
    i2 = O.topk_select(logits, 2)
    assert i2.tolist() == [[e - 1 for e in g["top2"]["experts_1based"]]]
    g2 = O.gate_weights(probs, i2, "renorm")
    assert [round(v, 2) for v in g2[0].tolist()] == g["top2"]["gates_printed_2dp"]
    s = g["top2"]["sum"]
    assert abs(g2[0, 0].item() - 0.45 / s) < 1e-12 and abs(g2[0, 1].item() - 0.31 / s) < 1e-12
    assert abs(g2.sum().item() - 1.0) < 1e-15


def test_router_example(golden_dir):
    check_router_example(golden_dir)


def test_router_example_through_linear_layer(golden_dir):
    """Same example driven through route(): one-hot x picks the column ln p of Wg."""
    g = _load(golden_dir, "router_example.json")
    cfg = _cfg(n=1, d=2, d_ff=32, E=4, k=1, gate="top_prob", act="relu")
    Wg = torch.tensor([[math.log(v), 7.0] for v in g["probs"]], dtype=torch.float32)
    inp = dict(x=torch.tensor([[1.0, 0.0]]), Wg=Wg, bias=None)
    r = O.route(cfg, inp)
    assert r["topk_idx"].tolist() == [[0]]
    assert abs(r["topk_gate"].item() - 0.45) < 1e-7
    # the bias belongs to the linear layer: lifting expert 4 past expert 1 moves the choice
    bias = torch.tensor([0.0, 0.0, 0.0, math.log(0.45 / 0.31) + 1e-3])
    r2 = O.route(cfg, dict(inp, bias=bias))
    assert r2["topk_idx"].tolist() == [[3]]


def check_softmax_example(golden_dir):
    g = _load(golden_dir, "softmax_example.json")
    x = torch.tensor([g["x"]], dtype=torch.float64)
    p = O.softmax_rows(x)
    denom = 1.0 / p[0, 3].item()          # p[max] = e^0 / denominator
    assert abs(denom - g["denominator_4dp"]) < 5e-5
    terms = (p * denom)[0].tolist()
    for t, want in zip(terms, g["terms_4dp"]):
        assert abs(t - want) < 5e-5
    assert abs(p.sum().item() - 1.0) < 1e-15
    # shifting all scores leaves softmax unchanged; huge scores must not overflow
    p2 = O.softmax_rows(x + 1000.0)
    assert torch.allclose(p, p2, rtol=0, atol=1e-15)


def test_softmax_example(golden_dir):
    check_softmax_example(golden_dir)


def test_softmax_rows_sum_to_one():
    g = torch.Generator().manual_seed(3)
    l = torch.randn(50, 256, generator=g, dtype=torch.float64) * 3
    p = O.softmax_rows(l)
    assert torch.all(p > 0)
    assert torch.allclose(p.sum(-1), torch.ones(50, dtype=torch.float64), atol=1e-14)


# ------------------------------------------------------------ selection pins

def brute_topk(row, k):
    """Max-sum k-subset, lowest indices among equal-sum subsets, then rank order."""
    E = len(row)
    best = None
    for sub in itertools.combinations(range(E), k):
        s = sum(row[i] for i in sub)
        if best is None or s > best[0]:
            best = (s, sub)
    chosen = list(best[1])
    # rank order: every permutation, keep the one that is non-increasing in
    # score with increasing index among equal scores
    for perm in itertools.permutations(chosen):
        ok = all(row[perm[i]] > row[perm[i + 1]] or
                 (row[perm[i]] == row[perm[i + 1]] and perm[i] < perm[i + 1])
                 for i in range(k - 1))
        if ok:
            return list(perm)
    raise AssertionError("no rank order")


def check_topk_bruteforce():
    g = torch.Generator().manual_seed(11)
    for E in (1, 2, 3, 5, 6):
        for k in range(1, E + 1):
            # scores rounded to one decimal so that ties are frequent
            l = torch.round(torch.randn(12, E, generator=g, dtype=torch.float64) * 4) / 10
            got = O.topk_select(l, k).tolist()
            for t in range(12):
                assert got[t] == brute_topk(l[t].tolist(), k), (E, k, l[t].tolist())


def test_topk_bruteforce():
    check_topk_bruteforce()


def test_topk_margin_examples():
    l = torch.tensor([[0.3, 0.1, 0.2], [1.0, 1.0, 0.0], [0.0, 5.0, 2.0]], dtype=torch.float64)
    m1 = O.topk_margin(l, 1).tolist()
    assert m1 == pytest.approx([0.1, 0.0, 3.0], abs=1e-15)
    m2 = O.topk_margin(l, 2).tolist()
    assert m2 == pytest.approx([0.1, 0.0, 2.0], abs=1e-15)
    m3 = O.topk_margin(l, 3).tolist()   # k == E: only the rank-order gaps count
    assert m3 == pytest.approx([0.1, 0.0, 2.0], abs=1e-15)
    assert math.isinf(O.topk_margin(torch.zeros(1, 1, dtype=torch.float64), 1).item())


def check_near_ties():
    """near_ties lists exactly the rows whose top-k margin is strictly below the
    threshold: gaps built from binary fractions so that "below" is exact."""
    h = 2.0 ** -16                        # the threshold of this check
    l = torch.tensor([[1.0, 1.0 - h, 0.0],            # margin h: not listed (not below)
                      [1.0, 1.0 - h / 2, 0.0],        # margin h/2: listed
                      [0.5, 0.5, 0.25],               # exact tie at rank 1: listed
                      [0.75, 0.5, 0.5 - h / 4],       # k = 2: boundary gap h/4 (k = 1: 0.25)
                      [0.0, 2.0, 1.0]], dtype=torch.float64)
    r1 = {"margin": O.topk_margin(l, 1)}
    assert O.near_ties(r1, h).tolist() == [1, 2]
    r2 = {"margin": O.topk_margin(l, 2)}
    assert O.near_ties(r2, h).tolist() == [1, 2, 3]
    # default threshold of the parity rules (1e-5 in logit units)
    r3 = {"margin": torch.tensor([0.0, 9.9e-6, 1e-5, 1.1e-5, math.inf], dtype=torch.float64)}
    assert O.near_ties(r3).tolist() == [0, 1]


def test_near_ties():
    check_near_ties()


def _bad_near_ties(routing, threshold=1e-5):       # "at most" instead of "below"
    return torch.nonzero(routing["margin"] <= threshold, as_tuple=True)[0]


# ------------------------------------------------------------- dispatch pins

def check_dispatch_example(golden_dir):
    g = _load(golden_dir, "dispatch_example.json")
    n, E = g["n_tokens"], g["n_experts"]
    assign = [g["assignment_1based"][f"t{t + 1}"] - 1 for t in range(n)]
    # router rows whose highest cell is the page's expert; t1 and t2 carry the
    # two printed maxima, the rest spread the remaining mass evenly
    probs = torch.zeros(n, E, dtype=torch.float64)
    for t, e in enumerate(assign):
        top = {0: 0.62, 1: 0.70}.get(t, 0.55)
        probs[t].fill_((1 - top) / (E - 1))
        probs[t, e] = top
    idx = O.topk_select(torch.log(probs), 1)
    assert idx.reshape(-1).tolist() == assign
    d = O.dispatch_arrays(idx, E)
    groups = [[int(g["groups_1based"][f"E{e + 1}"][i][1:]) - 1
               for i in range(len(g["groups_1based"][f"E{e + 1}"]))] for e in range(E)]
    assert d["counts"].tolist() == [len(gr) for gr in groups] == [2, 3, 0, 1]
    assert d["offsets"].tolist() == [0, 2, 5, 5, 6]
    assert d["perm"].tolist() == sum(groups, []) == [1, 4, 0, 3, 5, 2]
    assert d["inv_perm"][d["perm"]].tolist() == list(range(n))


def test_dispatch_example(golden_dir):
    check_dispatch_example(golden_dir)


def check_dispatch_invariants():
    g = torch.Generator().manual_seed(5)
    for (n, E, k) in [(1, 1, 1), (7, 3, 2), (64, 16, 4), (33, 8, 8), (200, 256, 8)]:
        l = torch.randn(n, E, generator=g, dtype=torch.float64)
        idx = O.topk_select(l, k)
        d = O.dispatch_arrays(idx, E)
        P = n * k
        assert int(d["counts"].sum()) == P
        off = d["offsets"].tolist()
        assert off[0] == 0 and off[-1] == P and all(a <= b for a, b in zip(off, off[1:]))
        perm = d["perm"].tolist()
        assert sorted(perm) == list(range(P))
        assert d["inv_perm"][d["perm"]].tolist() == list(range(P))
        flat = idx.reshape(-1).tolist()
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert all(flat[p] == e for p in seg)
            assert seg == sorted(seg)           # stable: token order inside a segment
        # every token reaches k distinct experts
        assert all(len(set(r)) == k for r in idx.tolist())


def test_dispatch_invariants():
    check_dispatch_invariants()


def test_permute_then_combine_is_identity():
    g = torch.Generator().manual_seed(9)
    n, E, k, d = 40, 6, 2, 5
    x = torch.randn(n, d, generator=g, dtype=torch.float64)
    idx = O.topk_select(torch.randn(n, E, generator=g, dtype=torch.float64), k)
    dd = O.dispatch_arrays(idx, E)
    x_perm = x[dd["perm"] // k]                    # segment q holds token perm[q] // k
    half = torch.full((n, k), 0.5, dtype=torch.float64)
    y = O.combine(x_perm, dd["inv_perm"], half)
    assert torch.equal(y, x)


def test_combine_one_hot():
    n, k, d = 3, 2, 6
    inv = torch.tensor([5, 0, 1, 4, 2, 3])
    y_perm = torch.eye(6, dtype=torch.float64)       # row q is the unit vector e_q
    gates = torch.tensor([[0.25, 0.75], [0.5, 0.5], [1.0, 2.0]], dtype=torch.float64)
    y = O.combine(y_perm, inv, gates)
    want = torch.zeros(n, d, dtype=torch.float64)
    for t in range(n):
        for j in range(k):
            want[t, inv[t * k + j]] += gates[t, j]
    assert torch.equal(y, want)


# ------------------------------------------------------------------ FFN pins

def check_ffn_closed_forms():
    ln3 = math.log(3.0)
    # SwiGLU: silu(ln 3) = ln3 * 3/4, silu(-ln 3) = -ln3 / 4, silu(0) = 0, silu(-1) = -1/(1+e)
    x = torch.tensor([[ln3, 2.0, -1.0]], dtype=torch.float64)
    W1 = torch.tensor([[1, 0, 0], [-1, 0, 0], [0, 0, 1], [0, 0, 0]], dtype=torch.float64)
    W3 = torch.tensor([[0, 1, 0], [0, 1, 0], [0, 0.5, 0], [1, 0, 0]], dtype=torch.float64)
    W2 = torch.tensor([[1, -1, 0, 0], [0, 0, 1, 0], [0, 1, 0, 3]], dtype=torch.float64)
    y = O.expert_ffn(x, W1, W2, "swiglu", W3)[0].tolist()
    want = [2 * ln3, -1.0 / (1.0 + math.e), -0.5 * ln3]
    assert y == pytest.approx(want, abs=1e-14)
    # ReLU
    x = torch.tensor([[1.5, -2.0, 0.25]], dtype=torch.float64)
    W1 = torch.tensor([[1, 0, 0], [-1, 0, 0], [0, 0, 2], [0, 1, -1]], dtype=torch.float64)
    W2 = torch.tensor([[1, 1, 0, 0], [0, 0, 2, -1], [0, 1, 0, 1]], dtype=torch.float64)
    y = O.expert_ffn(x, W1, W2, "relu")[0].tolist()
    assert y == pytest.approx([1.5, 1.0, 0.0], abs=1e-15)


def test_ffn_closed_forms():
    check_ffn_closed_forms()


def _np_bf16(t):
    """Independent bf16 decode for the library cross-check: bits << 16 as float32."""
    u = t.contiguous().view(torch.int16).numpy().astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype,act,gate", [("bf16", "swiglu", "renorm"), ("f32", "relu", "top_prob"),
                                            ("bf16", "relu", "renorm")])
def test_single_expert_is_dense_ffn(dtype, act, gate):
    """E = 1: the router's only choice has probability 1, so the layer is the dense FFN."""
    cfg = _cfg(n=9, d=64, d_ff=96, E=1, k=1, act_dtype=dtype, weight_dtype=dtype, gate=gate, act=act)
    inp = moe_synth.make_inputs(cfg, seed=1)
    res = O.forward(cfg, inp)
    assert torch.all(res["routing"]["topk_gate"] == 1.0)
    conv = _np_bf16 if dtype == "bf16" else (lambda t: t.numpy().astype(np.float64))
    X = conv(inp["x"])
    A = np.matmul(X, conv(inp["W1"][0]).T)
    if act == "relu":
        H = np.maximum(A, 0.0)
    else:
        H = A / (1.0 + np.exp(-A)) * np.matmul(X, conv(inp["W3"][0]).T)
    Y = np.matmul(H, conv(inp["W2"][0]).T)
    assert np.allclose(res["y"].numpy(), Y, rtol=1e-12, atol=1e-13)


def test_forward_bruteforce_tiny():
    """Scalar loops, no grouping and no matrix routine, on a tiny layer."""
    cfg = _cfg(n=5, d=32, d_ff=8, E=3, k=2, act_dtype="f32", weight_dtype="f32")
    inp = moe_synth.make_inputs(cfg, seed=2)
    res = O.forward(cfg, inp)
    x = inp["x"].double().tolist()
    Wg = inp["Wg"].double().tolist()
    W1, W3, W2 = (inp[k].double().tolist() for k in ("W1", "W3", "W2"))
    for t in range(cfg.n):
        logit = [sum(x[t][i] * Wg[e][i] for i in range(cfg.d)) for e in range(cfg.E)]
        mx = max(logit)
        ex = [math.exp(v - mx) for v in logit]
        p = [v / sum(ex) for v in ex]
        chosen = brute_topk(logit, cfg.k)
        z = sum(p[e] for e in chosen)
        y = [0.0] * cfg.d
        for e in chosen:
            h = []
            for f in range(cfg.d_ff):
                a = sum(W1[e][f][i] * x[t][i] for i in range(cfg.d))
                b = sum(W3[e][f][i] * x[t][i] for i in range(cfg.d))
                h.append(a / (1 + math.exp(-a)) * b)
            for o in range(cfg.d):
                y[o] += p[e] / z * sum(W2[e][o][f] * h[f] for f in range(cfg.d_ff))
        assert res["y"][t].tolist() == pytest.approx(y, rel=1e-10, abs=1e-13)


def test_shared_expert_added_unweighted():
    cfg = _cfg(n=4, d=32, d_ff=32, E=2, k=1, act_dtype="bf16", weight_dtype="bf16", d_ff_shared=64)
    inp = moe_synth.make_inputs(cfg, seed=4)
    res = O.forward(cfg, inp)
    inp0 = dict(inp, Ws1=None, Ws2=None, Ws3=None)
    res0 = O.forward(moe_synth.MoEConfig(**{**cfg.__dict__, "d_ff_shared": 0}), inp0)
    X = _np_bf16(inp["x"])
    A = X @ _np_bf16(inp["Ws1"]).T
    B = X @ _np_bf16(inp["Ws3"]).T
    S = (A / (1 + np.exp(-A)) * B) @ _np_bf16(inp["Ws2"]).T
    assert np.allclose(res["y"].numpy() - res0["y"].numpy(), S, rtol=1e-10, atol=1e-12)


# -------------------------------------------------------- routing statistics

def check_aux_loss_example(golden_dir):
    g = _load(golden_dir, "aux_loss_example.json")
    E = g["n_experts"]
    # four token distributions whose first column averages P1 = 0.5825 and whose
    # argmax is always expert 1 (the page's unbalanced router)
    probs = torch.tensor([[0.70, 0.10, 0.10, 0.10],
                          [0.55, 0.15, 0.15, 0.15],
                          [0.48, 0.40, 0.06, 0.06],
                          [0.60, 0.30, 0.05, 0.05]], dtype=torch.float64)
    assert abs(probs[:, 0].mean().item() - g["unbalanced"]["P1"]) < 1e-12
    top1 = O.topk_select(torch.log(probs), 1)[:, 0]
    st = O.routing_statistics(probs, top1, 1.0)
    assert st["f"].tolist() == [1.0, 0.0, 0.0, 0.0]
    assert abs(st["aux"] - E * g["unbalanced"]["P1"]) < 1e-12
    assert round(st["aux"], 2) == g["unbalanced"]["E_sum_fP_printed_2dp"]
    assert round(O.routing_statistics(probs, top1, g["alpha"])["aux"], 4) == \
        g["alpha_terms_printed"]["unbalanced"]
    # balanced: each expert is the argmax once; any rows that sum to one give 1.0
    bal = torch.tensor([[0.40, 0.20, 0.20, 0.20],
                        [0.10, 0.50, 0.20, 0.20],
                        [0.25, 0.05, 0.45, 0.25],
                        [0.30, 0.10, 0.10, 0.50]], dtype=torch.float64)
    t1 = O.topk_select(torch.log(bal), 1)[:, 0]
    sb = O.routing_statistics(bal, t1, 1.0)
    assert sb["f"].tolist() == g["balanced"]["f"]
    assert abs(sb["aux"] - g["balanced"]["E_sum_fP"]) < 1e-12
    assert abs(O.routing_statistics(bal, t1, g["alpha"])["aux"] -
               g["alpha_terms_printed"]["balanced"]) < 1e-12


def test_aux_loss_example(golden_dir):
    check_aux_loss_example(golden_dir)


def test_aux_loss_uniform_router_closed_form():
    """p_i(x) = 1/E for every token: P_i = 1/E, so aux = alpha * sum_i f_i = alpha."""
    g = torch.Generator().manual_seed(17)
    for E in (2, 8, 128):
        n = 97
        probs = torch.full((n, E), 1.0 / E, dtype=torch.float64)
        top1 = torch.randint(0, E, (n,), generator=g)
        st = O.routing_statistics(probs, top1, 0.37)
        assert abs(st["aux"] - 0.37) < 1e-12
        assert abs(st["f"].sum().item() - 1.0) < 1e-12


# ---------------------------------------------------------------- MXFP4 pins

def check_mxfp4(golden_dir):
    g = _load(golden_dir, "e2m1_values.json")
    codes = torch.arange(16, dtype=torch.uint8)
    vals = O.e2m1_value(codes).tolist()
    for c in range(16):
        want = g["e2m1_code_to_value"][str(c)]
        assert vals[c] == want and math.copysign(1, vals[c]) == math.copysign(1, want), c
    for s, want in g["e8m0_examples"].items():
        v = O.e8m0_value(torch.tensor([int(s)], dtype=torch.uint8)).item()
        if want == "NaN":
            assert math.isnan(v)
        else:
            assert v == want
    # every code at every scale the workloads draw (2^-8 .. 2^-4), 32 per block
    for s in range(119, 124):
        packed = torch.tensor([[c | (c << 4) for c in range(16)]], dtype=torch.uint8)
        scales = torch.tensor([[s]], dtype=torch.uint8)
        dec = O.mxfp4_decode(packed, scales)[0].tolist()
        for c in range(16):
            w = g["e2m1_code_to_value"][str(c)] * 2.0 ** (s - 127)
            assert dec[2 * c] == w and dec[2 * c + 1] == w
    pb = g["packed_bytes_example"]
    packed = torch.tensor([pb["bytes"] * 4], dtype=torch.uint8)    # 32 elements = one block
    dec = O.mxfp4_decode(packed, torch.tensor([[127]], dtype=torch.uint8))[0].tolist()
    assert dec[:8] == pb["elements"]
    assert [math.copysign(1, v) for v in dec[:8]] == [math.copysign(1, v) for v in pb["elements"]]
    # two blocks with different scales: the scale index is element // 32
    packed = torch.full((1, 32), 0x22, dtype=torch.uint8)          # all elements = 1.0
    dec = O.mxfp4_decode(packed, torch.tensor([[120, 126]], dtype=torch.uint8))[0]
    assert torch.all(dec[:32] == 2.0 ** -7) and torch.all(dec[32:] == 2.0 ** -1)


def test_mxfp4_codec(golden_dir):
    check_mxfp4(golden_dir)


def test_mxfp4_expert_bruteforce():
    """MXFP4 expert weights decoded element by element from the table, tiny layer."""
    cfg = _cfg(n=3, d=64, d_ff=32, E=2, k=1, act_dtype="bf16", weight_dtype="mxfp4")
    inp = moe_synth.make_inputs(cfg, seed=6)
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

    def dec(packed, scales, rows, cols):
        out = np.zeros((rows, cols))
        for r in range(rows):
            for c in range(cols):
                byte = int(packed[r, c // 2])
                code = (byte & 15) if c % 2 == 0 else (byte >> 4)
                v = table[code & 7] * (-1 if code & 8 else 1)
                out[r, c] = v * 2.0 ** (int(scales[r, c // 32]) - 127)
        return out

    res = O.forward(cfg, inp)
    X = _np_bf16(inp["x"])
    for t in range(cfg.n):
        e = int(res["routing"]["topk_idx"][t, 0])
        W1 = dec(inp["W1q"][e], inp["S1"][e], cfg.d_ff, cfg.d)
        W3 = dec(inp["W3q"][e], inp["S3"][e], cfg.d_ff, cfg.d)
        W2 = dec(inp["W2q"][e], inp["S2"][e], cfg.d, cfg.d_ff)
        A = W1 @ X[t]
        h = A / (1 + np.exp(-A)) * (W3 @ X[t])
        assert np.allclose(res["y"][t].numpy(), W2 @ h, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- NVFP4 pins

def check_e4m3(golden_dir):
    g = _load(golden_dir, "e4m3_values.json")
    for code, want in g["examples"].items():
        v = O.e4m3_value(torch.tensor([int(code)], dtype=torch.uint8)).item()
        if want == "NaN":
            assert math.isnan(v), code
        else:
            assert v == want and math.copysign(1, v) == math.copysign(1, want), code


def test_e4m3_examples(golden_dir):
    check_e4m3(golden_dir)


def test_e4m3_matches_library_type():
    """All 256 bytes against torch's float8_e4m3fn (the same OCP encoding)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ours = O.e4m3_value(codes)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64)
    assert torch.equal(torch.isnan(ours), torch.isnan(lib))
    ok = ~torch.isnan(ours)
    assert torch.equal(ours[ok], lib[ok])


def check_nvfp4_bruteforce():
    """NVFP4 expert weights decoded element by element (block = element // 16), tiny layer."""
    cfg = _cfg(n=3, d=64, d_ff=32, E=2, k=1, act_dtype="bf16", weight_dtype="nvfp4")
    inp = moe_synth.make_inputs(cfg, seed=6)
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    e4m3 = lambda b: float(torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn)
                           .to(torch.float64))

    def dec(packed, scales, gs, rows, cols):
        out = np.zeros((rows, cols))
        for r in range(rows):
            for c in range(cols):
                byte = int(packed[r, c // 2])
                code = (byte & 15) if c % 2 == 0 else (byte >> 4)
                v = table[code & 7] * (-1 if code & 8 else 1)
                out[r, c] = v * e4m3(int(scales[r, c // 16])) * float(gs)
        return out

    res = O.forward(cfg, inp)
    X = _np_bf16(inp["x"])
    for t in range(cfg.n):
        e = int(res["routing"]["topk_idx"][t, 0])
        W1 = dec(inp["W1q"][e], inp["S1"][e], inp["G1"][e], cfg.d_ff, cfg.d)
        W3 = dec(inp["W3q"][e], inp["S3"][e], inp["G3"][e], cfg.d_ff, cfg.d)
        W2 = dec(inp["W2q"][e], inp["S2"][e], inp["G2"][e], cfg.d, cfg.d_ff)
        A = W1 @ X[t]
        h = A / (1 + np.exp(-A)) * (W3 @ X[t])
        assert np.allclose(res["y"][t].numpy(), W2 @ h, rtol=1e-12, atol=1e-12)


def test_nvfp4_expert_bruteforce():
    check_nvfp4_bruteforce()


def test_nvfp4_unit_scales_equal_mxfp4():
    """Block scales of 1.0 (E4M3 0x38, E8M0 127) and a matrix scale of 1: both
    formats decode the same codes to the same values."""
    packed = torch.randint(0, 256, (5, 32), dtype=torch.uint8, generator=torch.Generator().manual_seed(1))
    nv = O.nvfp4_decode(packed, torch.full((5, 4), 0x38, dtype=torch.uint8), 1.0)
    mx = O.mxfp4_decode(packed, torch.full((5, 2), 127, dtype=torch.uint8))
    assert torch.equal(nv, mx)


# ------------------------------------------------- expert-slot classification

def check_expert_cache_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "expert_cache_example.json")))
    E = g["n_experts"]
    slot_of = torch.full((E,), -1, dtype=torch.int32)
    for e, s in g["slot_of"].items():
        slot_of[int(e)] = s
    r = O.classify_experts(torch.tensor(g["selections"]), E, slot_of)
    want = g["expected"]
    assert r["miss_list"].tolist() == want["miss_list"]
    assert torch.nonzero(r["state"] == 1, as_tuple=True)[0].tolist() == want["hits"]
    assert (r["state"] == -1).sum().item() == E - want["selected"]
    for key in ("selected", "resident", "lookups", "served"):
        assert r[key] == want[key], key


def test_expert_cache_example(golden_dir):
    check_expert_cache_example(golden_dir)


def _classify_bruteforce(idx, E, slot_of):
    """Loop over the (token, slot) lookups with a set of seen experts."""
    seen, served = set(), 0
    for row in idx.tolist():
        for e in row:
            seen.add(e)
            served += int(slot_of[e]) >= 0
    misses = sorted(e for e in seen if int(slot_of[e]) < 0)
    return seen, misses, served


def check_classify_bruteforce():
    g = torch.Generator().manual_seed(23)
    for _ in range(40):
        E = int(torch.randint(1, 40, (1,), generator=g))
        k = int(torch.randint(1, E + 1, (1,), generator=g))
        n = int(torch.randint(1, 12, (1,), generator=g))
        idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(n)])
        n_slots = int(torch.randint(1, E + 1, (1,), generator=g))
        resident = int(torch.randint(0, n_slots + 1, (1,), generator=g))
        slot_of = moe_synth.make_slot_table(E, n_slots, resident,
                                            seed=int(torch.randint(0, 1 << 30, (1,), generator=g)))
        r = O.classify_experts(idx, E, slot_of)
        seen, misses, served = _classify_bruteforce(idx, E, slot_of)
        assert r["miss_list"].tolist() == misses
        assert r["selected"] == len(seen)
        assert r["resident"] == len(seen) - len(misses)
        assert r["lookups"] == n * k and r["served"] == served
        for e in range(E):
            want = -1 if e not in seen else (1 if int(slot_of[e]) >= 0 else 0)
            assert int(r["state"][e]) == want


def test_classify_bruteforce():
    check_classify_bruteforce()


def test_classify_all_or_none_resident():
    idx = torch.tensor([[5, 1], [1, 2], [7, 5]])
    everyone = torch.arange(8, dtype=torch.int32)
    r = O.classify_experts(idx, 8, everyone)
    assert r["miss_list"].numel() == 0 and r["served"] == r["lookups"] == 6
    assert r["selected"] == r["resident"] == 4
    nobody = torch.full((8,), -1, dtype=torch.int32)
    r = O.classify_experts(idx, 8, nobody)
    assert r["miss_list"].tolist() == [1, 2, 5, 7] and r["served"] == 0 and r["resident"] == 0


def test_classify_random_router_serves_resident_fraction(golden_dir):
    """Uniformly random selections: the served share of lookups approaches the
    resident share of experts."""
    g = json.load(open(os.path.join(golden_dir, "expert_cache_example.json")))["random_router"]
    E, n, k = 4608, 4096, 4
    gen = torch.Generator().manual_seed(5)
    idx = torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(n)])
    resident = round(g["resident_fraction"] * E)
    slot_of = moe_synth.make_slot_table(E, resident, resident, seed=9)
    r = O.classify_experts(idx, E, slot_of)
    assert abs(r["served"] / r["lookups"] - g["resident_fraction"]) < 0.01


# ------------------------------------------------------------ mutation tests

def _bad_topk(logits, k):                        # ties go to the higher index
    E = logits.shape[-1]
    order = torch.sort(-logits.flip(-1), dim=-1, stable=True).indices
    return (E - 1 - order)[:, :k]


def _bad_gate(probs, idx, mode):                 # forgets to renormalise
    return probs.gather(1, idx.to(torch.int64))


def _bad_ffn(X, W1, W2, act, W3=None):           # silu on the linear branch
    if act == "relu":
        return torch.clamp(X @ W1.T, min=0) @ W2.T
    return (O.silu(X @ W3.T) * (X @ W1.T)) @ W2.T


def _e2m1_bias0(code):
    c = code.to(torch.int64)
    e = (c >> 1) & 3
    m = (c & 1).to(torch.float64)
    mag = torch.where(e == 0, m * 0.5, torch.pow(2.0, e.to(torch.float64)) * (1 + m * 0.5))
    return torch.where(((c >> 3) & 1) == 1, -mag, mag)


def _bad_dispatch(idx, E):                       # unstable order inside a segment
    d = _orig_dispatch(idx, E)
    perm = d["perm"].clone()
    off = d["offsets"].tolist()
    for e in range(E):
        perm[off[e]:off[e + 1]] = perm[off[e]:off[e + 1]].flip(0)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    return dict(d, perm=perm, inv_perm=inv)


_orig_dispatch = O.dispatch_arrays


def _bad_stats(probs, top1, alpha):             # P_i averaged over experts, not tokens
    n, E = probs.shape
    P = probs.sum(dim=1)[:E] / E if n >= E else probs.sum(dim=1).mean().repeat(E)
    f = torch.bincount(top1.reshape(-1).to(torch.int64), minlength=E).to(torch.float64) / n
    return dict(P=P, f=f, aux=alpha * E * float((f * P).sum()))


def _bad_nvfp4(packed, scales, gscale):          # one scale per 32 elements, not 16
    lo = packed & 0x0F
    hi = packed >> 4
    codes = torch.stack((lo, hi), dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = O.e2m1_value(codes)
    K = vals.shape[-1]
    sc = O.e4m3_value(scales[..., 0::2])
    return (vals.reshape(*vals.shape[:-1], K // 32, 32) * sc.unsqueeze(-1)).reshape(vals.shape) * gscale


def _bad_classify(idx, E, slot_of):              # counts distinct experts as lookups served
    r = _orig_classify(idx, E, slot_of)
    return dict(r, served=r["resident"])


_orig_classify = O.classify_experts


def _bad_classify_slot0(idx, E, slot_of):        # slot 0 taken for "not resident"
    return _orig_classify(idx, E, torch.where(slot_of.to(torch.int64) > 0, slot_of.to(torch.int64),
                                              torch.full_like(slot_of.to(torch.int64), -1)))


def _bad_softmax(logits):                        # no max subtraction and wrong axis
    ex = torch.exp(logits)
    return ex / ex.sum(dim=0, keepdim=True)


MUTANTS = [
    ("topk_select", _bad_topk, lambda gd: check_topk_bruteforce()),
    ("gate_weights", _bad_gate, check_router_example),
    ("expert_ffn", _bad_ffn, lambda gd: check_ffn_closed_forms()),
    ("e2m1_value", _e2m1_bias0, check_mxfp4),
    ("dispatch_arrays", _bad_dispatch, check_dispatch_example),
    ("softmax_rows", _bad_softmax, check_softmax_example),
    ("routing_statistics", _bad_stats, check_aux_loss_example),
    ("nvfp4_decode", _bad_nvfp4, lambda gd: check_nvfp4_bruteforce()),
    ("classify_experts", _bad_classify, check_expert_cache_example),
    ("classify_experts", _bad_classify_slot0, lambda gd: check_classify_bruteforce()),
    ("near_ties", _bad_near_ties, lambda gd: check_near_ties()),
]


@pytest.mark.parametrize("name,mutant,pin", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, golden_dir, name, mutant, pin):
    pin(golden_dir)                               # passes on the real oracle
    monkeypatch.setattr(O, name, mutant)
    with pytest.raises(AssertionError):
        pin(golden_dir)
