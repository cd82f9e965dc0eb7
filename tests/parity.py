"""Helpers shared by the GPU parity tests: run the library, run the oracle on the
same seeded inputs, and compare under the stated tolerances.

Tolerances (derived from the arithmetic: bf16 rounding of h and y_perm, fp32
accumulation, exact MXFP4 decode):
  * routing indices, counts, offsets, perm, inv_perm: bit-exact, except tokens
    whose oracle top-k margin is below NEAR_TIE (listed, then checked for
    validity instead of equality);
  * gates: |g - g_oracle| <= GATE_ATOL;
  * fp32 layer: |y - o| <= 1e-4 * max(|o|, 1e-2 * max_row |o|) per element;
  * bf16 / MXFP4 layer: max_i |y_i - o_i| <= 2e-2 * max_i |o_i| per row.
"""
from __future__ import annotations

import torch

import moe_synth
from oracle import moe_oracle as O

NEAR_TIE = 1e-5
GATE_ATOL = 1e-5
F32_RTOL = 1e-4
F32_FLOOR = 1e-2
LOWP_ROW_TOL = 2e-2


class LazyExperts:
    """Index e -> expert e's tensor copied to the host (the oracle reads experts one at a time)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu()


def oracle_inputs(inputs: dict) -> dict:
    out = {}
    for k, v in inputs.items():
        if v is None:
            out[k] = None
        elif k in ("W1", "W3", "W2", "W1q", "W3q", "W2q", "S1", "S3", "S2"):
            out[k] = LazyExperts(v)
        else:
            out[k] = v.cpu()
    return out


def ws_view(ws: torch.Tensor, layout: dict, name: str, dtype, count: int) -> torch.Tensor:
    off = layout[name]
    nbytes = count * torch.empty((), dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def run_forward(lib, cfg, inputs: dict):
    """moe_forward on device inputs -> (y, ws, layout, intermediates on host)."""
    w = lib.make_weights(inputs)
    ws = lib.alloc_workspace(cfg)
    y = torch.empty(cfg.n, cfg.d, dtype=inputs["x"].dtype, device="cuda")
    lib.moe_forward(cfg, inputs["x"], w, y, ws)
    st, detail = lib.moe_status_check(ws)
    assert st == 0, (lib.status_string(st), detail)
    L = lib.moe_workspace_layout_of(cfg)
    P = cfg.n * cfg.k
    inter = dict(
        topk_idx=ws_view(ws, L, "topk_idx", torch.int32, P).view(cfg.n, cfg.k).cpu(),
        topk_gate=ws_view(ws, L, "topk_gate", torch.float32, P).view(cfg.n, cfg.k).cpu(),
        counts=ws_view(ws, L, "counts", torch.int32, cfg.E).cpu(),
        offsets=ws_view(ws, L, "offsets", torch.int32, cfg.E + 1).cpu(),
        perm=ws_view(ws, L, "perm", torch.int32, P).cpu(),
        inv_perm=ws_view(ws, L, "inv_perm", torch.int32, P).cpu(),
        logits=ws_view(ws, L, "logits", torch.float32, cfg.n * cfg.E).view(cfg.n, cfg.E).cpu(),
    )
    return y, ws, L, inter


def check_routing(cfg, oracle_routing: dict, gpu_idx: torch.Tensor, gpu_gate: torch.Tensor):
    """Bit-exact selection except listed near ties; those must still be valid choices.

    Returns the list of near-tie tokens (oracle margin < NEAR_TIE)."""
    margin = oracle_routing["margin"]
    listed = torch.nonzero(margin < NEAR_TIE, as_tuple=True)[0]
    keep = torch.ones(cfg.n, dtype=torch.bool)
    keep[listed] = False
    o_idx = oracle_routing["topk_idx"].to(torch.int32)
    mism = torch.nonzero((o_idx != gpu_idx).any(dim=1) & keep, as_tuple=True)[0]
    assert mism.numel() == 0, (
        f"routing differs on {mism.numel()} tokens with margin >= {NEAR_TIE}: "
        f"{mism[:10].tolist()} margins {margin[mism[:10]].tolist()}")
    logits = oracle_routing["logits"]
    for t in listed.tolist():
        sel = gpu_idx[t].tolist()
        assert len(set(sel)) == cfg.k and all(0 <= e < cfg.E for e in sel)
        kth = torch.sort(logits[t], descending=True).values[cfg.k - 1].item()
        for e in sel:
            assert logits[t, e].item() >= kth - NEAR_TIE, (t, sel)
    gdiff = (gpu_gate.double() - oracle_routing["topk_gate"]).abs()
    gdiff[listed] = 0
    assert gdiff.max().item() <= GATE_ATOL, gdiff.max().item()
    return listed.tolist()


def check_dispatch(cfg, gpu_idx: torch.Tensor, inter: dict):
    """Dispatch arrays must equal the plain definition applied to the GPU's own selection."""
    d = O.dispatch_arrays(gpu_idx.to(torch.int64), cfg.E)
    for key in ("counts", "offsets", "perm", "inv_perm"):
        assert torch.equal(inter[key].to(torch.int64), d[key]), key


def routing_with_gpu_ties(cfg, oracle_routing: dict, gpu_idx: torch.Tensor, listed) -> dict:
    """Oracle routing where listed near-tie tokens take the GPU's (valid) choice."""
    if not listed:
        return oracle_routing
    r = dict(oracle_routing)
    idx = r["topk_idx"].clone()
    for t in listed:
        idx[t] = gpu_idx[t].to(idx.dtype)
    r["topk_idx"] = idx
    r["topk_gate"] = O.gate_weights(r["probs"], idx, cfg.gate)
    return r


def check_output(cfg, y_gpu: torch.Tensor, y_oracle: torch.Tensor):
    y = y_gpu.double().cpu()
    o = y_oracle
    if cfg.act_dtype == "f32":
        rowmax = o.abs().max(dim=1, keepdim=True).values
        denom = torch.maximum(o.abs(), F32_FLOOR * rowmax)
        err = ((y - o).abs() / denom).max().item()
        assert err <= F32_RTOL, f"fp32 relative error {err}"
        return err
    rowmax = o.abs().max(dim=1).values
    rowerr = (y - o).abs().max(dim=1).values
    ratio = (rowerr / rowmax).max().item()
    assert ratio <= LOWP_ROW_TOL, f"row error / row max-abs = {ratio}"
    return ratio


def sample_rows(cfg, topk_idx: torch.Tensor, sample: int, seed: int) -> torch.Tensor:
    """Seeded sample of `sample` token rows (first and last included), widened so
    that every expert some token selects has at least one of its tokens in it."""
    g = torch.Generator().manual_seed(1234 + seed)
    chosen = torch.zeros(cfg.n, dtype=torch.bool)
    chosen[torch.randperm(cfg.n, generator=g)[:sample]] = True
    chosen[0] = chosen[cfg.n - 1] = True
    idx = topk_idx.to(torch.int64)
    covered = torch.zeros(cfg.E, dtype=torch.bool)
    covered[idx[chosen].reshape(-1)] = True
    used = torch.bincount(idx.reshape(-1), minlength=cfg.E) > 0
    for e in torch.nonzero(used & ~covered, as_tuple=True)[0].tolist():
        t = torch.nonzero((idx == e).any(dim=1), as_tuple=True)[0][0].item()
        chosen[t] = True
        covered[idx[t]] = True
    return torch.nonzero(chosen, as_tuple=True)[0]


def full_parity(lib, cfg, seed=0, sample=None):
    """moe_forward vs oracle.  sample: number of token rows for the expert outputs
    (None = all); a sample is widened to cover every expert with c_e > 0.
    Routing and dispatch are always checked for every token."""
    inputs = moe_synth.make_inputs(cfg, seed=seed, device="cuda")
    y, ws, L, inter = run_forward(lib, cfg, inputs)
    oin = oracle_inputs(inputs)
    r = O.route(cfg, oin)
    listed = check_routing(cfg, r, inter["topk_idx"], inter["topk_gate"])
    check_dispatch(cfg, inter["topk_idx"], inter)
    r2 = routing_with_gpu_ties(cfg, r, inter["topk_idx"], listed)
    if sample is None or sample >= cfg.n:
        tokens = torch.arange(cfg.n)
    else:
        tokens = sample_rows(cfg, inter["topk_idx"], sample, seed)
    sel = inter["topk_idx"][tokens].to(torch.int64).reshape(-1)
    covered = torch.bincount(sel, minlength=cfg.E) > 0
    used = inter["counts"] > 0
    assert torch.equal(covered, used), "the checked rows miss a non-empty expert"
    res = O.forward(cfg, oin, tokens=tokens, routing=r2)
    err = check_output(cfg, y[tokens.cuda()], res["y"])
    logit_err = (inter["logits"].double() - r["logits"]).abs().max().item()
    ties = [dict(token=t, margin=float(r["margin"][t]),
                 oracle=[int(v) for v in r["topk_idx"][t].tolist()],
                 gpu=[int(v) for v in inter["topk_idx"][t].tolist()]) for t in listed]
    return dict(err=err, near_ties=listed, near_tie_records=ties, counts=inter["counts"], y=y,
                inputs=inputs, ws=ws, logit_err=logit_err, rows_checked=int(tokens.numel()),
                experts_covered=int(covered.sum()), experts_used=int(used.sum()))
