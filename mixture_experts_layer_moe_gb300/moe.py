"""Python binding of libmoe_gb300.so (argument marshalling only).

Every function here has the name of the C entry point it calls (include/moe.h)
and passes device pointers of torch tensors plus the current CUDA stream.  No
step of the layer runs in Python: if the library is missing, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

_DTYPE = {"f32": 0, "bf16": 1, "mxfp4": 2, "nvfp4": 3}
_GATE = {"top_prob": 0, "renorm": 1}
_ACT = {"relu": 0, "swiglu": 1}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


STAGE_HOOK = ctypes.CFUNCTYPE(None, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p)
STAGES = ("route", "dispatch", "ffn_up", "ffn_down", "shared", "combine", "end", "fused")


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n", "d", "d_ff", "n_experts", "top_k", "act_dtype", "weight_dtype", "gate",
                 "act", "d_ff_shared")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("Wg", "router_bias", "W1", "W3", "W2", "S1", "S3", "S2", "Ws1", "Ws3", "Ws2",
                 "G1", "G3", "G2")]


class moe_expert_pool(ctypes.Structure):
    _fields_ = [("slot_of", ctypes.c_void_p), ("n_slots", ctypes.c_int32),
                ("W1", ctypes.c_void_p), ("W3", ctypes.c_void_p), ("W2", ctypes.c_void_p),
                ("S1", ctypes.c_void_p), ("S3", ctypes.c_void_p), ("S2", ctypes.c_void_p)]


# indices of the classification counts (MOE_POOL_*)
POOL_SELECTED, POOL_RESIDENT, POOL_LOOKUPS, POOL_SERVED = 0, 1, 2, 3


class moe_workspace_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "logits", "topk_idx", "topk_gate", "counts", "offsets", "perm",
                 "inv_perm", "x_perm", "h", "y_perm", "y_shared", "h_shared", "act16", "total")]


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run mixture_experts_layer_moe_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    cfgp = ctypes.POINTER(moe_config)
    wp = ctypes.POINTER(moe_weights)
    pp = ctypes.POINTER(moe_expert_pool)
    sig = {
        "moe_workspace_size": [cfgp, ctypes.POINTER(SZ)],
        "moe_workspace_layout_of": [cfgp, ctypes.POINTER(moe_workspace_layout)],
        "moe_route": [cfgp, P, wp, P, P, P, P, SZ, P],
        "moe_route_noalloc": [cfgp, P, wp, P, P, P, P],
        "moe_route_noalloc_status": [P, ctypes.POINTER(ctypes.c_int32)],
        "moe_route_stats": [cfgp, P, P, ctypes.c_float, P, P, P, P, SZ, P],
        "moe_dispatch": [cfgp, P, P, P, P, P, P, P, P, SZ, P],
        "moe_expert_ffn": [cfgp, P, P, wp, P, P, SZ, P],
        "moe_combine": [cfgp, P, P, P, P, P, P, SZ, P],
        "moe_forward": [cfgp, P, wp, P, P, SZ, P],
        "moe_forward_staged": [cfgp, P, wp, P, P, SZ, P, STAGE_HOOK, P],
        "moe_classify_experts": [cfgp, P, P, ctypes.c_int32, P, P, P, P, SZ, P],
        "moe_forward_pooled": [cfgp, P, wp, pp, P, P, P, P, P, SZ, P],
        "moe_forward_pooled_staged": [cfgp, P, wp, pp, P, P, P, P, P, SZ, P, STAGE_HOOK, P],
        "moe_status_check": [P, P, ctypes.POINTER(ctypes.c_int32)],
        "moe_status_clear": [P, P],
        "moe_selftest_wait_timeout": [P, ctypes.c_uint64, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I32
    lib.moe_status_string.argtypes = [I32]
    lib.moe_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise MoEError(status, where)


def make_config(cfg) -> moe_config:
    """moe_config from any object with the MoEConfig fields (moe_synth.MoEConfig)."""
    if isinstance(cfg, moe_config):
        return cfg
    return moe_config(cfg.n, cfg.d, cfg.d_ff, cfg.E, cfg.k, _DTYPE[cfg.act_dtype],
                      _DTYPE[cfg.weight_dtype], _GATE[cfg.gate], _ACT[cfg.act],
                      cfg.d_ff_shared)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def make_weights(inputs: dict) -> moe_weights:
    """moe_weights from a dict of device tensors (keys as in moe_synth.make_inputs)."""
    g = inputs.get
    mx = g("W1q") is not None
    return moe_weights(
        _ptr(g("Wg")), _ptr(g("bias")),
        _ptr(g("W1q") if mx else g("W1")), _ptr(g("W3q") if mx else g("W3")),
        _ptr(g("W2q") if mx else g("W2")),
        _ptr(g("S1")), _ptr(g("S3")), _ptr(g("S2")),
        _ptr(g("Ws1")), _ptr(g("Ws3")), _ptr(g("Ws2")),
        _ptr(g("G1")), _ptr(g("G3")), _ptr(g("G2")))


def make_pool(slot_of: torch.Tensor, pool: dict) -> moe_expert_pool:
    """moe_expert_pool from the device slot table and a dict of device pool
    tensors (keys as in moe_synth.make_pool: W1q, W3q, W2q, S1, S3, S2)."""
    g = pool.get
    return moe_expert_pool(_ptr(slot_of), int(g("W1q").shape[0]), _ptr(g("W1q")), _ptr(g("W3q")),
                           _ptr(g("W2q")), _ptr(g("S1")), _ptr(g("S3")), _ptr(g("S2")))


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def moe_workspace_size(cfg) -> int:
    c = make_config(cfg)
    out = ctypes.c_size_t(0)
    _check(_lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_workspace_layout_of(cfg) -> dict:
    c = make_config(cfg)
    L = moe_workspace_layout()
    _check(_lib.moe_workspace_layout_of(ctypes.byref(c), ctypes.byref(L)), "moe_workspace_layout_of")
    return {name: getattr(L, name) for name, _ in moe_workspace_layout._fields_}


def alloc_workspace(cfg, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor of moe_workspace_size(cfg) bytes (256-byte aligned)."""
    ws = torch.zeros(moe_workspace_size(cfg), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def moe_route(cfg, x, w: moe_weights, topk_idx, topk_gate, probs, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_route(ctypes.byref(c), _ptr(x), ctypes.byref(w), _ptr(topk_idx),
                          _ptr(topk_gate), _ptr(probs), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route")


def moe_route_noalloc(cfg, x, w: moe_weights, topk_idx, topk_gate, probs, stream=None):
    """moe_route without a workspace (scratch in a static device array; calls must not overlap)."""
    c = make_config(cfg)
    _check(_lib.moe_route_noalloc(ctypes.byref(c), _ptr(x), ctypes.byref(w), _ptr(topk_idx),
                                  _ptr(topk_gate), _ptr(probs), _stream(stream)),
           "moe_route_noalloc")


def moe_route_noalloc_status(stream=None) -> tuple[int, int]:
    """(status, detail) of the last moe_route_noalloc on this device (synchronises the stream)."""
    detail = ctypes.c_int32(0)
    st = _lib.moe_route_noalloc_status(_stream(stream), ctypes.byref(detail))
    return st, detail.value


def moe_route_stats(cfg, probs, topk_idx, alpha, P, f, aux, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_route_stats(ctypes.byref(c), _ptr(probs), _ptr(topk_idx), float(alpha),
                                _ptr(P), _ptr(f), _ptr(aux), _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_route_stats")


def moe_dispatch(cfg, topk_idx, x, counts, offsets, perm, inv_perm, x_perm, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_dispatch(ctypes.byref(c), _ptr(topk_idx), _ptr(x), _ptr(counts),
                             _ptr(offsets), _ptr(perm), _ptr(inv_perm), _ptr(x_perm), _ptr(ws),
                             ws.numel(), _stream(stream)), "moe_dispatch")


def moe_expert_ffn(cfg, x_perm, offsets, w: moe_weights, y_perm, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_expert_ffn(ctypes.byref(c), _ptr(x_perm), _ptr(offsets), ctypes.byref(w),
                               _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(cfg, y_perm, inv_perm, topk_gate, y_shared, y, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_combine(ctypes.byref(c), _ptr(y_perm), _ptr(inv_perm), _ptr(topk_gate),
                            _ptr(y_shared), _ptr(y), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_combine")


def moe_forward(cfg, x, w: moe_weights, y, ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_forward(ctypes.byref(c), _ptr(x), ctypes.byref(w), _ptr(y), _ptr(ws),
                            ws.numel(), _stream(stream)), "moe_forward")


def moe_forward_staged(cfg, x, w: moe_weights, y, ws, hook, stream=None):
    """hook(stage: int, kernels_so_far: int) runs on this thread before each stage is enqueued."""
    c = make_config(cfg)
    cb = STAGE_HOOK(lambda st, k, _u: hook(st, k))
    _check(_lib.moe_forward_staged(ctypes.byref(c), _ptr(x), ctypes.byref(w), _ptr(y), _ptr(ws),
                                   ws.numel(), _stream(stream), cb, None), "moe_forward_staged")


def moe_classify_experts(cfg, topk_idx, slot_of, n_slots, state, miss_list, counts, ws,
                         stream=None):
    c = make_config(cfg)
    _check(_lib.moe_classify_experts(ctypes.byref(c), _ptr(topk_idx), _ptr(slot_of), int(n_slots),
                                     _ptr(state), _ptr(miss_list), _ptr(counts), _ptr(ws),
                                     ws.numel(), _stream(stream)), "moe_classify_experts")


def moe_forward_pooled(cfg, x, w: moe_weights, pool: moe_expert_pool, y, state, miss_list, counts,
                       ws, stream=None):
    c = make_config(cfg)
    _check(_lib.moe_forward_pooled(ctypes.byref(c), _ptr(x), ctypes.byref(w), ctypes.byref(pool),
                                   _ptr(y), _ptr(state), _ptr(miss_list), _ptr(counts), _ptr(ws),
                                   ws.numel(), _stream(stream)), "moe_forward_pooled")


def moe_forward_pooled_staged(cfg, x, w: moe_weights, pool: moe_expert_pool, y, state, miss_list,
                              counts, ws, hook, stream=None):
    """hook(stage: int, kernels_so_far: int) runs on this thread before each stage is enqueued."""
    c = make_config(cfg)
    cb = STAGE_HOOK(lambda st, k, _u: hook(st, k))
    _check(_lib.moe_forward_pooled_staged(ctypes.byref(c), _ptr(x), ctypes.byref(w),
                                          ctypes.byref(pool), _ptr(y), _ptr(state),
                                          _ptr(miss_list), _ptr(counts), _ptr(ws), ws.numel(),
                                          _stream(stream), cb, None), "moe_forward_pooled_staged")


def moe_status_check(ws, stream=None) -> tuple[int, int]:
    detail = ctypes.c_int32(0)
    st = _lib.moe_status_check(_ptr(ws), _stream(stream), ctypes.byref(detail))
    return st, detail.value


def moe_status_clear(ws, stream=None):
    _check(_lib.moe_status_clear(_ptr(ws), _stream(stream)), "moe_status_clear")


def moe_selftest_wait_timeout(ws, limit_ns: int, stream=None):
    _check(_lib.moe_selftest_wait_timeout(_ptr(ws), int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def raw_call(name: str, *args) -> int:
    """Call an entry point with raw ctypes arguments (for argument-check tests)."""
    return getattr(_lib, name)(*args)


def library() -> ctypes.CDLL:
    return _lib
