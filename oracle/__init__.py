"""ctypes wrapper of the CPU oracle (oracle/moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: tests/, the smoke check and the bench's CPU-baseline
leg use it.  The product path never imports this package.  Arrays are numpy,
host memory; bf16 travels as uint16 bit patterns, e4m3 as uint8 codes.

Every function mirrors one exported C function; the C source states the
definitions and cites the pages they follow.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import numpy as np

from . import build as _build

_LIB = None


class _Cfg(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("inter", C.c_int32), ("n_experts", C.c_int32),
                ("n_groups", C.c_int32), ("topk_groups", C.c_int32), ("topk", C.c_int32),
                ("n_shared", C.c_int32), ("routed_scaling", C.c_float)]


def _cfg(c) -> _Cfg:
    return _Cfg(c.hidden, c.inter, c.n_experts, c.n_groups, c.topk_groups, c.topk,
                c.n_shared, c.routed_scaling)


def lib() -> C.CDLL:
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_e4m3_decode.restype = C.c_float
        L.orc_e4m3_decode.argtypes = [C.c_uint8]
        L.orc_e4m3_encode.restype = C.c_uint8
        L.orc_e4m3_encode.argtypes = [C.c_float]
        L.orc_e4m3_encode_n.argtypes = [P, C.c_int64, P]
        L.orc_bf16_to_f32.restype = C.c_float
        L.orc_bf16_to_f32.argtypes = [C.c_uint16]
        L.orc_f64_to_bf16.restype = C.c_uint16
        L.orc_f64_to_bf16.argtypes = [C.c_double]
        L.orc_exp.restype = C.c_float
        L.orc_exp.argtypes = [C.c_float]
        L.orc_sigmoid.restype = C.c_float
        L.orc_sigmoid.argtypes = [C.c_float]
        L.orc_quant_1x128.argtypes = [P, C.c_int32, P, P]
        L.orc_router_logits.argtypes = [C.POINTER(_Cfg), P, P, C.c_int32, P]
        L.orc_route_from_logits.argtypes = [C.POINTER(_Cfg), P, P, P, C.c_int32, P, P]
        L.orc_route.argtypes = [C.POINTER(_Cfg), P, P, P, P, C.c_int32, P, P, P]
        L.orc_build_union.argtypes = [C.POINTER(_Cfg), P, C.c_int32, P, P, P, P, P, P]
        L.orc_expert_ffn.argtypes = [C.POINTER(_Cfg), P, P, P, P, P, P, P, P, P, P, P,
                                     C.c_int32]
        L.orc_moe_layer.argtypes = [C.POINTER(_Cfg)] + [P] * 15 + [P, C.c_int32, P,
                                                                   C.c_int32, P, P, P, P,
                                                                   C.c_int32]
        L.orc_expert_ffn_a16.argtypes = [C.POINTER(_Cfg)] + [P] * 8 + [C.c_int32, C.c_int32]
        L.orc_moe_layer_variant.argtypes = L.orc_moe_layer.argtypes + [C.c_int32]
        L.orc_greedy_verify.argtypes = [P, C.c_int32, C.c_int32, P, P, C.c_int32, P, P, P]
        L.orc_add_rmsnorm.argtypes = [P, P, P, C.c_float, P, C.c_int32, C.c_int32, P, P]
        L.orc_num_threads.restype = C.c_int
        L.orc_set_num_threads.argtypes = [C.c_int]
        _LIB = L
    return _LIB


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ------------------------------------------------------------------ formats --
def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    table = np.array([lib().orc_e4m3_decode(i) for i in range(256)], dtype=np.float32)
    return table[codes]


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_n(_p(v), v.size, _p(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(v: float) -> int:
    return int(lib().orc_f64_to_bf16(float(v)))


def own_exp(a: float) -> float:
    return float(lib().orc_exp(float(a)))


def sigmoid(l: float) -> float:
    return float(lib().orc_sigmoid(float(l)))


def quant_1x128(v) -> tuple[np.ndarray, np.ndarray]:
    v = _c(v, np.float32)
    assert v.ndim == 1 and v.size % 128 == 0
    q = np.empty(v.size, dtype=np.uint8)
    s = np.empty(v.size // 128, dtype=np.float32)
    lib().orc_quant_1x128(_p(v), v.size, _p(q), _p(s))
    return q, s


# ------------------------------------------------------------------ routing --
def router_logits(cfg, x_bf16, wr) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    wr = _c(wr, np.float32)
    R = x.shape[0]
    out = np.empty((R, cfg.n_experts), dtype=np.float32)
    c = _cfg(cfg)
    lib().orc_router_logits(C.byref(c), _p(x), _p(wr), R, _p(out))
    return out


def route_from_logits(cfg, logits, bias, row_valid=None):
    lg = _c(logits, np.float32)
    R = lg.shape[0]
    ids = np.empty((R, cfg.topk), dtype=np.int32)
    w = np.empty((R, cfg.topk), dtype=np.float32)
    rv = None if row_valid is None else _c(row_valid, np.uint8)
    c = _cfg(cfg)
    lib().orc_route_from_logits(C.byref(c), _p(lg), _p(_c(bias, np.float32)), _p(rv), R,
                                _p(ids), _p(w))
    return ids, w


def route(cfg, x_bf16, wr, bias, row_valid=None):
    """Returns (topk_ids [R,K] int32, topk_w [R,K] fp32, logits [R,E] fp32)."""
    x = _c(x_bf16, np.uint16)
    R = x.shape[0]
    ids = np.empty((R, cfg.topk), dtype=np.int32)
    w = np.empty((R, cfg.topk), dtype=np.float32)
    logits = np.empty((R, cfg.n_experts), dtype=np.float32)
    rv = None if row_valid is None else _c(row_valid, np.uint8)
    c = _cfg(cfg)
    lib().orc_route(C.byref(c), _p(x), _p(_c(wr, np.float32)), _p(_c(bias, np.float32)),
                    _p(rv), R, _p(ids), _p(w), _p(logits))
    return ids, w, logits


def build_union(cfg, topk_ids) -> dict:
    ids = _c(topk_ids, np.int32)
    R = ids.shape[0]
    E, K = cfg.n_experts, cfg.topk
    counts = np.empty(E + 1, dtype=np.int32)
    offsets = np.empty(E + 2, dtype=np.int32)
    ulist = np.empty(E + 1, dtype=np.int32)
    n_union = np.zeros(1, dtype=np.int32)
    pos = np.empty(R * (K + 1), dtype=np.int32)
    src = np.full(R * (K + 1), -1, dtype=np.int32)
    c = _cfg(cfg)
    lib().orc_build_union(C.byref(c), _p(ids), R, _p(counts), _p(offsets), _p(ulist),
                          _p(n_union), _p(pos), _p(src))
    U = int(n_union[0])
    T = int(offsets[E + 1])
    return {"counts": counts, "offsets": offsets, "ulist": ulist[:U + 1], "n_union": U,
            "pos": pos.reshape(R, K + 1), "src": src[:T], "n_gathered": T,
            "n_valid": int(counts[E])}


# --------------------------------------------------------------- expert FFN --
def expert_ffn(cfg, xq, xs, wg, sg, wu, su, wd, sd, acc64: bool = True):
    """One expert on one quantised row.  Returns (o [H] fp64, hq [I] u8, hs [I/128] f32)."""
    H, I = cfg.hidden, cfg.inter
    out = np.empty(H, dtype=np.float64)
    hq = np.empty(I, dtype=np.uint8)
    hs = np.empty(I // 128, dtype=np.float32)
    args = [_c(xq, np.uint8), _c(xs, np.float32), _c(wg, np.uint8), _c(sg, np.float32),
            _c(wu, np.uint8), _c(su, np.float32), _c(wd, np.uint8), _c(sd, np.float32)]
    c = _cfg(cfg)
    lib().orc_expert_ffn(C.byref(c), *[_p(a) for a in args], _p(out), _p(hq), _p(hs),
                         1 if acc64 else 0)
    return out, hq, hs


_VARIANTS = {"fp8": 0, "w8a16": 1, "exact": 2}


def expert_ffn_a16(cfg, x_bf16, wg, sg, wu, su, wd, sd, round16: bool = True,
                   acc64: bool = True) -> np.ndarray:
    """One expert on one bf16 row (uint16 [H]) with 16-bit activations: the
    w8a16 variant (round16) or the unrounded yardstick.  Returns o [H] fp64."""
    out = np.empty(cfg.hidden, dtype=np.float64)
    args = [_c(x_bf16, np.uint16), _c(wg, np.uint8), _c(sg, np.float32), _c(wu, np.uint8),
            _c(su, np.float32), _c(wd, np.uint8), _c(sd, np.float32)]
    c = _cfg(cfg)
    lib().orc_expert_ffn_a16(C.byref(c), *[_p(a) for a in args], _p(out), 1 if round16 else 0,
                             1 if acc64 else 0)
    return out


def moe_layer(cfg, t: dict, rows=None, acc64: bool = True, variant: str = "fp8"):
    """The whole layer on host arrays.

    t holds x (uint16 [R,H]), wr, bias, w_gate/s_gate, w_up/s_up, w_down/s_down,
    sh_gate/sh_s_gate, sh_up/sh_s_up, sh_down/sh_s_down and optionally row_valid.
    variant: "fp8" (activations and h quantised per 1x128 to e4m3), "w8a16"
    (bf16 activations, weights dequantised to bf16, h rounded to bf16) or
    "exact" (no activation or weight rounding).  Returns dict(out uint16 [R,H],
    ids, wts, y_acc fp64 [R,H]); rows not listed in `rows` are left zero.
    """
    x = _c(t["x"], np.uint16)
    R = x.shape[0]
    H, K = cfg.hidden, cfg.topk
    arrs = [_c(t["wr"], np.float32), _c(t["bias"], np.float32),
            _c(t["w_gate"], np.uint8), _c(t["s_gate"], np.float32),
            _c(t["w_up"], np.uint8), _c(t["s_up"], np.float32),
            _c(t["w_down"], np.uint8), _c(t["s_down"], np.float32),
            _c(t["sh_gate"], np.uint8), _c(t["sh_s_gate"], np.float32),
            _c(t["sh_up"], np.uint8), _c(t["sh_s_up"], np.float32),
            _c(t["sh_down"], np.uint8), _c(t["sh_s_down"], np.float32)]
    rv = t.get("row_valid")
    rv = None if rv is None else _c(rv, np.uint8)
    rl = None if rows is None else _c(rows, np.int32)
    out = np.zeros((R, H), dtype=np.uint16)
    ids = np.full((R, K), -1, dtype=np.int32)
    wts = np.zeros((R, K), dtype=np.float32)
    y = np.zeros((R, H), dtype=np.float64)
    c = _cfg(cfg)
    lib().orc_moe_layer_variant(C.byref(c), _p(x), *[_p(a) for a in arrs], _p(rv), R, _p(rl),
                                0 if rl is None else rl.size, _p(out), _p(ids), _p(wts), _p(y),
                                1 if acc64 else 0, _VARIANTS[variant])
    return {"out": out, "ids": ids, "wts": wts, "y_acc": y}


# ----------------------------------------------------- greedy verify + accept --
def greedy_verify(logits, draft, n_draft):
    """Spans of 8 rows: returns (accept_len [n_span], out [n_span*8], argmax [R]).

    logits: fp32 [R, V] or bf16 bit patterns (uint16) [R, V]; draft int32 [R];
    n_draft int32 [n_span] (drafts in each span, 0..7)."""
    lg = np.ascontiguousarray(logits)
    is_bf16 = 1 if lg.dtype == np.uint16 else 0
    if not is_bf16:
        lg = _c(lg, np.float32)
    R, V = lg.shape
    n_span = R // 8
    acc = np.empty(n_span, dtype=np.int32)
    out = np.empty(R, dtype=np.int32)
    am = np.empty(R, dtype=np.int32)
    lib().orc_greedy_verify(_p(lg), is_bf16, V, _p(_c(draft, np.int32)), _p(_c(n_draft, np.int32)),
                            n_span, _p(acc), _p(out), _p(am))
    return acc, out, am


# ------------------------------------------------------ residual add + RMSNorm --
def add_rmsnorm(y, residual_bf16, gamma, eps, row_valid=None):
    """(residual_out bf16 bits [R,H], normed bf16 bits [R,H]) from fp64 y [R,H]."""
    y = _c(y, np.float64)
    R, H = y.shape
    ro = np.empty((R, H), dtype=np.uint16)
    no = np.empty((R, H), dtype=np.uint16)
    rv = None if row_valid is None else _c(row_valid, np.uint8)
    lib().orc_add_rmsnorm(_p(y), _p(_c(residual_bf16, np.uint16)), _p(_c(gamma, np.float32)),
                          float(eps), _p(rv), R, H, _p(ro), _p(no))
    return ro, no
