"""Python binding of the fp8 MoE decode / speculative-verify layer (libmoe_verify.so).

Argument marshalling only: every function forwards to the C entry point of
the same name in include/moe_verify.h, passing torch tensors' device
pointers and the current CUDA stream.  Every step of the layer runs in the
library's sm_103a kernels; there is no Python or CPU fallback.  A missing
library raises at import of the first call.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "MoeError", "Config", "Weights", "load", "build", "moe_route", "moe_build_union",
    "moe_expert_ffn_fp8", "moe_combine", "moe_layer", "moe_union_bytes",
    "moe_ffn_workspace_bytes", "moe_workspace_bytes", "moe_get_device_error",
    "moe_diag_wait_timeout", "moe_status_string", "moe_dispatch", "moe_gate_up_fp8",
    "moe_down_fp8", "ffn_layout", "moe_layer_noalloc", "moe_expert_gemms_fp8",
    "moe_greedy_verify", "moe_combine_add_rmsnorm", "union_layout", "rows_per_item",
    "router_rows_per_warp",
    "MOE_MAX_ROWS", "moe_expert_ffn_w8a16", "moe_layer_w8a16", "W8A16_MAX_ROWS",
    "moe_tile_weights", "tile_weights", "LAYOUT_ROW_MAJOR", "LAYOUT_TILED",
    "moe_workspace_size",
]

LAYOUT_ROW_MAJOR = 0
LAYOUT_TILED = 1
CODE_KEYS = ("w_gate", "w_up", "w_down", "sh_gate", "sh_up", "sh_down")

MOE_MAX_ROWS = 4096
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_WORKSPACE"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("inter", C.c_int32), ("n_experts", C.c_int32),
                ("n_groups", C.c_int32), ("topk_groups", C.c_int32), ("topk", C.c_int32),
                ("n_shared", C.c_int32), ("routed_scaling", C.c_float),
                ("wait_timeout_us", C.c_uint32)]

    @classmethod
    def from_shape(cls, s, wait_timeout_us: int = 0) -> "Config":
        return cls(s.hidden, s.inter, s.n_experts, s.n_groups, s.topk_groups, s.topk,
                   s.n_shared, s.routed_scaling, wait_timeout_us)


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
        "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up", "sh_s_down")] + [
        ("layout", C.c_int32)]

    @classmethod
    def from_tensors(cls, t: dict, layout: int = LAYOUT_ROW_MAJOR) -> "Weights":
        """From a dict with w_gate/s_gate/... and sh_gate/sh_s_gate/... tensors
        whose code tensors are in the given layout (tile_weights makes a tiled
        dict).  The result holds references to those tensors, so the device
        memory its pointers name stays allocated while it exists."""
        def p(k):
            v = t.get(k)
            return None if v is None else v.data_ptr()
        w = cls(p("w_gate"), p("w_up"), p("w_down"), p("s_gate"), p("s_up"), p("s_down"),
                p("sh_gate"), p("sh_up"), p("sh_down"), p("sh_s_gate"), p("sh_s_up"),
                p("sh_s_down"), layout)
        w._tensors = [t[k] for k in CODE_KEYS + ("s_gate", "s_up", "s_down", "sh_s_gate",
                                                 "sh_s_up", "sh_s_down") if t.get(k) is not None]
        return w


_LIB: Optional[C.CDLL] = None


def build(force: bool = False) -> str:
    return _build.build(force=force)


def load() -> C.CDLL:
    """Load the in-tree library; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libmoe_verify.so is not built ({_build.LIB}); run "
                          "moe_speculative_verify_gb300.build()")
    L = C.CDLL(_build.LIB)
    P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
    cfg = C.POINTER(Config)
    L.moe_status_string.restype = C.c_char_p
    L.moe_status_string.argtypes = [C.c_int]
    for n in ("moe_union_bytes", "moe_ffn_workspace_bytes", "moe_workspace_bytes"):
        getattr(L, n).restype = SZ
        getattr(L, n).argtypes = [cfg, I32]
    L.moe_workspace_size.argtypes = [cfg, I32, C.POINTER(SZ)]
    L.moe_route.argtypes = [cfg, P, P, P, P, I32, P, P, P, P]
    L.moe_build_union.argtypes = [cfg, P, I32, P, SZ, P]
    L.moe_expert_ffn_fp8.argtypes = [cfg, P, C.POINTER(Weights), P, I32, P, P, P, SZ, P]
    L.moe_combine.argtypes = [cfg, P, P, P, P, I32, P, P]
    L.moe_dispatch.argtypes = [cfg, P, P, I32, P, SZ, P]
    L.moe_gate_up_fp8.argtypes = [cfg, C.POINTER(Weights), P, I32, P, SZ, P]
    L.moe_down_fp8.argtypes = [cfg, C.POINTER(Weights), P, I32, P, P, P, SZ, P]
    L.moe_expert_gemms_fp8.argtypes = [cfg, C.POINTER(Weights), P, I32, P, P, P, SZ, P]
    L.moe_layer.argtypes = [cfg, P, P, P, C.POINTER(Weights), P, I32, P, P, P, P, SZ, P]
    L.moe_get_device_error.argtypes = [P, I32, P]
    L.moe_tile_weights.argtypes = [P, P, C.c_int64, I32, I32, P]
    L.moe_combine_add_rmsnorm.argtypes = [cfg, P, P, P, P, I32, P, P, C.c_float, P, P, P]
    L.moe_greedy_verify.argtypes = [P, I32, I32, I32, P, P, P, P, P, P]
    L.moe_layer_noalloc.argtypes = [cfg, P, P, P, C.POINTER(Weights), P, I32, P, P, P, P, P]
    L.moe_expert_ffn_w8a16.argtypes = L.moe_expert_ffn_fp8.argtypes
    L.moe_layer_w8a16.argtypes = L.moe_layer.argtypes
    L.moe_diag_wait_timeout.argtypes = [P, C.c_uint32, P]
    for n in ("moe_route", "moe_build_union", "moe_expert_ffn_fp8", "moe_combine", "moe_layer",
              "moe_get_device_error", "moe_diag_wait_timeout", "moe_dispatch", "moe_layer_noalloc", "moe_greedy_verify", "moe_combine_add_rmsnorm",
              "moe_gate_up_fp8", "moe_down_fp8", "moe_expert_gemms_fp8", "moe_expert_ffn_w8a16",
              "moe_layer_w8a16", "moe_workspace_size"):
        getattr(L, n).restype = C.c_int
    _LIB = L
    return L


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MoeError(status, where)


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_union_bytes(cfg: Config, max_rows: int) -> int:
    return load().moe_union_bytes(C.byref(cfg), max_rows)


def moe_ffn_workspace_bytes(cfg: Config, max_rows: int) -> int:
    return load().moe_ffn_workspace_bytes(C.byref(cfg), max_rows)


def moe_workspace_bytes(cfg: Config, max_rows: int) -> int:
    return load().moe_workspace_bytes(C.byref(cfg), max_rows)


def moe_workspace_size(cfg: Config, max_rows: int) -> int:
    """Bytes of one buffer that serves every entry point at up to max_rows rows."""
    n = C.c_size_t(0)
    _check(load().moe_workspace_size(C.byref(cfg), max_rows, C.byref(n)), "moe_workspace_size")
    return n.value


def moe_route(cfg: Config, x, w_router, bias, row_valid, topk_ids, topk_w, logits,
              stream=None) -> None:
    R = 0 if x is None else x.shape[0]
    _check(load().moe_route(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(row_valid),
                            R, _ptr(topk_ids), _ptr(topk_w), _ptr(logits), _stream(stream)),
           "moe_route")


def moe_build_union(cfg: Config, topk_ids, union_buf, stream=None) -> None:
    R = topk_ids.shape[0]
    _check(load().moe_build_union(C.byref(cfg), _ptr(topk_ids), R, _ptr(union_buf),
                                  union_buf.numel() * union_buf.element_size(), _stream(stream)),
           "moe_build_union")


def moe_expert_ffn_fp8(cfg: Config, x, weights: Weights, union_buf, y_slots, y_shared, ws,
                       stream=None) -> None:
    R = x.shape[0]
    _check(load().moe_expert_ffn_fp8(C.byref(cfg), _ptr(x), C.byref(weights), _ptr(union_buf), R,
                                     _ptr(y_slots), _ptr(y_shared), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_fp8")


def moe_expert_ffn_w8a16(cfg: Config, x, weights: Weights, union_buf, y_slots, y_shared, ws,
                         stream=None) -> None:
    """The expert FFNs with bf16 activations and weights dequantised in the kernel."""
    R = x.shape[0]
    _check(load().moe_expert_ffn_w8a16(C.byref(cfg), _ptr(x), C.byref(weights), _ptr(union_buf),
                                       R, _ptr(y_slots), _ptr(y_shared), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_w8a16")


def moe_dispatch(cfg: Config, x, union_buf, ws, stream=None) -> None:
    _check(load().moe_dispatch(C.byref(cfg), _ptr(x), _ptr(union_buf), x.shape[0], _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "moe_dispatch")


def moe_gate_up_fp8(cfg: Config, weights: Weights, union_buf, R: int, ws, stream=None) -> None:
    _check(load().moe_gate_up_fp8(C.byref(cfg), C.byref(weights), _ptr(union_buf), R, _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "moe_gate_up_fp8")


def moe_down_fp8(cfg: Config, weights: Weights, union_buf, R: int, y_slots, y_shared, ws,
                 stream=None) -> None:
    _check(load().moe_down_fp8(C.byref(cfg), C.byref(weights), _ptr(union_buf), R,
                               _ptr(y_slots), _ptr(y_shared), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "moe_down_fp8")


def moe_expert_gemms_fp8(cfg: Config, weights: Weights, union_buf, R: int, y_slots, y_shared, ws,
                         stream=None) -> None:
    _check(load().moe_expert_gemms_fp8(C.byref(cfg), C.byref(weights), _ptr(union_buf), R,
                                       _ptr(y_slots), _ptr(y_shared), _ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_gemms_fp8")


def moe_combine(cfg: Config, y_slots, y_shared, topk_w, union_buf, out, stream=None) -> None:
    R = out.shape[0]
    _check(load().moe_combine(C.byref(cfg), _ptr(y_slots), _ptr(y_shared), _ptr(topk_w),
                              _ptr(union_buf), R, _ptr(out), _stream(stream)), "moe_combine")


def moe_combine_add_rmsnorm(cfg: Config, y_slots, y_shared, topk_w, union_buf, residual, gamma,
                            eps: float, residual_out, normed, stream=None) -> None:
    R = residual.shape[0]
    _check(load().moe_combine_add_rmsnorm(C.byref(cfg), _ptr(y_slots), _ptr(y_shared),
                                          _ptr(topk_w), _ptr(union_buf), R, _ptr(residual),
                                          _ptr(gamma), float(eps), _ptr(residual_out),
                                          _ptr(normed), _stream(stream)),
           "moe_combine_add_rmsnorm")


def moe_layer(cfg: Config, x, w_router, bias, weights: Weights, row_valid, out, ws,
              topk_ids=None, topk_w=None, stream=None) -> None:
    R = x.shape[0]
    _check(load().moe_layer(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), C.byref(weights),
                            _ptr(row_valid), R, _ptr(out), _ptr(topk_ids), _ptr(topk_w),
                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer")


def moe_layer_w8a16(cfg: Config, x, w_router, bias, weights: Weights, row_valid, out, ws,
                    topk_ids=None, topk_w=None, stream=None) -> None:
    """moe_layer with the w8a16 expert FFNs (R <= W8A16_MAX_ROWS)."""
    R = x.shape[0]
    _check(load().moe_layer_w8a16(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias),
                                  C.byref(weights), _ptr(row_valid), R, _ptr(out),
                                  _ptr(topk_ids), _ptr(topk_w), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_w8a16")


def moe_layer_noalloc(cfg: Config, x, w_router, bias, weights: Weights, row_valid, out,
                      topk_ids=None, topk_w=None, device_status=None, stream=None) -> None:
    """moe_layer with the library's own fixed scratch array (no workspace argument)."""
    R = x.shape[0]
    _check(load().moe_layer_noalloc(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias),
                                    C.byref(weights), _ptr(row_valid), R, _ptr(out),
                                    _ptr(topk_ids), _ptr(topk_w), _ptr(device_status),
                                    _stream(stream)), "moe_layer_noalloc")


def moe_greedy_verify(logits, draft, n_draft, argmax_out, accept_len, out_tokens,
                      stream=None) -> None:
    """Greedy verify of spans of 8 rows; logits fp32 or bf16 [R, V] on the device."""
    R, V = logits.shape
    _check(load().moe_greedy_verify(_ptr(logits), 1 if logits.dtype == torch.bfloat16 else 0, V, R,
                                    _ptr(draft), _ptr(n_draft), _ptr(argmax_out), _ptr(accept_len),
                                    _ptr(out_tokens), _stream(stream)), "moe_greedy_verify")


def moe_tile_weights(src, dst, stream=None) -> None:
    """src: uint8 [n, rows, cols] row-major codes on the device; dst: a device
    uint8 tensor of the same number of bytes, written in the tiled layout."""
    n, rows, cols = src.shape
    if dst.numel() != src.numel() or dst.dtype != torch.uint8 or src.dtype != torch.uint8:
        raise MoeError(1, "moe_tile_weights")
    _check(load().moe_tile_weights(_ptr(src), _ptr(dst), n, rows, cols, _stream(stream)),
           "moe_tile_weights")


def tile_weights(t: dict, stream=None) -> dict:
    """A copy of the weight dict t whose six code tensors are in the tiled
    layout (new tensors of the same shapes, bytes permuted by
    moe_tile_weights); the scales and any other entries are shared with t.
    Pass the result to Weights.from_tensors(..., layout=LAYOUT_TILED)."""
    out = dict(t)
    for k in CODE_KEYS:
        v = t.get(k)
        if v is None:
            continue
        src = v.view(torch.uint8).contiguous()
        dst = torch.empty_like(src)
        moe_tile_weights(src, dst, stream)
        out[k] = dst.view(v.dtype)
    return out


def moe_get_device_error(ws, clear: bool = True, stream=None) -> int:
    """Synchronises the stream; returns the workspace's device error code (0 = OK)."""
    return load().moe_get_device_error(_ptr(ws), 1 if clear else 0, _stream(stream))


def moe_diag_wait_timeout(ws, timeout_us: int, stream=None) -> None:
    _check(load().moe_diag_wait_timeout(_ptr(ws), timeout_us, _stream(stream)),
           "moe_diag_wait_timeout")


# ---------------------------------------------------------------- layouts --
W8A16_MAX_ROWS = 64          # the w8a16 variant's row limit (mirrors the library)

def router_rows_per_warp(R: int, E: int, n_sms: int = None) -> int:
    """Rows a consumer warp of the large-R router kernel takes per tile (tiles
    of 4x that many rows): 6, 7, 8 or 9 (mirrors the library's choice; n_sms
    defaults to the current device's SM count)."""
    if n_sms is None:
        import torch
        n_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cost = {6: 45, 7: 50, 8: 55, 9: 62}
    best, best_cost = 6, None
    for rt in (6, 7, 8, 9):
        tiles = -(-R // (4 * rt)) * -(-E // 32)
        grid = min(tiles, max(n_sms, 1))
        c = -(-tiles // grid) * cost[rt]
        if best_cost is None or c < best_cost:
            best, best_cost = rt, c
    return best


def rows_per_item(R: int) -> int:
    """Rows per GEMM work item chosen for a call with R rows (mirrors the library)."""
    return 16 if R <= 64 else (32 if R <= 256 else 64)


def union_layout(cfg: Config, R: int) -> dict:
    """Word offsets of the union buffer arrays (moe_build_union's documented layout)."""
    E, K, S = cfg.n_experts, cfg.topk, cfg.n_shared
    KS = K + S
    w = 8
    out = {"counts": w}
    w += E + 1
    out["offsets"] = w
    w += E + 2
    out["ulist"] = w
    w += E + 1
    out["pos"] = w
    w += R * KS
    out["src"] = w
    w += R * KS
    w = (w + 3) // 4 * 4
    out["items"] = w
    return out


def ffn_layout(cfg: Config, R: int) -> dict:
    """Byte offsets of the FFN workspace regions (mirrors the library's carve-up)."""
    def up(v, mlt):
        return (v + mlt - 1) // mlt * mlt
    H, I, E, K, S = cfg.hidden, cfg.inter, cfg.n_experts, cfg.topk, cfg.n_shared
    rows = up(R * (K + S), 64) + 64
    n_ready = R * (K + S) // 16 + min(E, R * K) + S + 1
    out = {"rows": rows, "ctl": 0, "ready": 256, "n_ready": n_ready,
           "sched": 256 + n_ready * 4}
    b = up(256 + (n_ready + 2) * 4, 256)     # per-item counters, then 2 scheduler words
    out["xg"] = b
    b = up(b + rows * H, 256)
    out["xs"] = b
    b = up(b + rows * (H // 128) * 4, 256)
    out["hq"] = b
    b = up(b + rows * I, 256)
    out["hs"] = b
    out["bytes"] = up(b + rows * (I // 128) * 4, 256)
    if R <= W8A16_MAX_ROWS:
        out["xb"] = out["xg"]
        out["hb"] = up(out["xb"] + rows * H * 2, 256)
        out["bytes"] = max(out["bytes"], up(out["hb"] + rows * I * 2, 256))
    return out
