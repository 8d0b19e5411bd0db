"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the oracle)."""
import numpy as np
import torch

import moe_speculative_verify_gb300 as m
import synth

MEDIUM = synth.LayerShape(hidden=1024, inter=512, n_experts=32, n_groups=4, topk_groups=2,
                          topk=4, n_shared=1, routed_scaling=2.5)

TOL = 1e-2       # relative Frobenius norm, bf16 out / fp32 accumulate


def rel_fro(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def run_layer(cfg, t, R, ws=None, out_fill=float("nan"), layout=m.LAYOUT_ROW_MAJOR):
    """moe_layer on the dict t; with layout=LAYOUT_TILED t's code tensors must
    already be tiled (m.tile_weights)."""
    dev = t["x"].device
    if ws is None:
        ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    out = torch.full((R, cfg.hidden), out_fill, dtype=torch.bfloat16, device=dev)
    ids = torch.empty((R, cfg.topk), dtype=torch.int32, device=dev)
    w = torch.empty((R, cfg.topk), dtype=torch.float32, device=dev)
    m.moe_layer(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t, layout),
                t.get("row_valid"), out, ws, topk_ids=ids, topk_w=w)
    torch.cuda.synchronize()
    err = m.moe_get_device_error(ws)
    assert err == 0, m.STATUS.get(err, err)
    return out, ids, w, ws


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
