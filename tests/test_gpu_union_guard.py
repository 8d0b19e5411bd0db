"""A union buffer built for another call is refused on the device.

The union's words [6] and [7] record the row count and the shape it was built
for.  Every call that reads a union compares them with its own before it
indexes anything whose offset depends on R: dispatch, the expert GEMMs, the
w8a16 GEMMs and both combine calls then compute nothing and record
MOE_ERR_INVALID_ARG (in the workspace error word, or in the union's word [5]
for the combine calls, which take no workspace).

The mismatched unions here are built for a SMALLER row count (or a smaller
top-k) inside a buffer sized for the larger call, so every index would still
stay inside the allocated buffers if a check were missing.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import synth
from gpu_helpers import MEDIUM

pytestmark = pytest.mark.gpu

INVALID_ARG = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    torch.cuda.set_device(0)


def _bufs(cfg, shape, R):
    dev = "cuda"
    return {
        "ws": torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev),
        "y_slots": torch.full((R * shape.topk, shape.hidden), 7.0, device=dev),
        "y_sh": torch.full((R, shape.hidden), 7.0, device=dev),
        "out": torch.full((R, shape.hidden), 3.0, dtype=torch.bfloat16, device=dev),
    }


def _route(cfg, shape, t, R):
    ids = torch.empty((R, shape.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((R, shape.topk), dtype=torch.float32, device="cuda")
    lg = torch.empty((R, shape.n_experts), dtype=torch.float32, device="cuda")
    m.moe_route(cfg, t["x"][:R], t["wr"], t["bias"], t["row_valid"][:R], ids, w, lg)
    return ids, w


@pytest.mark.parametrize("kind", ["rows", "topk"])
def test_union_for_another_call_is_refused(kind):
    shape, R = MEDIUM, 40
    wl = synth.Workload("guard", shape, rows=R)
    t = {k: v.cuda() for k, v in synth.make_layer(wl, device="cpu").items()}
    cfg = m.Config.from_shape(shape)
    W = m.Weights.from_tensors(t)
    # the union of a different call, in a buffer big enough for this one
    if kind == "rows":
        bcfg, bshape, bR = cfg, shape, 16
    else:
        bshape = dataclasses.replace(shape, topk=2)
        bcfg, bR = m.Config.from_shape(bshape), R
    ub = torch.zeros(max(m.moe_union_bytes(cfg, R), m.moe_union_bytes(bcfg, bR)) // 4,
                     dtype=torch.int32, device="cuda")
    bids, _ = _route(bcfg, bshape, t, bR)
    m.moe_build_union(bcfg, bids, ub)
    torch.cuda.synchronize()
    assert int(ub[6]) == bR and int(ub[5]) == 0
    _, w = _route(cfg, shape, t, R)

    b = _bufs(cfg, shape, R)
    m.moe_expert_ffn_fp8(cfg, t["x"], W, ub, b["y_slots"], b["y_sh"], b["ws"])
    assert m.moe_get_device_error(b["ws"]) == INVALID_ARG
    assert bool((b["y_slots"] == 7.0).all()) and bool((b["y_sh"] == 7.0).all())
    # the steps one by one: dispatch and each GEMM launch refuse it too
    for step in ("dispatch", "gemms", "gate_up", "down"):
        if step == "dispatch":
            m.moe_dispatch(cfg, t["x"], ub, b["ws"])
        elif step == "gemms":
            m.moe_expert_gemms_fp8(cfg, W, ub, R, b["y_slots"], b["y_sh"], b["ws"])
        elif step == "gate_up":
            m.moe_gate_up_fp8(cfg, W, ub, R, b["ws"])
        else:
            m.moe_down_fp8(cfg, W, ub, R, b["y_slots"], b["y_sh"], b["ws"])
        assert m.moe_get_device_error(b["ws"]) == INVALID_ARG, step
    assert bool((b["y_slots"] == 7.0).all())
    m.moe_expert_ffn_w8a16(cfg, t["x"], W, ub, b["y_slots"], b["y_sh"], b["ws"])
    assert m.moe_get_device_error(b["ws"]) == INVALID_ARG
    assert bool((b["y_slots"] == 7.0).all())

    # the combine calls record it in the union's word [5] and write nothing
    m.moe_combine(cfg, b["y_slots"], b["y_sh"], w, ub, b["out"])
    torch.cuda.synchronize()
    assert int(ub[5]) == INVALID_ARG
    assert bool((b["out"].float() == 3.0).all())
    ub[5] = 0
    residual = torch.zeros((R, shape.hidden), dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(shape.hidden, device="cuda")
    ro = torch.full((R, shape.hidden), 3.0, dtype=torch.bfloat16, device="cuda")
    no = torch.full((R, shape.hidden), 3.0, dtype=torch.bfloat16, device="cuda")
    m.moe_combine_add_rmsnorm(cfg, b["y_slots"], b["y_sh"], w, ub, residual, gamma, 1e-5, ro, no)
    torch.cuda.synchronize()
    assert int(ub[5]) == INVALID_ARG
    assert bool((ro.float() == 3.0).all()) and bool((no.float() == 3.0).all())

    # the union of this call goes through, in the same buffers
    ids, w = _route(cfg, shape, t, R)
    ub.zero_()
    m.moe_build_union(cfg, ids, ub)
    m.moe_expert_ffn_fp8(cfg, t["x"], W, ub, b["y_slots"], b["y_sh"], b["ws"])
    m.moe_combine(cfg, b["y_slots"], b["y_sh"], w, ub, b["out"])
    assert m.moe_get_device_error(b["ws"]) == 0
    torch.cuda.synchronize()
    assert int(ub[5]) == 0 and int(ub[6]) == R
    y = b["out"].float().cpu().numpy()
    assert np.all(np.isfinite(y)) and not np.all(y == 3.0)
