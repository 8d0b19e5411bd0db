"""moe_layer_noalloc: the layer for callers that cannot allocate device memory.

Such a caller (a plugin whose host framework owns all device memory, code that
must not call cudaMalloc) gets the layer with the library's own fixed scratch
array instead of a workspace.  The test calls it through the C ABI twice in a
row, on three cases one after the other (so the array holds the previous
call's leftovers each time) -- 8 and 37 rows (selection and union in one
kernel, one fused GEMM launch) and 100 rows (separate selection and union
kernels, gate/up and down GEMMs as two launches, whose tile scheduler words
stay in the array between calls) -- and checks it against moe_layer with a
workspace: the same routing ids and weights, the same output within the
parity tolerance, pads zero-filled, and a clean device status.  It also checks that a row count
whose workspace would not fit in the array is refused.

This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import synth
from gpu_helpers import MEDIUM, TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    torch.cuda.set_device(0)


def _layer(shape, rows, pads):
    wl = synth.Workload("noalloc", shape, rows=rows, pads=tuple(pads))
    return {k: v.cuda() for k, v in synth.make_layer(wl, device="cpu").items()}


def test_noalloc_matches_moe_layer_twice():
    for shape, R, pads in ((synth.TINY, 8, ()), (MEDIUM, 37, (0, 36)), (MEDIUM, 100, (5, 99))):
        t = _layer(shape, R, pads)
        cfg = m.Config.from_shape(shape)
        ref_out, ref_ids, ref_w, _ = run_layer(cfg, t, R)
        ref_y = bf16_bits_to_f64(bf16_to_np(ref_out))
        valid = t["row_valid"].cpu().numpy() != 0
        for _ in range(2):
            out = torch.full((R, shape.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
            ids = torch.empty((R, shape.topk), dtype=torch.int32, device="cuda")
            w = torch.empty((R, shape.topk), dtype=torch.float32, device="cuda")
            status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
            m.moe_layer_noalloc(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t),
                                t["row_valid"], out, topk_ids=ids, topk_w=w,
                                device_status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert np.array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
            assert np.array_equal(w.cpu().numpy(), ref_w.cpu().numpy())
            y = bf16_bits_to_f64(bf16_to_np(out))
            assert np.all(np.isfinite(y))
            assert rel_fro(y[valid], ref_y[valid]) <= TOL
            assert np.all(bf16_to_np(out)[~valid] == 0)


def test_noalloc_refuses_rows_beyond_the_array():
    cfg = m.Config.from_shape(synth.GLM52)
    lib = m.load()
    fake = 1 << 40                      # never dereferenced: the call is refused first
    wts = m.Weights(*([fake] * 12))
    st = lib.moe_layer_noalloc(C.byref(cfg), fake, fake, fake, C.byref(wts), None, 512, fake,
                               None, None, None, None)
    assert st == 2                      # MOE_ERR_UNSUPPORTED
    assert lib.moe_layer_noalloc(C.byref(cfg), None, None, None, C.byref(wts), None, 0, None,
                                 None, None, None, None) == 0
