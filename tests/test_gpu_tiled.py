"""The tiled weight layout (MOE_LAYOUT_TILED: every 128x128 block of a code
matrix stored as 16 KB of its own, row-block-major) on the GPU:

* moe_tile_weights is exactly the documented permutation of bytes (numpy
  reshape / transpose of the row-major codes), on shapes that span one block,
  ragged row-block and K-block counts, and more blocks than its grid (so the
  grid-stride loop wraps);
* the layer, the step-by-step GEMM entry points, the w8a16 variant and the
  no-allocation entry give the same bits with tiled weights as with row-major
  ones (only the addresses the GEMMs load from differ), and the tiled layer
  matches the oracle;
* a layout value other than 0 or 1 is refused.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import MEDIUM, TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def tiled_reference(codes: np.ndarray) -> np.ndarray:
    """The layout's definition: block (rb, kb) of matrix n at 16 KB slot
    (n * rows/128 + rb) * cols/128 + kb, its 128 rows of 128 bytes in order."""
    n, rows, cols = codes.shape
    b = codes.reshape(n, rows // 128, 128, cols // 128, 128).transpose(0, 1, 3, 2, 4)
    return np.ascontiguousarray(b).reshape(-1)


@pytest.mark.parametrize("shape", [(1, 128, 128), (3, 256, 384), (2, 640, 128), (3, 4096, 16384)])
def test_tile_weights_is_the_permutation(shape):
    g = torch.Generator().manual_seed(7)
    src = torch.randint(0, 256, shape, dtype=torch.uint8, generator=g)
    d_src = src.cuda()
    d_dst = torch.full(shape, 0xA5, dtype=torch.uint8, device="cuda")
    m.moe_tile_weights(d_src, d_dst)
    torch.cuda.synchronize()
    got = d_dst.cpu().numpy().reshape(-1)
    assert np.array_equal(got, tiled_reference(src.numpy()))
    assert torch.equal(d_src.cpu(), src)     # source untouched


def test_tile_weights_refusals():
    a = torch.zeros((2, 256, 256), dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    L = m.load()
    assert L.moe_tile_weights(a.data_ptr(), a.data_ptr() + 4096, 2, 256, 256, None) == 1  # overlap
    assert L.moe_tile_weights(a.data_ptr() + 8, b.data_ptr(), 1, 256, 256, None) == 1     # alignment
    assert L.moe_tile_weights(a.data_ptr(), b.data_ptr(), 2, 200, 256, None) == 1          # rows % 128
    assert L.moe_tile_weights(a.data_ptr(), b.data_ptr(), -1, 256, 256, None) == 1
    assert L.moe_tile_weights(a.data_ptr(), b.data_ptr(), 0, 256, 256, None) == 0


def _make(shape, rows, pads=(), seed=0):
    wl = synth.Workload("tl", shape, rows=rows, pads=tuple(pads), seed=seed)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    return wl, t, synth.to_numpy(t_cpu)


@pytest.mark.parametrize("shape,R,pads", [(synth.TINY, 8, ()), (MEDIUM, 37, (0, 36)),
                                          (MEDIUM, 200, (5,)), (synth.TINY, 600, (1, 599))])
def test_layer_tiled_bit_identical(shape, R, pads):
    wl, t, h = _make(shape, R, pads)
    cfg = m.Config.from_shape(shape)
    tt = m.tile_weights(t)
    for k in m.CODE_KEYS:
        if t[k].shape[-1] > 128:                       # one K-block per row: same bytes
            assert not torch.equal(tt[k], t[k])
    out0, ids0, w0, _ = run_layer(cfg, t, R)
    out1, ids1, w1, _ = run_layer(cfg, tt, R, layout=m.LAYOUT_TILED)
    assert np.array_equal(ids0.cpu().numpy(), ids1.cpu().numpy())
    assert np.array_equal(bf16_to_np(out0), bf16_to_np(out1))
    if R <= 37:
        ref = oracle.moe_layer(shape, h)
        y = bf16_bits_to_f64(bf16_to_np(out1))
        valid = h["row_valid"] != 0
        assert rel_fro(y[valid], ref["y_acc"][valid]) <= TOL


@pytest.mark.parametrize("shape,R", [(synth.TINY, 8), (MEDIUM, 200)])
def test_stepwise_gemms_tiled_bit_identical(shape, R):
    """Fused and two-launch GEMMs on tiled weights against the fused GEMM on
    row-major weights."""
    wl, t, h = _make(shape, R, pads=(1,))
    cfg = m.Config.from_shape(shape)
    dev = torch.device("cuda")
    K, H = shape.topk, shape.hidden
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, shape.n_experts), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    tt = m.tile_weights(t)
    outs = []
    for W, fused in ((m.Weights.from_tensors(t), True),
                     (m.Weights.from_tensors(tt, m.LAYOUT_TILED), True),
                     (m.Weights.from_tensors(tt, m.LAYOUT_TILED), False)):
        ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
        ys = torch.zeros((R * K, H), dtype=torch.float32, device=dev)
        ysh = torch.zeros((R, H), dtype=torch.float32, device=dev)
        m.moe_dispatch(cfg, t["x"], ub, ws)
        if fused:
            m.moe_expert_gemms_fp8(cfg, W, ub, R, ys, ysh, ws)
        else:
            m.moe_gate_up_fp8(cfg, W, ub, R, ws)
            m.moe_down_fp8(cfg, W, ub, R, ys, ysh, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        outs.append((ys.cpu().numpy().view(np.uint32), ysh.cpu().numpy().view(np.uint32)))
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])


@pytest.mark.parametrize("shape,R,pads", [(MEDIUM, 8, (3,)), (MEDIUM, 64, (7, 23, 39, 55))])
def test_w8a16_tiled_bit_identical(shape, R, pads):
    wl, t, h = _make(shape, R, pads)
    cfg = m.Config.from_shape(shape)
    tt = m.tile_weights(t)
    outs = []
    for d, layout in ((t, m.LAYOUT_ROW_MAJOR), (tt, m.LAYOUT_TILED)):
        ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
        out = torch.full((R, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.moe_layer_w8a16(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(d, layout),
                          t["row_valid"], out, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        outs.append(bf16_to_np(out))
    assert np.array_equal(outs[0], outs[1])
    ref = oracle.moe_layer(shape, h, variant="w8a16")
    y = bf16_bits_to_f64(outs[1])
    valid = h["row_valid"] != 0
    assert rel_fro(y[valid], ref["y_acc"][valid]) <= TOL


def test_noalloc_tiled_bit_identical():
    shape, R = MEDIUM, 24
    wl, t, h = _make(shape, R, pads=(2,))
    cfg = m.Config.from_shape(shape)
    tt = m.tile_weights(t)
    out0, _, _, _ = run_layer(cfg, tt, R, layout=m.LAYOUT_TILED)
    out1 = torch.full((R, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.moe_layer_noalloc(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(tt, m.LAYOUT_TILED),
                        t["row_valid"], out1)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_np(out0), bf16_to_np(out1))


def test_bad_layout_refused():
    shape, R = synth.TINY, 4
    wl, t, h = _make(shape, R)
    cfg = m.Config.from_shape(shape)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    out = torch.empty((R, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoeError):
        m.moe_layer(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t, 2), None, out, ws)
