"""Degenerate batches through the whole layer on the GPU.

* Every row a pad row, at 8 rows (selection + union in one block, one fused
  GEMM launch), 37 rows (16-row tiles) and 100 rows (separate selection and
  union kernels, the gate/up and down GEMM launches): the union is empty, no
  GEMM tile exists, and the layer must still return +0.0 rows, ids -1, weights
  0 and a clean device status -- also through the w8a16 layer.
* One valid row among pads (a union of a single row): parity with the oracle.
* All-pad, normal and all-pad calls in a row on one workspace: the GEMMs' tile
  scheduler words, reset by the last CTA of each launch, leave the following
  call unaffected (its outputs match a fresh workspace's bit for bit).
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


def _layer(shape, R, pads, seed=3):
    wl = synth.Workload("edge", shape, rows=R, pads=tuple(pads), seed=seed)
    t_cpu = synth.make_layer(wl, device="cpu")
    return t_cpu, {k: v.cuda() for k, v in t_cpu.items()}


@pytest.mark.parametrize("shape,R", [(synth.TINY, 8), (MEDIUM, 37), (MEDIUM, 100)])
def test_all_rows_pad(shape, R):
    _, t = _layer(shape, R, range(R))
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    assert np.all(bf16_to_np(out) == 0)
    assert np.all(ids.cpu().numpy() == -1)
    assert np.all(w.cpu().numpy().view(np.uint32) == 0)


def test_all_rows_pad_w8a16():
    shape, R = synth.TINY, 8
    _, t = _layer(shape, R, range(R))
    cfg = m.Config.from_shape(shape)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    out = torch.full((R, shape.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((R, shape.topk), dtype=torch.int32, device="cuda")
    w = torch.empty((R, shape.topk), dtype=torch.float32, device="cuda")
    m.moe_layer_w8a16(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t),
                      t["row_valid"], out, ws, topk_ids=ids, topk_w=w)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    assert np.all(bf16_to_np(out) == 0)
    assert np.all(ids.cpu().numpy() == -1)


@pytest.mark.parametrize("R,keep", [(8, 5), (100, 0), (100, 99)])
def test_single_valid_row(R, keep):
    shape = MEDIUM
    t_cpu, t = _layer(shape, R, [r for r in range(R) if r != keep], seed=R + keep)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    h = synth.to_numpy(t_cpu)
    ref = oracle.moe_layer(shape, h)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["wts"].view(np.uint32))
    y = bf16_bits_to_f64(bf16_to_np(out))
    assert rel_fro(y[keep], ref["y_acc"][keep]) <= TOL
    pads = np.arange(R) != keep
    assert np.all(bf16_to_np(out)[pads] == 0)


@pytest.mark.parametrize("R", [8, 100])
def test_pad_calls_leave_workspace_clean(R):
    shape = MEDIUM
    cfg = m.Config.from_shape(shape)
    _, t_pad = _layer(shape, R, range(R), seed=1)
    _, t = _layer(shape, R, (R - 1,), seed=2)
    fresh, _, _, _ = run_layer(cfg, t, R)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    for tt in (t_pad, t, t_pad, t):
        out, _, _, _ = run_layer(cfg, tt, R, ws=ws)
        if tt is t:
            assert np.array_equal(bf16_to_np(out), bf16_to_np(fresh))
        else:
            assert np.all(bf16_to_np(out) == 0)


@pytest.mark.parametrize("R", [8, 100])
def test_alternating_buffers_reuse_no_stale_maps(R):
    """The library keeps the tensor maps of recent calls per thread, keyed by
    the buffers they describe.  Calls that alternate between two workspaces,
    two copies of the weights (one zeroed: its maps must not be reused for
    the other) and two row counts give each call's own bits."""
    shape = MEDIUM
    cfg = m.Config.from_shape(shape)
    t_cpu, t = _layer(shape, R, (0,), seed=R)
    W1 = m.Weights.from_tensors(t)
    t2 = {k: v.clone() for k, v in t.items()}
    for k in ("w_gate", "w_up", "w_down"):
        t2[k].zero_()
    W2 = m.Weights.from_tensors(t2)
    ws_a = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    ws_b = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")

    def call(W, ws, rows=R):
        out = torch.full((rows, shape.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.moe_layer(cfg, t["x"][:rows], t["wr"], t["bias"], W, t["row_valid"][:rows], out, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        return bf16_to_np(out)

    ref1, ref2 = call(W1, ws_a), call(W2, ws_b)
    assert not np.array_equal(ref1, ref2)
    for W, ws, ref in ((W1, ws_b, ref1), (W2, ws_a, ref2), (W1, ws_a, ref1), (W2, ws_b, ref2)):
        assert np.array_equal(call(W, ws), ref)
    # a smaller call on the same workspace, then the full one again
    small = call(W1, ws_a, rows=R // 2)
    assert np.array_equal(small, ref1[: R // 2])
    assert np.array_equal(call(W1, ws_a), ref1)


def test_two_host_threads_two_shapes():
    """Two host threads, each on its own stream, call moe_layer on shapes whose
    expert GEMM needs different amounts of shared memory (the kernel attribute
    that allows it is process-wide and only ever raised): every call keeps its
    single-threaded bits and a clean status."""
    import threading
    cases = []
    for shape, R, seed in ((synth.TINY, 8, 11), (MEDIUM, 8, 12)):
        t_cpu, t = _layer(shape, R, (), seed=seed)
        cfg = m.Config.from_shape(shape)
        ref, _, _, _ = run_layer(cfg, t, R)
        cases.append((shape, R, cfg, t, bf16_to_np(ref)))
    errors = []

    def worker(case):
        shape, R, cfg, t, ref = case
        try:
            stream = torch.cuda.Stream()
            ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
            W = m.Weights.from_tensors(t)
            for _ in range(10):
                out = torch.full((R, shape.hidden), float("nan"), dtype=torch.bfloat16,
                                 device="cuda")
                with torch.cuda.stream(stream):
                    m.moe_layer(cfg, t["x"], t["wr"], t["bias"], W, t["row_valid"], out, ws,
                                stream=stream)
                stream.synchronize()
                if (m.moe_get_device_error(ws, stream=stream) != 0
                        or not np.array_equal(bf16_to_np(out), ref)):
                    errors.append(shape)
                    return
        except Exception as e:      # reported below, in the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(c,)) for c in cases]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
