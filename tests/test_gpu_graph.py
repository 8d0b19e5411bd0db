"""One captured CUDA graph serves any occupancy of the 8-row block.

openinfer #610 "TP8 span row mapping ...", commit on the span owner: the owner
moves from a launch parameter (baked at capture) to device memory read at
kernel time, so ONE captured graph serves any request.  Here the layer reads
its rows, their validity and every weight from device memory at kernel time;
the row count fixes the launch shapes.  A graph captured once at R = 8 and
replayed with other inputs and other pad patterns gives the same bits as
eager calls with those inputs (kernels chained by programmatic dependent
launch inside the graph), and every replay matches the oracle on those
inputs: routing ids and weights bit for bit, the output within the parity
tolerance, pad rows +0.0.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import MEDIUM, TOL, bf16_bits_to_f64, bf16_to_np, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def test_one_graph_any_occupancy():
    shape, R = MEDIUM, 8
    wl = synth.Workload("graph", shape, rows=R)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    host = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(shape)
    W = m.Weights.from_tensors(t)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    x = t["x"].clone()
    valid = torch.ones(R, dtype=torch.uint8, device="cuda")
    out = torch.empty((R, shape.hidden), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((R, shape.topk), dtype=torch.int32, device="cuda")
    wts = torch.empty((R, shape.topk), dtype=torch.float32, device="cuda")

    def layer():
        m.moe_layer(cfg, x, t["wr"], t["bias"], W, valid, out, ws, topk_ids=ids, topk_w=wts)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer()                                  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer()

    rng = np.random.default_rng(40)
    cases = [np.ones(R, np.uint8), np.array([1, 1, 1, 0, 0, 0, 0, 0], np.uint8),
             np.array([1, 0, 1, 0, 1, 0, 1, 0], np.uint8), np.zeros(R, np.uint8)]
    for vmask in cases:
        xv = torch.from_numpy(rng.normal(0, 1, (R, shape.hidden)).astype(np.float32))
        xv = xv.to(torch.bfloat16).cuda()
        xv[torch.from_numpy(vmask == 0).cuda()] = float("nan")   # pads may hold NaN
        x.copy_(xv)
        valid.copy_(torch.from_numpy(vmask))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = bf16_to_np(out).copy()
        got_ids = ids.cpu().numpy().copy()
        got_w = wts.cpu().numpy().copy()
        # the replay against the oracle on the inputs it read at kernel time
        h = dict(host)
        h["x"] = synth.to_numpy({"x": xv})["x"]
        h["row_valid"] = vmask
        ref = oracle.moe_layer(shape, h)
        assert np.array_equal(got_ids, ref["ids"])
        assert np.array_equal(got_w.view(np.uint32), ref["wts"].view(np.uint32))
        v = vmask != 0
        if v.any():
            y = bf16_bits_to_f64(got)
            assert np.all(np.isfinite(y))
            assert rel_fro(y[v], ref["y_acc"][v]) <= TOL
        out.fill_(float("nan"))
        layer()                                  # eager, same inputs
        torch.cuda.synchronize()
        assert np.array_equal(got, bf16_to_np(out))
        assert np.array_equal(got_ids, ids.cpu().numpy())
        assert np.all(got[vmask == 0] == 0)
        assert m.moe_get_device_error(ws) == 0


def test_one_graph_any_occupancy_two_gemm_launches():
    """The same at 100 rows, where the layer runs the selection and the union
    as two kernels and the expert GEMMs as a gate/up and a down launch."""
    shape, R = MEDIUM, 100
    wl = synth.Workload("graph100", shape, rows=R)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    host = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(shape)
    W = m.Weights.from_tensors(t)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    x = t["x"].clone()
    valid = torch.ones(R, dtype=torch.uint8, device="cuda")
    out = torch.empty((R, shape.hidden), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((R, shape.topk), dtype=torch.int32, device="cuda")

    def layer():
        m.moe_layer(cfg, x, t["wr"], t["bias"], W, valid, out, ws, topk_ids=ids)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer()
    rng = np.random.default_rng(41)
    for vmask in (np.ones(R, np.uint8), (rng.random(R) < 0.7).astype(np.uint8)):
        xv = torch.from_numpy(rng.normal(0, 1, (R, shape.hidden)).astype(np.float32))
        xv = xv.to(torch.bfloat16).cuda()
        xv[torch.from_numpy(vmask == 0).cuda()] = float("nan")
        x.copy_(xv)
        valid.copy_(torch.from_numpy(vmask))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        got = bf16_to_np(out).copy()
        h = dict(host)
        h["x"] = synth.to_numpy({"x": xv})["x"]
        h["row_valid"] = vmask
        rows = np.unique(np.linspace(0, R - 1, 16).astype(int))
        ref = oracle.moe_layer(shape, h, rows=rows)
        ref_ids, _, _ = oracle.route(shape, h["x"], h["wr"], h["bias"], vmask)
        assert np.array_equal(ids.cpu().numpy(), ref_ids)
        v = vmask != 0
        vr = [r for r in rows if v[r]]
        y = bf16_bits_to_f64(got)
        assert rel_fro(y[vr], ref["y_acc"][vr]) <= TOL
        assert np.all(got[~v] == 0)
