"""The expert GEMM's run-time tile scheduler (a global tile counter claimed by
each CTA's producer, reset by the last CTA to finish claiming):

* after every GEMM launch -- gate/up alone, down alone, both fused -- the
  scheduler words in the workspace are back at zero, so the next launch on
  the workspace starts from tile 0;
* launches repeated on the same workspace without a dispatch in between (the
  counter then comes only from the previous launch's reset) give the same
  bits, and so do repeated fused launches: which CTA computes a tile never
  changes its result.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import synth
from gpu_helpers import MEDIUM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    torch.cuda.set_device(0)


def _setup(shape, R):
    wl = synth.Workload("sc", shape, rows=R, pads=(1,), seed=3)
    t = {k: v.cuda() for k, v in synth.make_layer(wl, device="cpu").items()}
    cfg = m.Config.from_shape(shape)
    dev = torch.device("cuda")
    K = shape.topk
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, shape.n_experts), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    return cfg, t, ub


def _sched_words(cfg, R, ws):
    off = m.ffn_layout(cfg, R)["sched"]
    return ws[off:off + 8].cpu().view(torch.int32).tolist()


@pytest.mark.parametrize("shape,R", [(synth.TINY, 8), (MEDIUM, 200), (synth.TINY, 600)])
def test_counter_reset_and_repeat(shape, R):
    cfg, t, ub = _setup(shape, R)
    H, K = shape.hidden, shape.topk
    W = m.Weights.from_tensors(t)
    ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device="cuda")
    ys = torch.zeros((R * K, H), dtype=torch.float32, device="cuda")
    ysh = torch.zeros((R, H), dtype=torch.float32, device="cuda")
    m.moe_dispatch(cfg, t["x"], ub, ws)
    m.moe_gate_up_fp8(cfg, W, ub, R, ws)
    torch.cuda.synchronize()
    assert _sched_words(cfg, R, ws) == [0, 0]
    outs = []
    for _ in range(3):   # down alone, repeated: no dispatch in between
        ys.zero_()
        ysh.zero_()
        m.moe_down_fp8(cfg, W, ub, R, ys, ysh, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        assert _sched_words(cfg, R, ws) == [0, 0]
        outs.append((ys.cpu().numpy().view(np.uint32).copy(), ysh.cpu().numpy().view(np.uint32).copy()))
    for _ in range(3):   # fused, each after its dispatch
        ys.zero_()
        ysh.zero_()
        m.moe_dispatch(cfg, t["x"], ub, ws)
        m.moe_expert_gemms_fp8(cfg, W, ub, R, ys, ysh, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        assert _sched_words(cfg, R, ws) == [0, 0]
        outs.append((ys.cpu().numpy().view(np.uint32).copy(), ysh.cpu().numpy().view(np.uint32).copy()))
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])
