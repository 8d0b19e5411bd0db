"""GPU parity of the w8a16 variant (bf16 activations, e4m3 weights dequantised
to bf16 inside the GEMM kernel, bf16 tensor-core MMA) against the oracle's
w8a16 layer:

* routing ids and weights bit-exact (the routing is the fp8 path's);
* layer output within 1e-2 relative Frobenius norm of the oracle's w8a16 layer
  on every valid row, pad rows +0.0 (x = NaN there);
* the per-slot expert outputs of moe_expert_ffn_w8a16 against the oracle's
  expert, one by one;
* the variant's point: against the layer without any activation or weight
  rounding its error is far below the fp8 path's;
* the GLM-5.2 shape at 1, 4 and 8 rows (the verify span) on every row;
* refusals: more than 64 rows, and R = 0 is a no-op.
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


def _make(shape, rows, pads=(), seed=0, routing="uniform"):
    wl = synth.Workload("w16", shape, rows=rows, pads=tuple(pads), seed=seed, routing=routing)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    return wl, t, synth.to_numpy(t_cpu)


def run_w8a16(cfg, t, R):
    dev = t["x"].device
    ws = torch.zeros(m.moe_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    out = torch.full((R, cfg.hidden), float("nan"), dtype=torch.bfloat16, device=dev)
    ids = torch.empty((R, cfg.topk), dtype=torch.int32, device=dev)
    w = torch.empty((R, cfg.topk), dtype=torch.float32, device=dev)
    m.moe_layer_w8a16(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t),
                      t.get("row_valid"), out, ws, topk_ids=ids, topk_w=w)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    return out, ids, w


@pytest.mark.parametrize("shape,R,pads", [(synth.TINY, 8, ()), (MEDIUM, 8, (3,)),
                                          (MEDIUM, 37, (0, 36)), (MEDIUM, 64, (7, 23, 39, 55)),
                                          (MEDIUM, 1, ())])
def test_layer_w8a16_matches_oracle(shape, R, pads):
    wl, t, h = _make(shape, R, pads)
    cfg = m.Config.from_shape(shape)
    out, ids, w = run_w8a16(cfg, t, R)
    ref = oracle.moe_layer(shape, h, variant="w8a16")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["wts"].view(np.uint32))
    ob = bf16_to_np(out)
    y = bf16_bits_to_f64(ob)
    valid = h["row_valid"] != 0
    assert np.all(np.isfinite(y))
    assert rel_fro(y[valid], ref["y_acc"][valid]) <= TOL
    for r in np.nonzero(valid)[0]:
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL
    assert np.all(ob[~valid] == 0)


def test_expert_ffn_w8a16_slots():
    shape, R = MEDIUM, 12
    wl, t, h = _make(shape, R, pads=(4,))
    cfg = m.Config.from_shape(shape)
    K, H, E = shape.topk, shape.hidden, shape.n_experts
    dev = torch.device("cuda")
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, E), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    ys = torch.full((R * K, H), float("nan"), dtype=torch.float32, device=dev)
    ysh = torch.full((R, H), float("nan"), dtype=torch.float32, device=dev)
    m.moe_expert_ffn_w8a16(cfg, t["x"], m.Weights.from_tensors(t), ub, ys, ysh, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    gids = ids.cpu().numpy()
    ys = ys.cpu().numpy().reshape(R, K, H)
    ysh = ysh.cpu().numpy()
    valid = h["row_valid"] != 0
    for r in np.nonzero(valid)[0]:
        for k in range(K + 1):
            if k < K:
                e = gids[r, k]
                args = (h["w_gate"][e], h["s_gate"][e], h["w_up"][e], h["s_up"][e],
                        h["w_down"][e], h["s_down"][e])
                got = ys[r, k]
            else:
                args = (h["sh_gate"][0], h["sh_s_gate"][0], h["sh_up"][0], h["sh_s_up"][0],
                        h["sh_down"][0], h["sh_s_down"][0])
                got = ysh[r]
            ref = oracle.expert_ffn_a16(shape, h["x"][r], *args, round16=True)
            assert rel_fro(got, ref) <= TOL
    assert np.all(np.isnan(ys[~valid])) and np.all(np.isnan(ysh[~valid]))


def test_w8a16_error_below_fp8_on_gpu():
    shape, R = MEDIUM, 16
    wl, t, h = _make(shape, R)
    cfg = m.Config.from_shape(shape)
    out16, _, _ = run_w8a16(cfg, t, R)
    out8, _, _, _ = run_layer(cfg, t, R)
    ex = oracle.moe_layer(shape, h, variant="exact")["y_acc"]
    e16 = rel_fro(bf16_bits_to_f64(bf16_to_np(out16)), ex)
    e8 = rel_fro(bf16_bits_to_f64(bf16_to_np(out8)), ex)
    assert e16 * 4 < e8, (e16, e8)


@pytest.mark.parametrize("R", [1, 4, 8])
def test_glm_shape_w8a16(R):
    base = synth.WORKLOADS["verify8"]
    wl = synth.Workload("w16glm", base.shape, rows=R, routing=base.routing,
                        hot_per_group=base.hot_per_group, hot_delta=base.hot_delta)
    dev_w = synth.make_expert_weights(base, device="cuda")
    ri = synth.make_router_inputs(wl, device="cuda")
    t = dict(ri)
    t.update(dev_w)
    cfg = m.Config.from_shape(wl.shape)
    out, ids, w = run_w8a16(cfg, t, R)
    h = synth.to_numpy(ri)
    h.update({k: v.cpu().numpy() for k, v in dev_w.items()})
    ref = oracle.moe_layer(wl.shape, h, variant="w8a16")
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    y = bf16_bits_to_f64(bf16_to_np(out))
    for r in range(R):
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL
    del dev_w
    torch.cuda.empty_cache()


def test_w8a16_limits():
    shape = MEDIUM
    cfg = m.Config.from_shape(shape)
    wl, t, h = _make(shape, 65)
    ws = torch.zeros(m.moe_workspace_bytes(cfg, 65), dtype=torch.uint8, device="cuda")
    out = torch.empty((65, shape.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoeError):
        m.moe_layer_w8a16(cfg, t["x"], t["wr"], t["bias"], m.Weights.from_tensors(t), None, out, ws)
    x0 = t["x"][:0]
    m.moe_layer_w8a16(cfg, x0, t["wr"], t["bias"], m.Weights.from_tensors(t), None, out[:0], ws)
    torch.cuda.synchronize()
