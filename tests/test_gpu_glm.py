"""GPU parity at the full GLM-5.2-class layer shape (hidden 6144, inter 2048,
256 experts in 8 groups, top-4 groups, top-8, one shared expert) on the four
workload mixes, in the launch configuration the bench times:

* verify8     -- 8 rows (1 committed + 7 drafts), skewed router, ~40 experts;
* verify64    -- 64 rows (8 requests x span 8), pad rows 7, 23, 39, 55 (x = NaN);
* decode512   -- 512 rows, Zipf(1.1) expert popularity;
* prefill4096 -- 4096 rows (the compiled maximum), uniform routing.

Routing ids and weights are compared bit-exact on every row; the layer output
on sampled rows (the oracle computes rows independently) within 1e-2
relative Frobenius norm; pad rows must be +0.0.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def weights():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS["verify8"]
    dev = synth.make_expert_weights(wl, device="cuda")
    host = {k: v.cpu().numpy() for k, v in dev.items()}
    yield dev, host
    del dev
    torch.cuda.empty_cache()


SAMPLES = {
    "verify8": list(range(8)),
    "verify64": [0, 7, 22, 23, 40, 63],
    "decode512": [0, 137, 301, 511],
    "prefill4096": [0, 1023, 2900, 4095],
}


@pytest.mark.parametrize("name", ["verify8", "verify64", "decode512", "prefill4096"])
def test_glm_workload(weights, name):
    dev_w, host_w = weights
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    ri = synth.make_router_inputs(wl, device="cuda")
    t = dict(ri)
    t.update(dev_w)
    cfg = m.Config.from_shape(shape)
    R = wl.rows
    out, ids, w, _ = run_layer(cfg, t, R)
    h = synth.to_numpy(ri)
    h.update(host_w)
    ref_ids, ref_w, _ = oracle.route(shape, h["x"], h["wr"], h["bias"], h["row_valid"])
    gid = ids.cpu().numpy()
    assert np.array_equal(gid, ref_ids)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    rows = SAMPLES[name]
    ref = oracle.moe_layer(shape, h, rows=rows)
    ob = bf16_to_np(out)
    y = bf16_bits_to_f64(ob)
    valid = h["row_valid"] != 0
    vr = [r for r in rows if valid[r]]
    assert rel_fro(y[vr], ref["y_acc"][vr]) <= TOL
    for r in vr:
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL
    assert np.all(ob[~valid] == 0)
    assert np.all(np.isfinite(y))
    if name == "verify8":
        U = len(np.unique(gid))
        assert 30 <= U <= 48, U


@pytest.mark.parametrize("name", ["verify8", "prefill4096"])
def test_glm_tiled_layout_bit_identical(weights, name):
    """The layout the bench gives the layer -- weight codes in 16 KB 128x128
    blocks (moe_tile_weights) -- gives the same output bits as the row-major
    codes at the full shape, on the verify and the prefill row tile."""
    dev_w, _ = weights
    wl = synth.WORKLOADS[name]
    t = dict(synth.make_router_inputs(wl, device="cuda"))
    t.update(dev_w)
    cfg = m.Config.from_shape(wl.shape)
    out_rm, ids_rm, w_rm, _ = run_layer(cfg, t, wl.rows)
    tt = m.tile_weights(t)
    out_t, ids_t, w_t, _ = run_layer(cfg, tt, wl.rows, layout=m.LAYOUT_TILED)
    assert torch.equal(ids_t, ids_rm)
    assert torch.equal(w_t, w_rm)
    assert torch.equal(out_t.view(torch.int16), out_rm.view(torch.int16))
    del tt
    torch.cuda.empty_cache()
