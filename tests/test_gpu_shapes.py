"""GPU parity on layer shapes away from the GLM-5.2 defaults, against the
oracle: routing ids and weights bit-exact, outputs within 1e-2 relative
Frobenius norm on every valid row, pad rows +0.0.

* top-16 of 64 experts (the compiled top-k maximum: combine and union arrays
  at full length);
* 32 groups of 8 experts (the compiled group maximum: one lane per group in
  the selection);
* hidden 384 and intermediate 640 (3 and 5 K-blocks: the scalar scale-table
  path, a router chunk shorter than 1024 columns);
* each at 16- and 32-row tiles of the expert GEMM, with tiled weight codes
  giving the same bits as row-major ones;
* a DeepSeek-V3-style layer (hidden 7168, 56 K-blocks and 56 output blocks;
  intermediate 2048; 256 experts in 8 groups, top-4 groups, top-8, one shared
  expert) at 8 rows and at 100 rows (the large-R router and the two GEMM
  launches), on sampled rows.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu

SHAPES = {
    "top16": synth.LayerShape(hidden=512, inter=256, n_experts=64, n_groups=8, topk_groups=4,
                              topk=16, n_shared=1, routed_scaling=2.5),
    "groups32": synth.LayerShape(hidden=256, inter=128, n_experts=256, n_groups=32,
                                 topk_groups=8, topk=8, n_shared=1, routed_scaling=1.0),
    "odd_blocks": synth.LayerShape(hidden=384, inter=640, n_experts=16, n_groups=4,
                                   topk_groups=2, topk=4, n_shared=1, routed_scaling=2.5),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("R,pads", [(11, (4,)), (90, (0, 89))])
def test_shape_against_oracle(name, R, pads):
    shape = SHAPES[name]
    wl = synth.Workload(f"shape_{name}", shape, rows=R, pads=tuple(pads), seed=11)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    h = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    ref = oracle.moe_layer(shape, h)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["wts"].view(np.uint32))
    ob = bf16_to_np(out)
    y = bf16_bits_to_f64(ob)
    valid = h["row_valid"] != 0
    assert np.all(np.isfinite(y))
    for r in np.nonzero(valid)[0]:
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL
    assert np.all(ob[~valid] == 0)
    tt = m.tile_weights(t)
    out2, _, _, _ = run_layer(cfg, tt, R, layout=m.LAYOUT_TILED)
    assert np.array_equal(ob, bf16_to_np(out2))


DSV3 = synth.LayerShape(hidden=7168, inter=2048, n_experts=256, n_groups=8, topk_groups=4,
                        topk=8, n_shared=1, routed_scaling=2.5)


@pytest.fixture(scope="module")
def dsv3_layer():
    # 256 experts of 44 MB: generated once, on the device, for both cases
    wl = synth.Workload("shape_dsv3", DSV3, rows=100, pads=(0, 57), seed=23)
    t = dict(synth.make_router_inputs(wl, device="cuda"))
    t.update(synth.make_expert_weights(wl, device="cuda"))
    t_cpu = {k: v.cpu() for k, v in t.items()}
    yield t_cpu, t
    del t
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R,rows", [(8, None), (100, (1, 2, 33, 58, 77, 99))])
def test_dsv3_shape_against_oracle(dsv3_layer, R, rows):
    t_cpu_all, t_all = dsv3_layer
    per_row = ("x", "row_valid")
    t = {k: (v[:R].contiguous() if k in per_row else v) for k, v in t_all.items()}
    t_cpu = {k: (v[:R].contiguous() if k in per_row else v) for k, v in t_cpu_all.items()}
    h = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(DSV3)
    out, ids, w, _ = run_layer(cfg, t, R)
    ref = oracle.moe_layer(DSV3, h, rows=rows)
    valid = h["row_valid"] != 0
    check = np.nonzero(valid)[0] if rows is None else np.array(rows)
    ids_np, w_np = ids.cpu().numpy(), w.cpu().numpy()
    assert np.array_equal(ids_np[check], ref["ids"][check])
    assert np.array_equal(w_np[check].view(np.uint32), ref["wts"][check].view(np.uint32))
    ob = bf16_to_np(out)
    y = bf16_bits_to_f64(ob)
    for r in check:
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL, r
    assert np.all(ob[~valid] == 0)
    assert np.all(np.isfinite(y[valid]))
