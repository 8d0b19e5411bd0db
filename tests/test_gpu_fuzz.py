"""Seeded random layer shapes through the whole layer, against the oracle.

Each case draws a layer shape within the library's limits -- experts, groups,
kept groups and top-k; hidden and intermediate sizes (multiples of 128, odd
block counts included); with or without the shared expert -- and a row count
on either side of the kernels' switches (64 rows: selection + union in one
block and one fused GEMM; 65-256: 32-row tiles; above: 64-row tiles and the
TMA router), with pad rows anywhere.  Routing ids and weights must be
bit-exact, every valid row within the parity tolerance and every pad row +0.0.
The seeds are fixed, so a failure names a case that reproduces.
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([16, 24, 32, 48, 64, 96, 128, 256]))
    groups = [g for g in (1, 2, 4, 8, 16, 32) if E % g == 0 and E // g <= 32]
    G = int(rng.choice(groups))
    TG = int(rng.integers(1, G + 1))
    K = int(rng.integers(1, min(16, TG * (E // G)) + 1))
    H = 128 * int(rng.choice([2, 3, 5, 8, 9]))
    inter = 128 * int(rng.choice([1, 2, 3, 5]))
    S = int(rng.integers(0, 2))
    R = int(rng.choice([1, 5, 8, 37, 64, 65, 100, 257, 333]))
    shape = synth.LayerShape(hidden=H, inter=inter, n_experts=E, n_groups=G, topk_groups=TG,
                             topk=K, n_shared=S, routed_scaling=float(rng.choice([1.0, 2.5])))
    n_pad = int(rng.integers(0, max(1, R // 4) + 1)) if R > 1 else 0
    pads = tuple(sorted(int(p) for p in rng.choice(R, size=n_pad, replace=False)))
    return shape, R, pads


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shape_against_oracle(seed):
    shape, R, pads = _draw(seed)
    wl = synth.Workload(f"fuzz{seed}", shape, rows=R, pads=pads, seed=seed)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    h = synth.to_numpy(t_cpu)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    ref = oracle.moe_layer(shape, h)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"]), (shape, R, pads)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["wts"].view(np.uint32))
    ob = bf16_to_np(out)
    y = bf16_bits_to_f64(ob)
    valid = h["row_valid"] != 0
    assert np.all(np.isfinite(y[valid]))
    for r in np.nonzero(valid)[0]:
        assert rel_fro(y[r], ref["y_acc"][r]) <= TOL, (shape, R, r)
    assert np.all(ob[~valid] == 0)
