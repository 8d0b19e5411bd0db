"""The large-row router logits kernel against the oracle, bit for bit.

Above 64 rows moe_route's logits come from a persistent kernel that takes
tiles of 24, 28, 32 or 36 rows (whichever finishes sooner) x 32 experts,
streams x and the router weights through
shared memory in stages of two 128-column blocks, keeps each 1024-column
chunk's lane sums in tensor memory and ends each pair's reduction tree by
recursive halving.  Its logits must be the header's fixed-order IEEE sums,
i.e. the oracle's bits, at every edge of that structure:

* row counts with a ragged last row tile (65, 100, 333) and the maximum, 4096;
  every tile height, each at the first row count that takes it at 256
  experts (456 rows: 24-row tiles, 457: 28, 533: 32, 609: 36, and 685 back to
  24 in two waves) -- the odd heights end each pair's reduction without the
  last halving;
* expert counts that leave a partial expert tile (48, 72 of 32) or a single
  one (16);
* hidden sizes whose 128-column block count is odd (a stage's second half
  past the end: 384, 1152, 6272) or fits one chunk (no chunk sums kept:
  384, 1024), and the GLM-5.2 width 6144 (six chunks);
* pad rows anywhere (their logits stay untouched: a sentinel survives);
* 16 seeded shapes (48 to 256 experts, hidden 384 to 6144, random groups and
  top-k) at 400 to 2200 rows, which between them take every tile height.

ids and weights are compared bit for bit too (the selection reads the
logits).
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth

pytestmark = pytest.mark.gpu

SENTINEL = np.float32(-12345.5)


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def _shape(H, E, G, TG, K):
    return synth.LayerShape(hidden=H, inter=128, n_experts=E, n_groups=G, topk_groups=TG,
                            topk=K, n_shared=1, routed_scaling=2.5)


def _route(shape, R, pads, seed):
    wl = synth.Workload("router", shape, rows=R, pads=tuple(pads), seed=seed)
    ri = synth.make_router_inputs(wl, device="cpu")
    E, K = shape.n_experts, shape.topk
    cfg = m.Config.from_shape(shape)
    ids = torch.empty((R, K), dtype=torch.int32, device="cuda")
    w = torch.empty((R, K), dtype=torch.float32, device="cuda")
    lg = torch.full((R, E), float(SENTINEL), dtype=torch.float32, device="cuda")
    m.moe_route(cfg, ri["x"].cuda(), ri["wr"].cuda(), ri["bias"].cuda(),
                ri["row_valid"].cuda(), ids, w, lg)
    torch.cuda.synchronize()
    h = synth.to_numpy(ri)
    return h, ids.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()


def _check(shape, R, pads, seed, rows=None):
    h, ids, w, lg = _route(shape, R, pads, seed)
    valid = h["row_valid"] != 0
    assert np.all(lg[~valid] == SENTINEL)
    sel = np.arange(R) if rows is None else np.asarray(rows)
    sel = sel[valid[sel]]
    ref_ids, ref_w, ref_lg = oracle.route(shape, h["x"][sel], h["wr"], h["bias"])
    assert np.array_equal(lg[sel].view(np.uint32), ref_lg.view(np.uint32))
    assert np.array_equal(ids[sel], ref_ids)
    assert np.array_equal(w[sel].view(np.uint32), ref_w.view(np.uint32))
    assert np.all(ids[~valid] == -1) and np.all(w[~valid] == 0)


@pytest.mark.parametrize("R,pads", [(65, (64,)), (100, (0, 37, 99)), (333, (200,))])
@pytest.mark.parametrize("H", [384, 1024, 1152, 6272])
def test_ragged_rows_and_odd_blocks(R, pads, H):
    _check(_shape(H, 48, 4, 2, 6), R, pads, seed=R + H)


@pytest.mark.parametrize("E,G,TG,K", [(16, 2, 1, 4), (72, 8, 4, 8), (256, 8, 4, 8)])
def test_expert_tiles(E, G, TG, K):
    _check(_shape(1152, E, G, TG, K), 97, (3, 50), seed=E)


@pytest.mark.parametrize("R,rt", [(456, 6), (457, 7), (533, 8), (609, 9), (685, 6)])
def test_tile_height_switch(R, rt):
    assert m.router_rows_per_warp(R, 256) == rt
    rows = np.unique(np.r_[np.arange(0, 30), np.arange(R - 30, R), np.arange(0, R, 23)])
    _check(_shape(6144, 256, 8, 4, 8), R, (0, R // 2, R - 1), seed=R, rows=rows)


def test_full_size_sampled_rows():
    # 4096 rows at the GLM-5.2 router shape: every pad and a sample of rows
    R = 4096
    rows = np.unique(np.r_[np.arange(0, 40), np.arange(R - 40, R), np.arange(0, R, 97)])
    _check(_shape(6144, 256, 8, 4, 8), R, (1, 2047, 4095), seed=5, rows=rows)


def _draw_router(seed):
    """A seeded router shape and row count between 400 and 2200 rows, where
    every tile height occurs at one expert count or another."""
    rng = np.random.default_rng(5000 + seed)
    E = int(rng.choice([48, 64, 96, 128, 160, 256]))
    H = 128 * int(rng.choice([3, 9, 16, 48]))
    R = int(rng.integers(400, 2200))
    groups = [g for g in (1, 2, 4, 8, 16, 32) if E % g == 0 and E // g <= 32]
    G = int(rng.choice(groups))
    TG = int(rng.integers(1, G + 1))
    K = int(rng.integers(1, min(16, TG * (E // G)) + 1))
    pads = tuple(sorted(int(p) for p in rng.choice(R, size=3, replace=False)))
    return _shape(H, E, G, TG, K), R, pads


N_ROUTER_CASES = 16


def test_random_cases_cover_every_tile_height():
    heights = {m.router_rows_per_warp(R, s.n_experts)
               for s, R, _ in (_draw_router(i) for i in range(N_ROUTER_CASES))}
    assert heights == {6, 7, 8, 9}


@pytest.mark.parametrize("seed", range(N_ROUTER_CASES))
def test_random_router_shapes(seed):
    shape, R, pads = _draw_router(seed)
    rows = np.unique(np.r_[np.arange(0, 12), np.arange(R - 12, R), np.arange(0, R, 37), list(pads)])
    _check(shape, R, pads, seed=seed, rows=rows)
