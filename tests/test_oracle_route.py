"""Pins of the oracle's router: logits, grouped top-k, weights, pads.

* logits: within the fp32 rounding bound of an fp64 dot product;
* selection: equal to a library sort (Python sorted) of the pinned scores,
  and to exhaustive enumeration of group subsets / expert subsets;
* ties: hand-derived cases (tests/golden/route_ties.txt), lowest id wins;
* weights: sum to routed_scaling, proportional to the unbiased sigmoid;
* pads: ids -1, weights 0, whatever their x holds.
"""
import itertools
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_ties.txt")


def _shape(**kw):
    base = dict(hidden=256, inter=128, n_experts=16, n_groups=4, topk_groups=2, topk=4,
                n_shared=1, routed_scaling=2.5)
    base.update(kw)
    return synth.LayerShape(**base)


def test_logits_within_fp32_bound(orc):
    wl = synth.WORKLOADS["tiny"]
    for H in (256, 1024, 1152, 6144):
        sh = _shape(hidden=H)
        ri = synth.to_numpy(synth.make_router_inputs(synth.variant(wl, shape=sh, rows=5)))
        lg = orc.router_logits(sh, ri["x"], ri["wr"])
        xf = orc.bf16_to_f32(ri["x"]).astype(np.float64)
        wr = ri["wr"].astype(np.float64)
        exact = xf @ wr.T
        mag = np.abs(xf) @ np.abs(wr).T
        u = 2.0 ** -24
        n = H
        bound = (n * u / (1 - n * u)) * mag
        assert np.all(np.abs(lg - exact) <= bound), H
        # a dropped or duplicated term would be far outside the bound
        assert np.max(np.abs(lg - exact) / mag) < 1e-5


def _brute_route(sh, logits, bias, orc):
    """Selection by library sort of the pinned sigmoid scores."""
    E, G, K, TG = sh.n_experts, sh.n_groups, sh.topk, sh.topk_groups
    epg = E // G
    s = np.array([orc.sigmoid(float(l)) for l in logits], np.float32)
    b = (s + bias.astype(np.float32)).astype(np.float32)
    gs = []
    for g in range(G):
        v = sorted(b[g * epg:(g + 1) * epg].tolist(), reverse=True)
        gs.append(np.float32(v[0]) + np.float32(v[1]) if epg >= 2 else np.float32(v[0]))
    groups = sorted(range(G), key=lambda g: (-gs[g], g))[:TG]
    cand = [e for g in groups for e in range(g * epg, (g + 1) * epg)]
    ids = sorted(cand, key=lambda e: (-b[e], e))[:K]
    return ids, s, b, gs


@pytest.mark.parametrize("shape", [dict(), dict(n_experts=64, n_groups=8, topk_groups=3, topk=6),
                                   dict(n_experts=256, n_groups=8, topk_groups=4, topk=8)])
def test_topk_matches_library_sort(orc, shape):
    sh = _shape(**shape)
    rng = np.random.default_rng(5)
    R = 40
    logits = rng.normal(0, 1, (R, sh.n_experts)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, sh.n_experts).astype(np.float32)
    ids, w = orc.route_from_logits(sh, logits, bias)
    for r in range(R):
        want, s, b, _ = _brute_route(sh, logits[r], bias, orc)
        assert ids[r].tolist() == want
        # weights: proportional to the unbiased sigmoid, summing to the scaling
        sel = s[want].astype(np.float64)
        np.testing.assert_allclose(w[r], sel / sel.sum() * sh.routed_scaling, rtol=3e-7)
        assert abs(float(w[r].astype(np.float64).sum()) - sh.routed_scaling) < 8 * 2.5 * 2 ** -23


def test_selection_by_enumeration(orc):
    """Chosen groups maximise the summed group score over all C(G,TG) subsets, and
    the chosen experts maximise the summed biased score over all K-subsets of the
    candidates (distinct scores, so the maximiser is unique)."""
    sh = _shape(n_experts=16, n_groups=4, topk_groups=2, topk=3)
    rng = np.random.default_rng(6)
    for _ in range(30):
        logits = rng.normal(0, 1, sh.n_experts).astype(np.float32)
        bias = rng.uniform(-0.1, 0.1, sh.n_experts).astype(np.float32)
        ids, _ = orc.route_from_logits(sh, logits[None], bias)
        _, s, b, gs = _brute_route(sh, logits, bias, orc)
        epg = sh.n_experts // sh.n_groups
        best_groups = max(itertools.combinations(range(sh.n_groups), sh.topk_groups),
                          key=lambda c: sum(float(gs[g]) for g in c))
        cand = [e for g in best_groups for e in range(g * epg, (g + 1) * epg)]
        best = max(itertools.combinations(cand, sh.topk), key=lambda c: sum(float(b[e]) for e in c))
        assert sorted(ids[0].tolist()) == sorted(best)
        # listed by biased score, descending
        assert all(b[ids[0][k]] >= b[ids[0][k + 1]] for k in range(sh.topk - 1))


def _ties():
    cases = []
    with open(GOLDEN) as f:
        block = {}
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, val = line.split("=", 1)
            block[key.strip()] = val.strip()
            if key.strip() == "ids":
                cases.append(block)
                block = {}
    return cases


def test_ties_lowest_id_wins(orc):
    for case in _ties():
        sh = _shape(**{k: int(case[k]) for k in ("n_experts", "n_groups", "topk_groups", "topk")})
        logits = np.array([float(v) for v in case["logits"].split()], np.float32)
        bias = np.array([float(v) for v in case["bias"].split()], np.float32)
        ids, w = orc.route_from_logits(sh, logits[None], bias)
        assert ids[0].tolist() == [int(v) for v in case["ids"].split()], case


def test_pads_not_routed(orc):
    sh = _shape()
    rng = np.random.default_rng(7)
    logits = rng.normal(0, 1, (6, sh.n_experts)).astype(np.float32)
    logits[2] = np.nan
    bias = np.zeros(sh.n_experts, np.float32)
    valid = np.array([1, 1, 0, 1, 0, 1], np.uint8)
    ids, w = orc.route_from_logits(sh, logits, bias, valid)
    assert np.all(ids[valid == 0] == -1) and np.all(w[valid == 0] == 0)
    assert np.all(ids[valid == 1] >= 0)


def test_row_permutation_equivariance(orc):
    wl = synth.WORKLOADS["tiny"]
    ri = synth.to_numpy(synth.make_router_inputs(synth.variant(wl, rows=24)))
    ids, w, lg = orc.route(wl.shape, ri["x"], ri["wr"], ri["bias"])
    perm = np.random.default_rng(8).permutation(24)
    ids2, w2, lg2 = orc.route(wl.shape, ri["x"][perm], ri["wr"], ri["bias"])
    assert np.array_equal(ids2, ids[perm])
    assert np.array_equal(w2.view(np.uint32), w[perm].view(np.uint32))
    assert np.array_equal(lg2.view(np.uint32), lg[perm].view(np.uint32))
