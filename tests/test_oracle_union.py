"""Pins of the oracle's expert union / dispatch order against a brute-force scan."""
import numpy as np

import synth


def _brute(ids, E, K):
    R = ids.shape[0]
    valid = ids[:, 0] >= 0
    slots = []                                   # (expert, r, k) for every valid slot
    for r in range(R):
        if not valid[r]:
            continue
        for k in range(K):
            slots.append((int(ids[r, k]), r, k))
    for r in range(R):
        if valid[r]:
            slots.append((E, r, K))
    # stable sort by expert keeps (r, k) order inside an expert
    order = sorted(range(len(slots)), key=lambda i: slots[i][0])
    pos = -np.ones((R, K + 1), np.int64)
    src = []
    for p, i in enumerate(order):
        e, r, k = slots[i]
        pos[r, k] = p
        src.append(r * (K + 1) + k)
    counts = np.bincount([s[0] for s in slots], minlength=E + 1)
    return counts, pos, np.array(src)


def test_union_matches_brute_force(orc):
    sh = synth.TINY
    rng = np.random.default_rng(9)
    for R in (1, 3, 8, 37):
        ids = np.stack([rng.choice(sh.n_experts, sh.topk, replace=False) for _ in range(R)])
        ids = ids.astype(np.int32)
        if R > 2:
            ids[1] = -1                                  # a pad row
        u = orc.build_union(sh, ids)
        counts, pos, src = _brute(ids, sh.n_experts, sh.topk)
        assert np.array_equal(u["counts"], counts)
        assert np.array_equal(u["pos"], pos)
        assert np.array_equal(u["src"], src)
        assert u["offsets"][0] == 0 and np.array_equal(np.diff(u["offsets"]), counts)
        hit = np.nonzero(counts[:sh.n_experts])[0]
        assert u["n_union"] == len(hit)
        assert u["ulist"].tolist() == hit.tolist() + [sh.n_experts]
        assert u["n_valid"] == int((ids[:, 0] >= 0).sum())


def test_union_empty_and_all_pads(orc):
    sh = synth.TINY
    ids = -np.ones((4, sh.topk), np.int32)
    u = orc.build_union(sh, ids)
    assert u["n_union"] == 0 and u["n_gathered"] == 0 and u["n_valid"] == 0
    assert np.all(u["pos"] == -1)
