"""Exact routing ties on the GPU, decided as the oracle decides them.

The rule (lowest group id, then lowest expert id wins; experts listed by
biased score descending) makes the routing bit-exact.  openinfer #610 "TP8
span row mapping ...", section "Gates", had to tolerate tie-flips between two
mappings; here none is allowed, so the GPU is handed real ties:

* a row of x = 0 gives every logit exactly +0 and every sigmoid score exactly
  0.5; biases that are multiples of 1/8 keep every biased score and every
  group score exact, so equal values are equal bits (the hand-derived cases of
  tests/golden/route_ties.txt, whose ids are also checked here);
* a row of x that is 1.0 in one column h and 0 elsewhere gives logits that are
  exactly the router weights of that column; columns drawn from {-1, 0, 1}
  give each row its own pattern of tied sigmoid scores, and a few columns put
  the tied maxima across lane boundaries of the selection warp (experts 31 and
  32, 63 and 64).

Routing ids, weights and logits are compared bit for bit with the oracle
through moe_route, and ids and weights through moe_layer: at 40 rows (the
one-block selection + union kernel) and at 72 rows (separate selection and
union kernels); the layer output stays within the parity tolerance.
"""
import os

import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle
import synth
from gpu_helpers import TOL, bf16_bits_to_f64, bf16_to_np, rel_fro, run_layer

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_ties.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def _golden():
    cases, block = [], {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            block[key] = val
            if key == "ids":
                cases.append(block)
                block = {}
    return cases


def _shape(E, G, TG, K, hidden=256, inter=128):
    return synth.LayerShape(hidden=hidden, inter=inter, n_experts=E, n_groups=G,
                            topk_groups=TG, topk=K, n_shared=1, routed_scaling=2.5)


def _tie_inputs(shape, R, seed):
    """x, wr, bias whose logits are exact small values with many ties.

    Row 0 is all zeros; row 1 is a N(0,1) row (no ties); every other row r is
    1.0 in its own column h_r, whose router weights are drawn from {-1, 0, 1}
    (columns 2 and 3 put the largest value on experts 31, 32 and 63, 64 only).
    Biases are multiples of 1/8 in [0, 1/4]."""
    E, H = shape.n_experts, shape.hidden
    rng = np.random.default_rng(seed)
    assert R <= H
    x = np.zeros((R, H), np.float32)
    wr = np.zeros((E, H), np.float32)
    x[1] = rng.normal(0.0, 1.0, H)
    wr += rng.normal(0.0, 1.0 / np.sqrt(H), (E, H)).astype(np.float32) * (x[1] != 0)
    for r in range(2, R):
        h = r                                         # one column per row
        x[r] = 0.0
        x[r, h] = 1.0
        wr[:, h] = rng.choice(np.array([-1.0, 0.0, 1.0], np.float32), E)
    for r, top in ((2, (31, 32)), (3, (31, 32, 63, 64))):
        if r < R and E > max(top):
            wr[:, r] = -1.0
            wr[list(top), r] = 1.0
    bias = (rng.integers(0, 3, E) / 8.0).astype(np.float32)
    if E > 64:
        bias[[31, 32, 63, 64]] = 0.25
    xb = torch.from_numpy(x).to(torch.bfloat16)
    return xb, torch.from_numpy(wr), torch.from_numpy(bias)


def _route_gpu(shape, x, wr, bias, valid=None):
    R, E, K = x.shape[0], shape.n_experts, shape.topk
    cfg = m.Config.from_shape(shape)
    ids = torch.empty((R, K), dtype=torch.int32, device="cuda")
    w = torch.empty((R, K), dtype=torch.float32, device="cuda")
    logits = torch.zeros((R, E), dtype=torch.float32, device="cuda")
    m.moe_route(cfg, x.cuda(), wr.cuda(), bias.cuda(),
                None if valid is None else valid.cuda(), ids, w, logits)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), logits.cpu().numpy()


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("case", range(len(_golden())))
def test_golden_ties_on_gpu(case):
    c = _golden()[case]
    E, G, TG, K = (int(c[k]) for k in ("n_experts", "n_groups", "topk_groups", "topk"))
    shape = _shape(E, G, TG, K)
    bias = torch.tensor([float(v) for v in c["bias"].split()], dtype=torch.float32)
    assert all(float(v) == 0.0 for v in c["logits"].split())
    R = 8
    x = torch.zeros((R, shape.hidden), dtype=torch.bfloat16)
    wr = torch.from_numpy(np.random.default_rng(case).normal(0, 1, (E, shape.hidden))
                          .astype(np.float32))
    ids, w, lg = _route_gpu(shape, x, wr, bias)
    want = [int(v) for v in c["ids"].split()]
    assert np.all(lg == 0.0)
    for r in range(R):
        assert ids[r].tolist() == want
    ref_ids, ref_w, _ = oracle.route(shape, synth.to_numpy({"x": x})["x"], wr.numpy(),
                                     bias.numpy())
    assert np.array_equal(ids, ref_ids)
    assert np.array_equal(_bits(w), _bits(ref_w))
    # through the whole layer (one-block selection + union at 8 rows)
    wl = synth.Workload("ties", shape, rows=R)
    t = {k: v.cuda() for k, v in synth.make_expert_weights(wl).items()}
    t.update({"x": x.cuda(), "wr": wr.cuda(), "bias": bias.cuda(),
              "row_valid": torch.ones(R, dtype=torch.uint8, device="cuda")})
    out, lids, lw, _ = run_layer(m.Config.from_shape(shape), t, R)
    assert np.array_equal(lids.cpu().numpy(), ref_ids)
    assert np.array_equal(_bits(lw.cpu().numpy()), _bits(ref_w))
    assert np.all(bf16_to_np(out) == 0)          # x = 0: every expert output is 0


# The GLM-5.2 routing shape (256 experts in 8 groups, top-4 groups, top-8) at
# the real hidden size for moe_route, and 32 groups of 8 experts.
ROUTE_SHAPES = [_shape(256, 8, 4, 8, hidden=6144), _shape(256, 32, 4, 8, hidden=6144),
                _shape(256, 32, 8, 16, hidden=6144)]


@pytest.mark.parametrize("si", range(len(ROUTE_SHAPES)))
@pytest.mark.parametrize("seed", [0, 1])
def test_route_ties_bit_exact(si, seed):
    shape = ROUTE_SHAPES[si]
    R = 48
    x, wr, bias = _tie_inputs(shape, R, seed)
    ids, w, lg = _route_gpu(shape, x, wr, bias)
    ref_ids, ref_w, ref_lg = oracle.route(shape, synth.to_numpy({"x": x})["x"], wr.numpy(),
                                          bias.numpy())
    assert np.array_equal(_bits(lg), _bits(ref_lg))
    # the one-hot rows' logits are exactly their column of router weights
    for r in range(2, R):
        assert np.array_equal(lg[r], wr[:, r].numpy())
    assert np.array_equal(ids, ref_ids)
    assert np.array_equal(_bits(w), _bits(ref_w))
    # the lane-boundary rows: the tied maxima come first, lower id first
    assert ids[2][:2].tolist() == [31, 32]
    assert ids[3][:4].tolist() == [31, 32, 63, 64]


# The same routing shapes at 128-wide experts for whole-layer calls.
LAYER_SHAPES = [_shape(256, 8, 4, 8), _shape(256, 32, 4, 8)]


@pytest.mark.parametrize("si", range(len(LAYER_SHAPES)))
@pytest.mark.parametrize("R", [40, 72])
def test_layer_ties_bit_exact(si, R):
    shape = LAYER_SHAPES[si]
    x, wr, bias = _tie_inputs(shape, R, seed=R)
    valid = torch.ones(R, dtype=torch.uint8)
    valid[R - 1] = 0                              # one pad row (NaN x)
    x[R - 1] = float("nan")
    wl = synth.Workload("ties", shape, rows=R)
    w_cpu = synth.make_expert_weights(wl)
    t = {k: v.cuda() for k, v in w_cpu.items()}
    t.update({"x": x.cuda(), "wr": wr.cuda(), "bias": bias.cuda(), "row_valid": valid.cuda()})
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    h = synth.to_numpy({"x": x, "wr": wr, "bias": bias, "row_valid": valid})
    h.update(synth.to_numpy(w_cpu))
    ref = oracle.moe_layer(shape, h)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(_bits(w.cpu().numpy()), _bits(ref["wts"]))
    y = bf16_bits_to_f64(bf16_to_np(out))
    v = valid.numpy() != 0
    assert np.all(np.isfinite(y))
    assert rel_fro(y[v], ref["y_acc"][v]) <= TOL
    assert np.all(bf16_to_np(out)[~v] == 0)
