"""GPU parity on small shapes the oracle finishes in seconds: every C entry
point against the oracle, invariants, edge cases.

* routing: logits, ids and weights bit-exact (the same IEEE fp32 op order);
* union: every word of the documented layout bit-exact;
* dispatch: quantised activation codes and scales bit-exact;
* expert FFN and combine: within 1e-2 relative Frobenius norm of the oracle;
* pads: +0.0 whatever x holds, NaN-poisoned outputs overwritten;
* a row's outputs are bit-identical wherever it sits in the batch;
* every row-tile variant (16 / 32 / 64 rows per item) with ragged tails.
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
    wl = synth.Workload("t", shape, rows=rows, pads=tuple(pads), seed=seed, routing=routing)
    t_cpu = synth.make_layer(wl, device="cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    return wl, t, synth.to_numpy(t_cpu)


@pytest.mark.parametrize("shape,rows,pads", [(synth.TINY, 8, ()), (MEDIUM, 8, (3,)),
                                             (MEDIUM, 37, (0, 36))])
def test_layer_matches_oracle(shape, rows, pads):
    wl, t, h = _make(shape, rows, pads)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, rows)
    ref = oracle.moe_layer(shape, h)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["wts"].view(np.uint32))
    y = bf16_bits_to_f64(bf16_to_np(out))
    assert np.all(np.isfinite(y))
    valid = h["row_valid"] != 0
    assert rel_fro(y[valid], ref["y_acc"][valid]) <= TOL
    assert np.all(bf16_to_np(out)[~valid] == 0)


def test_stepwise_entry_points():
    shape = MEDIUM
    R = 24
    wl, t, h = _make(shape, R, pads=(5,))
    cfg = m.Config.from_shape(shape)
    E, K, H, I = shape.n_experts, shape.topk, shape.hidden, shape.inter
    dev = torch.device("cuda")
    # --- moe_route
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.zeros((R, E), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ref_ids, ref_w, ref_logits = oracle.route(shape, h["x"], h["wr"], h["bias"], h["row_valid"])
    valid = h["row_valid"] != 0
    lg = logits.cpu().numpy()
    assert np.array_equal(lg[valid].view(np.uint32), ref_logits[valid].view(np.uint32))
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    # --- moe_build_union
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    u = ub.cpu().numpy()
    ref = oracle.build_union(shape, ref_ids)
    lay = m.union_layout(cfg, R)
    KS = K + 1
    assert u[0] == ref["n_union"] and u[1] == ref["n_valid"] and u[2] == ref["n_gathered"]
    assert u[4] == m.rows_per_item(R) and u[5] == 0
    assert np.array_equal(u[lay["counts"]:lay["counts"] + E + 1], ref["counts"])
    assert np.array_equal(u[lay["offsets"]:lay["offsets"] + E + 2], ref["offsets"])
    assert np.array_equal(u[lay["ulist"]:lay["ulist"] + ref["n_union"] + 1], ref["ulist"])
    assert np.array_equal(u[lay["pos"]:lay["pos"] + R * KS].reshape(R, KS), ref["pos"])
    T = ref["n_gathered"]
    assert np.array_equal(u[lay["src"]:lay["src"] + T], ref["src"])
    items = u[lay["items"]:lay["items"] + 4 * u[3]].reshape(-1, 4)
    covered = np.zeros(T, np.int32)
    nt = m.rows_per_item(R)
    off = ref["offsets"]
    for e, r0, n, _ in items:
        assert 1 <= n <= nt and off[e] <= r0 and r0 + n <= off[e + 1]
        covered[r0:r0 + n] += 1
    assert np.all(covered == 1)
    # --- moe_expert_ffn_fp8
    ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    y_slots = torch.full((R * K, H), float("nan"), dtype=torch.float32, device=dev)
    y_sh = torch.full((R, H), float("nan"), dtype=torch.float32, device=dev)
    m.moe_expert_ffn_fp8(cfg, t["x"], m.Weights.from_tensors(t), ub, y_slots, y_sh, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    fl = m.ffn_layout(cfg, R)
    wsh = ws.cpu().numpy()
    xg = wsh[fl["xg"]:fl["xg"] + T * H].reshape(T, H)
    xs = wsh[fl["xs"]:fl["xs"] + T * (H // 128) * 4].view(np.float32).reshape(T, H // 128)
    hq = wsh[fl["hq"]:fl["hq"] + T * I].reshape(T, I)
    xf = oracle.bf16_to_f32(h["x"])
    ys = y_slots.cpu().numpy().reshape(R, K, H)
    ysh = y_sh.cpu().numpy()
    hq_mismatch = 0
    for r in np.nonzero(valid)[0]:
        q, s = oracle.quant_1x128(xf[r])
        for k in range(KS):
            p = ref["pos"][r, k]
            assert np.array_equal(xg[p], q) and np.array_equal(xs[p], s)
            e = ref_ids[r, k] if k < K else None
            if e is None:
                args = (h["sh_gate"][0], h["sh_s_gate"][0], h["sh_up"][0], h["sh_s_up"][0],
                        h["sh_down"][0], h["sh_s_down"][0])
                got = ysh[r]
            else:
                args = (h["w_gate"][e], h["s_gate"][e], h["w_up"][e], h["s_up"][e],
                        h["w_down"][e], h["s_down"][e])
                got = ys[r, k]
            o, hq_ref, _ = oracle.expert_ffn(shape, q, s, *args)
            assert rel_fro(got, o) <= TOL
            hq_mismatch += int(np.sum(hq[p] != hq_ref))
    assert hq_mismatch <= 0.001 * valid.sum() * KS * I + 2
    # pad rows of the outputs are untouched
    assert np.all(np.isnan(ys[~valid])) and np.all(np.isnan(ysh[~valid]))
    # --- moe_combine: fixed-order weighted sum of the GPU's own slot outputs
    out = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=dev)
    m.moe_combine(cfg, y_slots, y_sh, w, ub, out)
    torch.cuda.synchronize()
    got = bf16_bits_to_f64(bf16_to_np(out))
    wn = ref_w.astype(np.float64)
    for r in np.nonzero(valid)[0]:
        acc = sum(wn[r, k] * ys[r, k].astype(np.float64) for k in range(K)) + ysh[r]
        assert rel_fro(got[r], acc) <= 2 ** -8
    assert np.all(bf16_to_np(out)[~valid] == 0)


@pytest.mark.parametrize("shape,R,pads", [(synth.TINY, 8, ()), (MEDIUM, 8, (2, 5)),
                                          (MEDIUM, 37, (0, 36)), (MEDIUM, 64, (7, 23, 39, 55)),
                                          (synth.TINY, 1, ())])
def test_layer_routing_matches_stepwise(shape, R, pads):
    """moe_layer selects and builds the union in one kernel at these row counts;
    its ids, weights and output equal moe_route + moe_build_union +
    moe_expert_ffn_fp8 + moe_combine bit for bit."""
    wl, t, h = _make(shape, R, pads)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    dev = torch.device("cuda")
    K, H, E = shape.topk, shape.hidden, shape.n_experts
    ids2 = torch.empty((R, K), dtype=torch.int32, device=dev)
    w2 = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, E), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids2, w2, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids2, ub)
    ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
    ys = torch.empty((R * K, H), dtype=torch.float32, device=dev)
    ysh = torch.empty((R, H), dtype=torch.float32, device=dev)
    m.moe_expert_ffn_fp8(cfg, t["x"], m.Weights.from_tensors(t), ub, ys, ysh, ws)
    out2 = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=dev)
    m.moe_combine(cfg, ys, ysh, w2, ub, out2)
    torch.cuda.synchronize()
    assert m.moe_get_device_error(ws) == 0
    assert np.array_equal(ids.cpu().numpy(), ids2.cpu().numpy())
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w2.cpu().numpy().view(np.uint32))
    assert np.array_equal(bf16_to_np(out), bf16_to_np(out2))
    ref_ids, _, _ = oracle.route(shape, h["x"], h["wr"], h["bias"], h["row_valid"])
    assert np.array_equal(ids.cpu().numpy(), ref_ids)


@pytest.mark.parametrize("shape,R", [(synth.TINY, 8), (MEDIUM, 37), (MEDIUM, 200), (synth.TINY, 600)])
def test_fused_gemms_match_two_launches(shape, R):
    """moe_expert_gemms_fp8 (one persistent launch, down tiles gated by per-item
    counters) gives the same bits as moe_gate_up_fp8 followed by moe_down_fp8."""
    wl, t, h = _make(shape, R, pads=(1,) if R > 2 else ())
    cfg = m.Config.from_shape(shape)
    dev = torch.device("cuda")
    K, H = shape.topk, shape.hidden
    ids = torch.empty((R, K), dtype=torch.int32, device=dev)
    w = torch.empty((R, K), dtype=torch.float32, device=dev)
    logits = torch.empty((R, shape.n_experts), dtype=torch.float32, device=dev)
    m.moe_route(cfg, t["x"], t["wr"], t["bias"], t["row_valid"], ids, w, logits)
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device=dev)
    m.moe_build_union(cfg, ids, ub)
    W = m.Weights.from_tensors(t)
    outs = []
    for fused in (True, False):
        ws = torch.zeros(m.moe_ffn_workspace_bytes(cfg, R), dtype=torch.uint8, device=dev)
        ys = torch.zeros((R * K, H), dtype=torch.float32, device=dev)
        ysh = torch.zeros((R, H), dtype=torch.float32, device=dev)
        m.moe_dispatch(cfg, t["x"], ub, ws)
        if fused:
            m.moe_expert_gemms_fp8(cfg, W, ub, R, ys, ysh, ws)
        else:
            m.moe_gate_up_fp8(cfg, W, ub, R, ws)
            m.moe_down_fp8(cfg, W, ub, R, ys, ysh, ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        outs.append((ys.cpu().numpy(), ysh.cpu().numpy()))
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][1].view(np.uint32), outs[1][1].view(np.uint32))


def test_pads_nan_zero_filled():
    wl, t, h = _make(synth.TINY, 16, pads=(0, 7, 15))
    cfg = m.Config.from_shape(synth.TINY)
    out, ids, w, _ = run_layer(cfg, t, 16)
    o = bf16_to_np(out)
    for p in (0, 7, 15):
        assert np.all(o[p] == 0)                       # +0.0, not -0.0, not NaN
        assert np.all(ids.cpu().numpy()[p] == -1) and np.all(w.cpu().numpy()[p] == 0)
    # the other rows do not see the pads: same bits as a run with valid copies
    t2 = dict(t)
    x2 = t["x"].clone()
    x2[[0, 7, 15]] = 0
    t2["x"] = x2
    t2["row_valid"] = torch.ones_like(t["row_valid"])
    out2, _, _, _ = run_layer(cfg, t2, 16)
    keep = [r for r in range(16) if r not in (0, 7, 15)]
    assert np.array_equal(o[keep], bf16_to_np(out2)[keep])


@pytest.mark.parametrize("shape,R", [(synth.TINY, 8), (MEDIUM, 64), (MEDIUM, 200), (MEDIUM, 300)])
def test_row_slot_bit_identity(shape, R):
    """The same row gives the same bits wherever it sits in the batch
    (openinfer #610, "Gates": same rows through both mappings bit-identical)."""
    wl, t, h = _make(shape, R)
    cfg = m.Config.from_shape(shape)
    out, ids, _, _ = run_layer(cfg, t, R)
    perm = torch.from_numpy(np.random.default_rng(11).permutation(R)).cuda()
    t2 = dict(t)
    t2["x"] = t["x"][perm].contiguous()
    out2, ids2, _, _ = run_layer(cfg, t2, R)
    pc = perm.cpu().numpy()
    assert np.array_equal(bf16_to_np(out2), bf16_to_np(out)[pc])
    assert np.array_equal(ids2.cpu().numpy(), ids.cpu().numpy()[pc])


@pytest.mark.parametrize("R", [1, 13, 64, 65, 100, 256, 257, 512, 513, 600])
def test_row_counts_and_tiles(R):
    """Every row-tile variant with ragged tails, on both sides of each switch
    (16 rows up to 64, 32 up to 256, 64 above, the deeper ring up to 512);
    several items per expert."""
    shape = synth.TINY
    wl, t, h = _make(shape, R, seed=R)
    cfg = m.Config.from_shape(shape)
    out, ids, w, _ = run_layer(cfg, t, R)
    rows = np.unique(np.linspace(0, R - 1, min(R, 24)).astype(int))
    ref = oracle.moe_layer(shape, h, rows=rows)
    ref_ids, ref_w, _ = oracle.route(shape, h["x"], h["wr"], h["bias"])
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))
    y = bf16_bits_to_f64(bf16_to_np(out))
    assert rel_fro(y[rows], ref["y_acc"][rows]) <= TOL


def test_zero_rows_and_limits():
    shape = synth.TINY
    cfg = m.Config.from_shape(shape)
    dev = torch.device("cuda")
    x = torch.zeros((0, shape.hidden), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    wl, t, h = _make(shape, 4)
    out = torch.zeros((0, shape.hidden), dtype=torch.bfloat16, device=dev)
    m.moe_layer(cfg, x, t["wr"], t["bias"], m.Weights.from_tensors(t), None, out,
                torch.zeros(max(256, m.moe_workspace_bytes(cfg, 0)), dtype=torch.uint8, device=dev))
    big = torch.zeros((m.MOE_MAX_ROWS + 1, shape.hidden), dtype=torch.bfloat16, device=dev)
    with pytest.raises(m.MoeError) as ei:
        m.moe_layer(cfg, big, t["wr"], t["bias"], m.Weights.from_tensors(t), None, big, ws)
    assert ei.value.status == 2


def test_all_rows_pad():
    wl, t, h = _make(synth.TINY, 8, pads=tuple(range(8)))
    cfg = m.Config.from_shape(synth.TINY)
    out, ids, w, _ = run_layer(cfg, t, 8)
    assert np.all(bf16_to_np(out) == 0) and np.all(ids.cpu().numpy() == -1)


def test_union_rejects_bad_ids():
    cfg = m.Config.from_shape(synth.TINY)
    R, K = 4, synth.TINY.topk
    ids = torch.tensor([[0, 1, 2, 3], [4, 4, 5, 6], [-1, -1, -1, -1], [7, 8, 99, 9]],
                       dtype=torch.int32, device="cuda")
    ub = torch.zeros(m.moe_union_bytes(cfg, R) // 4, dtype=torch.int32, device="cuda")
    m.moe_build_union(cfg, ids, ub)
    u = ub.cpu().numpy()
    lay = m.union_layout(cfg, R)
    pos = u[lay["pos"]:lay["pos"] + R * (K + 1)].reshape(R, K + 1)
    assert u[5] == 1 and u[1] == 1                      # error flagged, one valid row
    assert np.all(pos[1:] == -1) and np.all(pos[0] >= 0)


def test_bounded_wait_times_out_without_fault():
    """A wait nothing releases gives up, reports MOE_ERR_TIMEOUT, and the context
    stays usable."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    m.moe_diag_wait_timeout(ws, 20000)
    assert m.moe_get_device_error(ws, clear=True) == 4
    assert m.moe_get_device_error(ws) == 0
    wl, t, h = _make(synth.TINY, 8)
    out, ids, _, _ = run_layer(m.Config.from_shape(synth.TINY), t, 8)
    assert np.all(np.isfinite(bf16_bits_to_f64(bf16_to_np(out))))
