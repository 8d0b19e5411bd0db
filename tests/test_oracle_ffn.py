"""Pins of the oracle's activation quantisation, expert FFN and combine.

* quantisation: per-128 scale = amax/448, the amax element lands on +-448,
  every decoded value within half a grid step of x, zero blocks stay zero;
* expert FFN: equal to an fp64 numpy matmul on weights dequantised through
  torch's float8_e4m3fn conversion (a library routine, not the oracle's decode);
* combine: closed forms -- identical experts give routed_scaling * f + f_shared,
  a zero row gives exact zeros, one expert per group with K = 1 reduces to that
  expert, pad rows give +0.0 even when x is NaN, rows are independent;
* the whole tiny layer against the same library composition.
"""
import numpy as np
import pytest
import torch

import synth


def lib_dequant(codes, scales):
    w = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(np.ascontiguousarray(scales)).double()
    s = s.repeat_interleave(128, -2).repeat_interleave(128, -1)
    return (w * s).numpy()


def lib_quant(v32):
    """Per-128 e4m3 quantisation through torch's cast: codes, scales."""
    v32 = np.asarray(v32, np.float32).reshape(-1, 128)
    amax = np.abs(v32).max(axis=1)
    s = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32))
    q = torch.from_numpy((v32 / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy().reshape(-1), s.astype(np.float32)


def lib_expert(xhat, wg, sg, wu, su, wd, sd):
    g = lib_dequant(wg, sg) @ xhat
    u = lib_dequant(wu, su) @ xhat
    h = (g / (1.0 + np.exp(-g)) * u).astype(np.float32)
    hq, hs = lib_quant(h)
    hhat = torch.from_numpy(hq).view(torch.float8_e4m3fn).double().numpy() * np.repeat(hs, 128)
    return lib_dequant(wd, sd) @ hhat, hq


def test_quant_rule(orc):
    rng = np.random.default_rng(10)
    v = rng.normal(0, 1, 128 * 6).astype(np.float32)
    v[128:256] = 0.0
    v[256:384] *= 1e-3
    q, s = orc.quant_1x128(v)
    dec = orc.e4m3_decode(q)
    for b in range(6):
        blk = v[b * 128:(b + 1) * 128]
        amax = np.abs(blk).max()
        if amax == 0:
            assert s[b] == 1.0 and np.all(dec[b * 128:(b + 1) * 128] == 0)
            continue
        assert s[b] == np.float32(amax) / np.float32(448)
        assert np.max(np.abs(dec[b * 128:(b + 1) * 128])) == 448.0
        xhat = dec[b * 128:(b + 1) * 128].astype(np.float64) * s[b]
        # e4m3 keeps 4 significant bits: relative error <= 2^-4, absolute <= 2^-10 * s
        err = np.abs(xhat - blk)
        assert np.all(err <= np.maximum(np.abs(blk) * 2.0 ** -4, 2.0 ** -10 * s[b]) * 1.0001)
    q2, s2 = lib_quant(v)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    return wl, synth.to_numpy(synth.make_layer(wl))


def test_expert_ffn_matches_library(orc, tiny):
    wl, t = tiny
    sh = wl.shape
    xf = orc.bf16_to_f32(t["x"])
    for r, e in ((0, 3), (5, 11), (7, 0)):
        xq, xs = orc.quant_1x128(xf[r])
        xhat = torch.from_numpy(xq).view(torch.float8_e4m3fn).double().numpy() * np.repeat(xs, 128)
        args = (t["w_gate"][e], t["s_gate"][e], t["w_up"][e], t["s_up"][e], t["w_down"][e],
                t["s_down"][e])
        o, hq, hs = orc.expert_ffn(sh, xq, xs, *args)
        o_ref, hq_ref = lib_expert(xhat, *args)
        assert np.sum(hq != hq_ref) <= 1
        # the oracle dequantises to fp32 (one rounding per weight), the library
        # path in fp64: norm-wise they agree to ~1e-7; a dropped term or a wrong
        # scale index shows up at 1e-2 or more
        assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) < 1e-6
        # fp32 accumulation stays close to fp64
        o32, _, _ = orc.expert_ffn(sh, xq, xs, *args, acc64=False)
        assert np.linalg.norm(o32 - o) / np.linalg.norm(o) < 1e-4


def _lib_layer_row(orc, sh, t, r, ids, wts):
    xf = orc.bf16_to_f32(t["x"][r])
    xq, xs = orc.quant_1x128(xf)
    xhat = torch.from_numpy(xq).view(torch.float8_e4m3fn).double().numpy() * np.repeat(xs, 128)
    acc = None
    for k in range(sh.topk):
        e = ids[k]
        o, _ = lib_expert(xhat, t["w_gate"][e], t["s_gate"][e], t["w_up"][e], t["s_up"][e],
                          t["w_down"][e], t["s_down"][e])
        acc = wts[k] * o if acc is None else acc + wts[k] * o
    o_sh, _ = lib_expert(xhat, t["sh_gate"][0], t["sh_s_gate"][0], t["sh_up"][0],
                         t["sh_s_up"][0], t["sh_down"][0], t["sh_s_down"][0])
    return acc + o_sh


def test_layer_matches_library_composition(orc, tiny):
    wl, t = tiny
    res = orc.moe_layer(wl.shape, t)
    ids, w, _ = orc.route(wl.shape, t["x"], t["wr"], t["bias"])
    assert np.array_equal(res["ids"], ids) and np.array_equal(res["wts"], w)
    for r in range(wl.rows):
        ref = _lib_layer_row(orc, wl.shape, t, r, ids[r], w[r].astype(np.float64))
        assert np.linalg.norm(res["y_acc"][r] - ref) / np.linalg.norm(ref) < 1e-6
    y = orc.bf16_to_f32(res["out"]).astype(np.float64)
    rel = np.linalg.norm(y - res["y_acc"]) / np.linalg.norm(res["y_acc"])
    assert rel < 2.0 ** -8


def test_identical_experts_closed_form(orc, tiny):
    wl, t = tiny
    t = dict(t)
    for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"):
        t[k] = np.repeat(t[k][:1], wl.shape.n_experts, axis=0)
    res = orc.moe_layer(wl.shape, t)
    xf = orc.bf16_to_f32(t["x"])
    for r in range(wl.rows):
        xq, xs = orc.quant_1x128(xf[r])
        f, _, _ = orc.expert_ffn(wl.shape, xq, xs, t["w_gate"][0], t["s_gate"][0], t["w_up"][0],
                                 t["s_up"][0], t["w_down"][0], t["s_down"][0])
        fs, _, _ = orc.expert_ffn(wl.shape, xq, xs, t["sh_gate"][0], t["sh_s_gate"][0],
                                  t["sh_up"][0], t["sh_s_up"][0], t["sh_down"][0],
                                  t["sh_s_down"][0])
        ref = 2.5 * f + fs
        # the routed weights sum to 2.5 up to fp32 rounding
        assert np.linalg.norm(res["y_acc"][r] - ref) / np.linalg.norm(ref) < 1e-6


def test_zero_row_and_pads(orc, tiny):
    wl, t = tiny
    t = dict(t)
    x = t["x"].copy()
    x[2] = 0                              # +0.0 bf16
    x[5] = 0x7FC0                         # NaN
    t["x"] = x
    valid = np.ones(wl.rows, np.uint8)
    valid[5] = 0
    t["row_valid"] = valid
    res = orc.moe_layer(wl.shape, t)
    assert np.all(res["out"][2] == 0) and np.all(res["out"][5] == 0)
    assert np.all(res["ids"][5] == -1) and np.all(res["wts"][5] == 0)
    # rows are independent: the others match a run without the edits
    ref = orc.moe_layer(wl.shape, dict(t, x=tiny[1]["x"], row_valid=None))
    for r in (0, 1, 3, 4, 6, 7):
        assert np.array_equal(res["out"][r], ref["out"][r])
    sub = orc.moe_layer(wl.shape, t, rows=[6, 1])
    assert np.array_equal(sub["out"][[1, 6]], res["out"][[1, 6]])


def test_single_expert_per_group_k1(orc, tiny):
    wl, t = tiny
    sh = synth.LayerShape(hidden=256, inter=128, n_experts=4, n_groups=4, topk_groups=1,
                          topk=1, n_shared=1, routed_scaling=2.5)
    t = dict(t)
    for k in ("w_gate", "s_gate", "w_up", "s_up", "w_down", "s_down"):
        t[k] = t[k][:4]
    t["wr"] = t["wr"][:4]
    t["bias"] = t["bias"][:4]
    res = orc.moe_layer(sh, t)
    xf = orc.bf16_to_f32(t["x"])
    for r in range(wl.rows):
        lg = orc.router_logits(sh, t["x"][r:r + 1], t["wr"])[0]
        b = [orc.sigmoid(float(l)) + float(np.float32(t["bias"][e])) for e, l in enumerate(lg)]
        e = int(np.argmax(b))
        assert res["ids"][r, 0] == e and res["wts"][r, 0] == np.float32(2.5)
        xq, xs = orc.quant_1x128(xf[r])
        f, _, _ = orc.expert_ffn(sh, xq, xs, t["w_gate"][e], t["s_gate"][e], t["w_up"][e],
                                 t["s_up"][e], t["w_down"][e], t["s_down"][e])
        fs, _, _ = orc.expert_ffn(sh, xq, xs, t["sh_gate"][0], t["sh_s_gate"][0], t["sh_up"][0],
                                  t["sh_s_up"][0], t["sh_down"][0], t["sh_s_down"][0])
        np.testing.assert_allclose(res["y_acc"][r], 2.5 * f + fs, rtol=1e-12, atol=1e-15)


def test_fp32_vs_fp64_accumulation(orc, tiny):
    wl, t = tiny
    a = orc.moe_layer(wl.shape, t, acc64=True)["y_acc"]
    b = orc.moe_layer(wl.shape, t, acc64=False)["y_acc"]
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-4
