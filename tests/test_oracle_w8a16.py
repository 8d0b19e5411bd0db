"""Pins of the oracle's 16-bit-activation variants of the expert FFN.

w8a16 (mstar #388, commit on kernel switches and the FlashInfer commit: fp8
weights with bf16 activations at decode sizes) and the unrounded yardstick:

* the bf16 rounding used here is the library's round-half-even (numpy rint
  at 8 significant bits), itself checked against torch's fp32 -> bf16 cast;
* one expert, w8a16: equal to an fp64 numpy matmul on weights dequantised by
  torch's float8_e4m3fn cast, rounded to bf16, with h rounded to bf16;
* one expert, unrounded: the same without either rounding;
* the tiny layer in both variants against the library composition (ids and
  weights from the routing, which the routing pins cover);
* the point of the variant: its error against the unrounded layer is far below
  the fp8 path's (no activation quantisation), and the routing is the same.
"""
import numpy as np
import pytest
import torch

import synth


def lib_bf16(v):
    """Round float64 values in bf16's normal range to bf16 (8 significant
    bits), half to even."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def lib_dequant(codes, scales):
    w = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(np.ascontiguousarray(scales)).double()
    s = s.repeat_interleave(128, -2).repeat_interleave(128, -1)
    return (w * s).numpy()


def lib_expert_a16(x, wg, sg, wu, su, wd, sd, round16):
    r = lib_bf16 if round16 else (lambda a: a)
    g = r(lib_dequant(wg, sg)) @ x
    u = r(lib_dequant(wu, su)) @ x
    h = r(g / (1.0 + np.exp(-g)) * u)
    return r(lib_dequant(wd, sd)) @ h


def x_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def tiny():
    wl = synth.WORKLOADS["tiny"]
    return wl, synth.to_numpy(synth.make_layer(wl))


def test_lib_bf16_is_the_library_rounding():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-4, 20000),
                        rng.normal(0, 300, 20000)]).astype(np.float32)
    # exact ties of bf16 (the 16 dropped bits 1000...0) both ways, normal range
    ties = ((np.arange(0, 2000, dtype=np.uint32) + 0x3E00) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, ties, -ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(lib_bf16(v.astype(np.float64)), ref)


@pytest.mark.parametrize("round16", [True, False])
def test_expert_a16_matches_library(orc, tiny, round16):
    wl, t = tiny
    s = wl.shape
    for r, e in [(0, 0), (3, 7), (5, s.n_experts - 1)]:
        args = (t["w_gate"][e], t["s_gate"][e], t["w_up"][e], t["s_up"][e], t["w_down"][e],
                t["s_down"][e])
        got = orc.expert_ffn_a16(s, t["x"][r], *args, round16=round16)
        ref = lib_expert_a16(x_values(t["x"][r]), *args, round16)
        assert np.linalg.norm(got - ref) <= 1e-12 * np.linalg.norm(ref)


def test_w8a16_rounds_weights_and_h(orc, tiny):
    """A dropped rounding would be caught: the two variants differ by far more
    than the comparison tolerance above."""
    wl, t = tiny
    s = wl.shape
    args = (t["w_gate"][2], t["s_gate"][2], t["w_up"][2], t["s_up"][2], t["w_down"][2],
            t["s_down"][2])
    a = orc.expert_ffn_a16(s, t["x"][1], *args, round16=True)
    b = orc.expert_ffn_a16(s, t["x"][1], *args, round16=False)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-5 < rel < 2e-2


@pytest.mark.parametrize("variant", ["w8a16", "exact"])
def test_layer_a16_matches_library_composition(orc, tiny, variant):
    wl, t = tiny
    s = wl.shape
    res = orc.moe_layer(s, t, variant=variant)
    ids, wts = res["ids"], res["wts"]
    for r in range(wl.rows):
        x = x_values(t["x"][r])
        acc = None
        for k in range(s.topk):
            e = ids[r, k]
            o = lib_expert_a16(x, t["w_gate"][e], t["s_gate"][e], t["w_up"][e], t["s_up"][e],
                               t["w_down"][e], t["s_down"][e], variant == "w8a16")
            acc = float(wts[r, k]) * o if acc is None else acc + float(wts[r, k]) * o
        acc = acc + lib_expert_a16(x, t["sh_gate"][0], t["sh_s_gate"][0], t["sh_up"][0],
                                   t["sh_s_up"][0], t["sh_down"][0], t["sh_s_down"][0],
                                   variant == "w8a16")
        assert np.linalg.norm(res["y_acc"][r] - acc) <= 1e-12 * np.linalg.norm(acc)


def test_w8a16_error_far_below_fp8(orc, tiny):
    wl, t = tiny
    s = wl.shape
    fp8 = orc.moe_layer(s, t)
    w16 = orc.moe_layer(s, t, variant="w8a16")
    ex = orc.moe_layer(s, t, variant="exact")
    assert np.array_equal(fp8["ids"], w16["ids"]) and np.array_equal(fp8["ids"], ex["ids"])
    assert np.array_equal(fp8["wts"].view(np.uint32), w16["wts"].view(np.uint32))

    def rel(a):
        return np.linalg.norm(a["y_acc"] - ex["y_acc"]) / np.linalg.norm(ex["y_acc"])

    assert rel(w16) < 1e-2
    assert rel(w16) * 4 < rel(fp8)
