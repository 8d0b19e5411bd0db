"""Pins of the oracle's number formats: e4m3 (OCP FP8 e4m3fn) and bf16.

The decode is pinned to the format's closed form (landmark values from the OCP
FP8 definition, tests/golden/e4m3_landmarks.txt) and to torch's own
float8_e4m3fn conversion; the encoder to a brute-force nearest-value search.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_landmarks.txt")


def _landmarks():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                code, val = line.split()
                out.append((int(code, 16), val))
    return out


def test_e4m3_landmarks(orc):
    for code, val in _landmarks():
        got = orc.e4m3_decode(np.array([code], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got), hex(code)
        else:
            assert got == float(Fraction(val)), (hex(code), got, val)


def test_e4m3_decode_matches_torch_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(codes[nan].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_roundtrip(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


def _brute_nearest(v, finite_vals, finite_codes):
    """Nearest e4m3 by exhaustive search; ties to the even code; saturating."""
    if v >= 448.0:
        return 0x7E
    if v <= -448.0:
        return 0xFE
    d = np.abs(finite_vals.astype(np.float64) - float(v))
    m = d.min()
    cands = finite_codes[d == m]
    if len(cands) > 1:
        # a tie between two neighbours: keep the even mantissa; for a tie at zero
        # the sign of the input decides between +0 and -0
        if set(cands.tolist()) >= {0x00, 0x80}:
            return 0x80 if math.copysign(1.0, v) < 0 else 0x00
        even = [c for c in cands.tolist() if c % 2 == 0]
        assert len(even) == 1
        return even[0]
    c = int(cands[0])
    if c in (0x00, 0x80):
        return 0x80 if math.copysign(1.0, v) < 0 else 0x00
    return c


def test_e4m3_encode_brute_force(orc):
    finite_codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    finite_vals = orc.e4m3_decode(finite_codes)
    pos = np.sort(np.unique(finite_vals[finite_vals >= 0]))
    mids = (pos[1:].astype(np.float64) + pos[:-1]) / 2.0       # exact in fp32 here
    rng = np.random.default_rng(1)
    sweep = np.concatenate([
        mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
        np.nextafter(mids.astype(np.float32), np.float32(1e9)),
        rng.uniform(-500, 500, 4000), rng.uniform(-1, 1, 4000),
        rng.uniform(-0.02, 0.02, 2000), [0.0, -0.0, 448.0, 449.0, 463.9, 464.0, 1e30, -1e30,
                                         2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]]).astype(np.float32)
    ours = orc.e4m3_encode(sweep)
    for v, c in zip(sweep.tolist(), ours.tolist()):
        assert c == _brute_nearest(v, finite_vals, finite_codes), (v, hex(c))


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 30, 20000), rng.normal(0, 0.01, 5000)]).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(v), ref)


def test_e4m3_encode_nan_and_saturation(orc):
    out = orc.e4m3_encode(np.array([np.nan, np.inf, -np.inf, 1e9, -500.0], np.float32))
    assert out[0] in (0x7F, 0xFF)
    assert out[1:].tolist() == [0x7E, 0xFE, 0x7E, 0xFE]


def _bf16_nearest_exact(v: float) -> int:
    """Nearest bf16 by exact rational comparison of the two neighbours."""
    f = np.float32(v)
    if not math.isfinite(v):
        raise ValueError
    fr = Fraction(v)
    # candidates: bf16 values bracketing v (truncate fp32 toward zero, next up)
    bits = int(np.array([v], np.float32).view(np.uint32)[0]) & 0xFFFF0000
    lo = bits
    hi = bits + 0x10000
    def val(b):
        return Fraction(float(np.array([b], np.uint32).view(np.float32)[0]))
    cands = []
    for b in (lo - 0x10000, lo, hi):
        if b < 0:
            continue
        x = val(b & 0xFFFFFFFF)
        cands.append((abs(x - fr), (b >> 16) & 1, b >> 16))
    cands.sort()
    best = [c for c in cands if c[0] == cands[0][0]]
    if len(best) > 1:
        best = [c for c in best if c[1] == 0]
    return best[0][2]


def test_bf16_rounding(orc):
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-3, 1000)])
    for v in vals.tolist():
        sgn = 0x8000 if v < 0 else 0
        want = _bf16_nearest_exact(abs(v)) | sgn
        assert orc.f64_to_bf16(v) == want, v
    # fp32-representable inputs: a single rounding, which torch also does
    f32 = rng.normal(0, 5, 5000).astype(np.float32)
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = np.array([orc.f64_to_bf16(float(v)) for v in f32], np.uint16)
    assert np.array_equal(ours, ref)
    # ties go to the even mantissa: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.f64_to_bf16(0.0) == 0 and orc.f64_to_bf16(-0.0) == 0x8000


def test_bf16_widening_exact(orc):
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    ours = orc.bf16_to_f32(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok].view(np.uint32), ref[ok].view(np.uint32))
