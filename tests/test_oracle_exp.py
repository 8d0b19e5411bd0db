"""Pins of the oracle's own exp / sigmoid (Cody-Waite reduction + Taylor series).

The routing sigmoid uses an exp written from a published method so that the
CPU oracle and the GPU router can follow one IEEE op sequence.  Pinned here
against math.exp in double precision (error in fp32 ulps) and exact special
values.
"""
import math

import numpy as np


def _ulp32(x: float) -> float:
    f = np.float32(abs(x))
    return float(np.nextafter(f, np.float32(np.inf)) - f)


def test_own_exp_accuracy(orc):
    rng = np.random.default_rng(4)
    pts = np.concatenate([np.linspace(-87.0, 87.0, 60001), rng.uniform(-87, 87, 20000),
                          rng.uniform(-3, 3, 20000)]).astype(np.float32)
    worst = 0.0
    for a in pts.tolist():
        got = orc.own_exp(a)
        ref = math.exp(a)
        err = abs(got - ref) / _ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst


def test_own_exp_special_values(orc):
    assert orc.own_exp(0.0) == 1.0
    assert orc.own_exp(1.0) == float(np.float32(math.e)) or \
        abs(orc.own_exp(1.0) - math.e) <= _ulp32(math.e)
    for n in range(-20, 21):
        a = float(np.float32(n * math.log(2.0)))      # the argument is an fp32
        v = orc.own_exp(a)
        assert abs(v - math.exp(a)) <= 2 * _ulp32(math.exp(a))
    # clamped range: stays finite and normal
    assert orc.own_exp(200.0) == orc.own_exp(87.0)
    assert orc.own_exp(-200.0) == orc.own_exp(-87.0) > np.finfo(np.float32).tiny
    assert math.isnan(orc.own_exp(float("nan")))


def test_sigmoid(orc):
    assert orc.sigmoid(0.0) == 0.5
    xs = np.linspace(-20, 20, 4001, dtype=np.float32)
    s = np.array([orc.sigmoid(float(x)) for x in xs])
    assert np.all(np.diff(s) >= 0)
    ref = 1.0 / (1.0 + np.exp(-xs.astype(np.float64)))
    assert np.max(np.abs(s - ref) / ref) < 4e-7
    assert orc.sigmoid(100.0) == 1.0
    assert 0.0 < orc.sigmoid(-100.0) < 1e-37
