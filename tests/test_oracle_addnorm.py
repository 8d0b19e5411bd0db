"""Pins of the oracle's residual add + RMSNorm.

* torch.nn.functional.rms_norm (a library routine) on the fp64 sum;
* closed forms: a constant row normalises to gamma * c / sqrt(c^2 + eps); a zero
  row stays zero; scaling the row scales residual_out and leaves normed alone;
* pad rows give zeros in both outputs.
"""
import numpy as np
import torch


def _bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_matches_torch_rms_norm(orc):
    rng = np.random.default_rng(50)
    R, H = 6, 512
    y = rng.normal(0, 0.3, (R, H))
    res = torch.from_numpy(rng.normal(0, 1, (R, H)).astype(np.float32)).to(torch.bfloat16)
    gamma = rng.uniform(0.5, 1.5, H).astype(np.float32)
    ro, no = orc.add_rmsnorm(y, _bits(res), gamma, 1e-5)
    z = res.double() + torch.from_numpy(y)
    ref = torch.nn.functional.rms_norm(z, (H,), weight=torch.from_numpy(gamma).double(), eps=1e-5)
    assert np.array_equal(ro, _bits(z))
    assert np.array_equal(no, _bits(ref))


def test_closed_forms(orc):
    H = 256
    gamma = np.linspace(0.5, 2.0, H).astype(np.float32)
    res = np.zeros((3, H), np.uint16)                     # bf16 zeros
    y = np.zeros((3, H))
    y[0] = 3.0                                            # constant row
    y[2] = 1e-3 * np.arange(H)
    ro, no = orc.add_rmsnorm(y, res, gamma, 1e-6)
    expect = gamma.astype(np.float64) * 3.0 / np.sqrt(9.0 + 1e-6)
    assert np.array_equal(no[0], _bits(torch.from_numpy(expect)))
    assert np.all(no[1] == 0) and np.all(ro[1] == 0)      # a zero row stays zero
    ro2, no2 = orc.add_rmsnorm(y * 8.0, res, gamma, 0.0)  # scale invariance (eps = 0)
    _, no3 = orc.add_rmsnorm(y, res, gamma, 0.0)
    assert np.array_equal(no2[[0, 2]], no3[[0, 2]])


def test_pads_zero(orc):
    R, H = 4, 128
    y = np.full((R, H), np.nan)
    res = np.full((R, H), 0x7FC0, np.uint16)              # NaN residual on the pad
    valid = np.array([0, 1, 0, 1], np.uint8)
    y[1] = 1.0
    y[3] = 2.0
    res[1] = 0
    res[3] = 0
    ro, no = orc.add_rmsnorm(y, res, np.ones(H, np.float32), 1e-5, valid)
    assert np.all(ro[[0, 2]] == 0) and np.all(no[[0, 2]] == 0)
    assert np.all(np.isfinite(ro[[1, 3]].astype(np.float32)))
