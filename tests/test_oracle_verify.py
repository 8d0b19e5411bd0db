"""Pins of the oracle's greedy verify + acceptance (spans of 8 rows).

* argmax: against numpy's argmax (first maximal index) on fp32 and bf16 logits;
* acceptance: for every m in 0..7 a constructed span whose first m drafts
  match and the next one does not (or all match) gives accept_len m+1, the m
  drafts, then the target's token at row m; brute force over every prefix;
* n_draft < 7: rows beyond the drafts are never accepted.
"""
import numpy as np
import torch


def _logits_with_argmax(targets, V, rng):
    lg = rng.normal(0, 1, (len(targets), V)).astype(np.float32)
    for r, t in enumerate(targets):
        lg[r, t] = lg[r].max() + 1.0
    return lg


def test_argmax_ties_and_dtypes(orc):
    rng = np.random.default_rng(20)
    V = 1000
    lg = rng.normal(0, 1, (16, V)).astype(np.float32)
    lg[3, [5, 900]] = 50.0                    # a tie: the lower index wins
    lg[4, 0] = np.nan                         # NaN never wins
    lg[5, :] = np.nan                         # an all-NaN row gives index 0
    lg[6, :] = -np.inf
    _, _, am = orc.greedy_verify(lg, np.zeros(16, np.int32), np.zeros(2, np.int32))
    ref = np.argmax(np.where(np.isnan(lg), -np.inf, lg), axis=1)
    assert np.array_equal(am, ref) and am[3] == 5 and am[5] == 0 and am[6] == 0
    bf = torch.from_numpy(lg).to(torch.bfloat16)
    bits = bf.view(torch.int16).numpy().view(np.uint16)
    _, _, am2 = orc.greedy_verify(bits, np.zeros(16, np.int32), np.zeros(2, np.int32))
    f = bf.float().numpy()
    assert np.array_equal(am2, np.argmax(np.where(np.isnan(f), -np.inf, f), axis=1))


def test_acceptance_every_m(orc):
    rng = np.random.default_rng(21)
    V = 300
    for m in range(8):
        targets = rng.integers(0, V, 8)
        draft = np.zeros(8, np.int32)
        for j in range(1, 8):
            draft[j] = targets[j - 1] if j <= m else (targets[j - 1] + 1) % V
        lg = _logits_with_argmax(targets, V, rng)
        acc, out, _ = orc.greedy_verify(lg, draft, np.array([7], np.int32))
        assert acc[0] == m + 1
        assert out[:m].tolist() == draft[1:m + 1].tolist()
        assert out[m] == targets[m]
        assert np.all(out[m + 1:] == -1)


def test_acceptance_brute_force(orc):
    rng = np.random.default_rng(22)
    V = 5                                     # small vocab: many chance matches
    n_span = 200
    targets = rng.integers(0, V, n_span * 8)
    draft = rng.integers(0, V, n_span * 8).astype(np.int32)
    nd = rng.integers(0, 8, n_span).astype(np.int32)
    lg = _logits_with_argmax(targets, V, rng)
    acc, out, _ = orc.greedy_verify(lg, draft, nd)
    for q in range(n_span):
        t = targets[q * 8:(q + 1) * 8]
        d = draft[q * 8:(q + 1) * 8]
        best = 0
        for m in range(nd[q] + 1):            # the longest prefix whose drafts all match
            if all(d[j] == t[j - 1] for j in range(1, m + 1)):
                best = m
        assert acc[q] == best + 1
        assert list(out[q * 8:q * 8 + best]) == list(d[1:best + 1])
        assert out[q * 8 + best] == t[best]
