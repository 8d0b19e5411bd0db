"""GPU parity of moe_greedy_verify against the oracle (bit-exact: integer work
decided by exact comparisons of the same values).

* every accepted-draft count m in 0..7 on a constructed span;
* random spans with a tiny vocabulary (many chance matches and ties);
* a GLM-5.2-sized vocabulary, fp32 and bf16 logits, vector and scalar paths;
* NaN rows, ties, n_draft < 7, R = 0 and a refused R (not a multiple of 8).
"""
import numpy as np
import pytest
import torch

import moe_speculative_verify_gb300 as m
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    m.build()
    m.load()
    oracle.lib()
    torch.cuda.set_device(0)


def _run(logits, draft, n_draft):
    dev = torch.device("cuda")
    lg = logits.to(dev)
    R = lg.shape[0]
    am = torch.empty(R, dtype=torch.int32, device=dev)
    acc = torch.empty(R // 8, dtype=torch.int32, device=dev)
    out = torch.empty(R, dtype=torch.int32, device=dev)
    m.moe_greedy_verify(lg, torch.from_numpy(draft).to(dev), torch.from_numpy(n_draft).to(dev),
                        am, acc, out)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), am.cpu().numpy()


def _check(logits_t, draft, n_draft):
    got = _run(logits_t, draft, n_draft)
    if logits_t.dtype == torch.bfloat16:
        host = logits_t.view(torch.int16).numpy().view(np.uint16)
    else:
        host = logits_t.numpy()
    ref = oracle.greedy_verify(host, draft, n_draft)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)
    return got


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_every_m(dtype):
    rng = np.random.default_rng(30)
    V = 4096
    n_span = 8
    targets = rng.integers(0, V, n_span * 8)
    lg = rng.normal(0, 1, (n_span * 8, V)).astype(np.float32)
    lg[np.arange(n_span * 8), targets] = 10.0
    draft = np.zeros(n_span * 8, np.int32)
    for q in range(n_span):                      # span q accepts exactly q drafts
        for j in range(1, 8):
            t = targets[q * 8 + j - 1]
            draft[q * 8 + j] = t if j <= q else (t + 1) % V
    acc, out, _ = _check(torch.from_numpy(lg).to(dtype), draft, np.full(n_span, 7, np.int32))
    assert acc.tolist() == [q + 1 for q in range(n_span)]


def test_random_small_vocab():
    rng = np.random.default_rng(31)
    R, V = 8 * 300, 6
    lg = rng.integers(-2, 3, (R, V)).astype(np.float32)      # many exact ties
    draft = rng.integers(0, V, R).astype(np.int32)
    nd = rng.integers(0, 8, R // 8).astype(np.int32)
    _check(torch.from_numpy(lg), draft, nd)


@pytest.mark.parametrize("V,dtype", [(151552, torch.bfloat16), (151552, torch.float32),
                                     (151553, torch.bfloat16), (1001, torch.float32)])
def test_large_vocab_and_scalar_paths(V, dtype):
    rng = np.random.default_rng(V)
    R = 16
    lg = torch.from_numpy(rng.normal(0, 3, (R, V)).astype(np.float32)).to(dtype)
    lg[2, :] = float("nan")
    lg[3, 17] = float("nan")
    lg[4, 5] = lg[4, 9] = lg[4].float().max() + 1        # a tie at the maximum
    am_ref = oracle.greedy_verify(lg.view(torch.int16).numpy().view(np.uint16)
                                  if dtype == torch.bfloat16 else lg.numpy(),
                                  np.zeros(R, np.int32), np.zeros(2, np.int32))[2]
    draft = np.zeros(R, np.int32)
    draft[1:4] = am_ref[0:3]                            # span 0 accepts 3 drafts
    _check(lg, draft, np.array([7, 5], np.int32))


def test_refusals():
    dev = torch.device("cuda")
    lg = torch.zeros((12, 10), device=dev)
    z = torch.zeros(12, dtype=torch.int32, device=dev)
    with pytest.raises(m.MoeError):
        m.moe_greedy_verify(lg, z, z, z, z, z)
    m.moe_greedy_verify(torch.zeros((0, 10), device=dev), z, z, z, z, z)
