"""Pins for the oracle's per-depth top-W extraction.

What is pinned (JetSpec summary on paperlayer.ai, App. E "Drafting": top-k
tokens and their log-probabilities at each future position; the Chinese
summary on paper.rainbus.top, "方法步骤详情": top-W candidates per depth):
  * indices = the first W of a stable descending sort (numpy's argsort);
  * log-probabilities = log-softmax over the full vocabulary (scipy);
  * with W = V the probabilities sum to one.
"""
import numpy as np
import pytest
from scipy.special import log_softmax


@pytest.mark.parametrize("batch,N,V,W,sigma", [(2, 3, 1024, 4, 3.0), (1, 5, 4096, 8, 10.0),
                                               (3, 2, 64, 1, 0.1), (1, 1, 151936, 32, 3.0)])
def test_topw_against_library_sort_and_log_softmax(orc, batch, N, V, W, sigma):
    rng = np.random.default_rng(V + W)
    x = (rng.standard_normal((batch, N, V)) * sigma).astype(np.float32)
    tok, logp = orc.topw(x, W)
    order = np.argsort(-x, axis=-1, kind="stable")[..., :W]
    assert np.array_equal(tok, order)
    ls = log_softmax(x.astype(np.float64), axis=-1)
    ref = np.take_along_axis(ls, order, -1)
    # fp64 result rounded once to fp32: within half an ulp of |logp|.
    np.testing.assert_allclose(logp, ref, rtol=2 ** -24, atol=1e-30)
    assert (np.diff(logp, axis=-1) <= 0).all()


def test_topw_full_vocab_is_a_sorted_distribution(orc):
    rng = np.random.default_rng(3)
    V = 2048
    x = (rng.standard_normal((2, 2, V)) * 3).astype(np.float32)
    tok, logp = orc.topw(x, V)
    for row in tok.reshape(-1, V):
        assert np.array_equal(np.sort(row), np.arange(V))
    total = np.exp(logp.astype(np.float64)).sum(-1)
    np.testing.assert_allclose(total, 1.0, atol=1e-5)


def test_topw_ties_rank_lower_index_first(orc):
    x = np.zeros((1, 1, 16), np.float32)
    x[0, 0, [3, 9, 12]] = 2.0
    x[0, 0, [1, 14]] = 1.0
    x[0, 0, 5] = -0.0  # equal to +0.0
    tok, logp = orc.topw(x, 7)
    assert tok[0, 0].tolist() == [3, 9, 12, 1, 14, 0, 2]
    assert logp[0, 0, 0] == logp[0, 0, 1] == logp[0, 0, 2]


def test_topw_negative_infinity_entries(orc):
    V = 32
    x = np.full((1, 1, V), -np.inf, np.float32)
    x[0, 0, 7] = 0.0
    x[0, 0, 20] = 0.0
    tok, logp = orc.topw(x, 3)
    assert tok[0, 0, :2].tolist() == [7, 20]
    np.testing.assert_allclose(logp[0, 0, :2], np.log(0.5), rtol=1e-7)
    assert tok[0, 0, 2] == 0 and logp[0, 0, 2] == -np.inf


def test_topw_rejects_w_above_vocab(orc):
    with pytest.raises(orc.OracleError):
        orc.topw(np.zeros((1, 1, 4), np.float32), 5)
