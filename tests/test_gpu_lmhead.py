"""GPU LM head fused with top-W (jt_lmhead_topw) vs the oracle.

JetSpec summary on paperlayer.ai, App. E: the draft reuses the frozen target
LM head; the proposer keeps the top-k tokens and log-probs per position.

Exact case: small dyadic values make every product and every fp32 partial
sum exact, so the GPU's logits equal the oracle's and indices (with their
many ties) must match bit for bit. Random case: the GPU sums in fp32 in the
tensor cores' order, so a returned token must be within the rounding
allowance of the oracle's W-th best logit and its log-prob within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import LOGP_ABS, to_np
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_bf16_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(DEV).to(torch.bfloat16)


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rows,d,V,W", [(1, 64, 1000, 1), (16, 512, 4096, 4), (130, 256, 5000, 8),
                                        (257, 128, 1536, 32), (3, 4096, 151936, 4)])
def test_lmhead_exact_values(rows, d, V, W):
    rng = np.random.default_rng(rows + d + V)
    h = rng.integers(-2, 3, (rows, d)) / 4.0
    w = rng.integers(-4, 5, (V, d)) / 8.0
    hd, wd = to_bf16_dev(h), to_bf16_dev(w)
    tok, logp, ent = jtree.jt_lmhead_topw(hd, wd, W, with_entropy=True)
    tok_o, logp_o, logits = oracle.lmhead_topw(bits_of(hd), bits_of(wd), W)
    assert np.array_equal(to_np(tok), tok_o)
    assert np.abs(to_np(logp) - logp_o).max() <= LOGP_ABS
    h_o = oracle.row_entropy(logits.astype(np.float32))
    assert np.abs(to_np(ent) - h_o).max() <= 2e-4


@pytest.mark.parametrize("rows,d,V,W", [(16, 4096, 151936, 4), (257, 1024, 20000, 4),
                                        (64, 2048, 32768, 16)])
def test_lmhead_random_values(rows, d, V, W):
    rng = np.random.default_rng(rows * 3 + V)
    h = rng.standard_normal((rows, d)).astype(np.float32)
    w = (rng.standard_normal((V, d)) * 0.02).astype(np.float32)
    hd, wd = to_bf16_dev(h), to_bf16_dev(w)
    tok, logp = jtree.jt_lmhead_topw(hd, wd, W)
    tok, logp = to_np(tok), to_np(logp)
    _, _, logits = oracle.lmhead_topw(bits_of(hd), bits_of(wd), W)
    # fp32 sums of d exact products: error below d * 2^-24 * sum |terms| (loose bound).
    hw = (bits_of(hd).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ww = (bits_of(wd).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    allow = 1e-6 * np.abs(hw).max(axis=1, keepdims=True) * np.abs(ww).sum(axis=1).max() + 1e-6
    lse = np.log(np.exp(logits - logits.max(1, keepdims=True)).sum(1)) + logits.max(1)
    kth = -np.sort(-logits, axis=1)[:, W - 1]
    for r in range(rows):
        assert len(set(tok[r].tolist())) == W
        got = logits[r, tok[r]]
        assert (got >= kth[r] - 2 * allow[r, 0]).all(), r
        assert (np.diff(got) <= 2 * allow[r, 0]).all(), r     # non-increasing up to rounding
        np.testing.assert_allclose(logp[r], got - lse[r], atol=2e-3)
