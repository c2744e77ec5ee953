"""Pins for the oracle's LM-head + top-W composition (no GPU).

JetSpec summary on paperlayer.ai, App. E "Training and evaluation details"
(draft model architecture): the draft reuses the frozen target LM head, so
the per-depth draft logits are hidden states times the LM-head matrix; App. E
"Drafting": the proposer keeps the top-k tokens and log-probs per position.

The matmul step is a library primitive; pinned here: one-hot hidden rows
select a column of logits exactly, a hand-worked 2-d example, and agreement
with the already-pinned top-W applied to independently computed logits.
"""
import numpy as np


def bits(x):
    u = np.asarray(x, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def test_one_hot_rows_select_vocab_columns(orc):
    rng = np.random.default_rng(0)
    d, V = 64, 300
    w = np.round(rng.standard_normal((V, d)) * 8) / 8          # exact in bf16
    h = np.zeros((3, d))
    h[0, 5] = 1.0
    h[1, 63] = 2.0
    h[2, 0] = -1.0
    logits = orc.lmhead_logits(bits(h), bits(w))
    np.testing.assert_array_equal(logits[0], w[:, 5])
    np.testing.assert_array_equal(logits[1], 2.0 * w[:, 63])
    np.testing.assert_array_equal(logits[2], -w[:, 0])


def test_hand_example():
    import oracle
    # d = 2, vocab = 4: logits of hidden (1, 2) are w @ (1, 2) = (5, -1, 2.5, 5).
    w = np.array([[1.0, 2.0], [1.0, -1.0], [0.5, 1.0], [3.0, 1.0]])
    tok, logp, logits = oracle.lmhead_topw(bits(np.array([[1.0, 2.0]])), bits(w), 3)
    np.testing.assert_array_equal(logits[0], [5.0, -1.0, 2.5, 5.0])
    assert tok[0].tolist() == [0, 3, 2]                         # tie 5 = 5: lower id first
    z = np.log(2 * np.exp(5.0) + np.exp(-1.0) + np.exp(2.5))
    np.testing.assert_allclose(logp[0], [5.0 - z, 5.0 - z, 2.5 - z], atol=1e-6)


def test_matches_topw_of_independent_logits(orc):
    rng = np.random.default_rng(1)
    d, V, R, W = 256, 5000, 5, 4
    h = rng.standard_normal((R, d)).astype(np.float32)
    w = (rng.standard_normal((V, d)) * 0.05).astype(np.float32)
    hb = (h.view(np.uint32) >> 16).astype(np.uint16)
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    tok, logp, logits = orc.lmhead_topw(hb, wb, W)
    hw = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ww = (wb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.einsum("rd,vd->rv", hw, ww)                        # independent contraction
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    t2, l2 = orc.topw(ref.astype(np.float32)[None], W)
    assert np.array_equal(tok, t2[0]) and np.array_equal(logp, l2[0])
