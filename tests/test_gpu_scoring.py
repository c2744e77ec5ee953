"""GPU per-depth entropy (jt_topw_entropy) and scored expansion
(jt_tree_expand_scored) vs the oracle.

JetSpec summary on paperlayer.ai, App. C "Tree-Drafting Algorithm Ablation"
and App. E "Drafting": cumulative log-prob, entropy-guided and hybrid scores.
Entropy within 2e-4 nats of the fp64 oracle (fp32 online sums over up to
151936 logits); indices and log-probs exactly as jt_topw; expansion fed the
same inputs as the oracle is bit-exact in every mode.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity_util import LOGP_ABS, to_np
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
H_ABS = 2e-4


@pytest.mark.parametrize("batch,N,V,W,sigma", [
    (1, 16, 151936, 4, 3.0), (3, 5, 4096, 1, 3.0), (2, 3, 256, 32, 1.0), (7, 2, 8192, 8, 0.01),
    (1, 1, 4, 3, 1.0), (33, 3, 2048, 4, 30.0), (16, 8, 151936, 4, 3.0)])
def test_topw_entropy_random(batch, N, V, W, sigma):
    rng = np.random.default_rng(V + W + N)
    x = (rng.standard_normal((batch, N, V)) * sigma).astype(np.float32)
    if V >= 8:
        x[0, 0, : V // 3] = -np.inf            # -inf logits contribute nothing
    tok_o, logp_o = oracle.topw(x, W)
    h_o = oracle.row_entropy(x)
    xd = torch.from_numpy(x).to(DEV)
    tok, logp, h = jtree.jt_topw(xd, W, with_entropy=True)
    tok2, logp2 = jtree.jt_topw(xd, W)
    assert np.array_equal(to_np(tok), tok_o)
    assert np.abs(to_np(logp) - logp_o).max() <= LOGP_ABS
    assert np.array_equal(to_np(tok), to_np(tok2)) and np.array_equal(to_np(logp), to_np(logp2))
    assert np.abs(to_np(h) - h_o).max() <= H_ABS, np.abs(to_np(h) - h_o).max()


def test_topw_entropy_closed_forms():
    V = 151936
    x = np.zeros((3, 1, V), np.float32)
    x[1] = -np.inf
    x[1, 0, 5], x[1, 0, 77] = 2.0, -1.0                       # two-point distribution
    x[2] = -np.inf                                             # no distribution: reported 0
    x[2, 0, 0] = -np.inf
    _, _, h = jtree.jt_topw(torch.from_numpy(x[:2]).to(DEV), 2, with_entropy=True)
    h = to_np(h)
    p = 1 / (1 + np.exp(-3.0))
    assert abs(h[0, 0] - np.log(V)) <= H_ABS
    assert abs(h[1, 0] + p * np.log(p) + (1 - p) * np.log(1 - p)) <= 1e-5


@pytest.mark.parametrize("mode,alpha", [(0, 0.0), (1, 0.0), (1, 0.25), (1, 2.0), (2, 0.0)])
@pytest.mark.parametrize("batch,N,W,B", [(4, 4, 2, 16), (3, 16, 4, 256), (5, 8, 4, 64),
                                         (2, 16, 1, 16), (9, 64, 2, 200), (2, 12, 1, 9)])
def test_expand_scored(mode, alpha, batch, N, W, B):
    rng = np.random.default_rng(N * W + B + mode)
    tok = np.stack([np.stack([rng.choice(5000, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    logp[::2] = np.round(logp[::2] * 4) / 4                    # exact score ties
    H = rng.uniform(0.0, 5.0, (batch, N)).astype(np.float32)
    H[0, ::3] = 1.0
    ref = oracle.tree_expand(tok, logp, B, entropy=H, mode=mode, alpha=alpha)
    d = lambda a: torch.from_numpy(a).to(DEV)
    out = jtree.jt_tree_expand(d(tok), d(logp), B, entropy=d(H), mode=mode, alpha=alpha)
    for k in ("parent", "token", "depth", "score", "n_nodes"):
        assert np.array_equal(to_np(out[k]), ref[k]), k


def test_scored_pipeline_on_workload_rows():
    """GPU entropy feeding GPU expansion equals the oracle expansion fed the
    GPU's own candidates and entropy (hybrid, entropy-only)."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((2, 16, 151936)) * 3).astype(np.float32)
    xd = torch.from_numpy(x).to(DEV)
    tok, logp, h = jtree.jt_topw(xd, 4, with_entropy=True)
    for mode, alpha in [(1, 0.5), (2, 0.0)]:
        out = jtree.jt_tree_expand(tok, logp, 128, entropy=h, mode=mode, alpha=alpha)
        ref = oracle.tree_expand(to_np(tok), to_np(logp), 128, entropy=to_np(h), mode=mode,
                                 alpha=alpha)
        for k in ("parent", "token", "depth", "score", "n_nodes"):
            assert np.array_equal(to_np(out[k]), ref[k]), k


def test_scored_host_checks():
    lib = jtree.load()
    z = torch.zeros(64, dtype=torch.int32, device=DEV)
    f = torch.zeros(64, dtype=torch.float32, device=DEV)
    ex = jtree.Exec(DEV).c()
    args = lambda ent, mode, alpha: (z.data_ptr(), f.data_ptr(), ent, 1, 4, 2, 8, mode,
                                     ctypes.c_float(alpha), z.data_ptr(), z.data_ptr(),
                                     z.data_ptr(), f.data_ptr(), z.data_ptr(), ctypes.byref(ex))
    assert lib.jt_tree_expand_scored(*args(f.data_ptr(), 3, 0.0)) == 1       # bad mode
    assert lib.jt_tree_expand_scored(*args(f.data_ptr(), 1, -1.0)) == 1      # negative alpha
    assert lib.jt_tree_expand_scored(*args(None, 2, 0.0)) == 1               # no entropy
    assert lib.jt_topw_entropy(f.data_ptr(), 1, 1, 64, 2, z.data_ptr(), f.data_ptr(), None,
                               ctypes.byref(ex)) == 1
