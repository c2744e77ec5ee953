"""Pins for the oracle's per-depth entropy and scored expansion (no GPU).

JetSpec summary on paperlayer.ai, App. C "Tree-Drafting Algorithm Ablation"
and App. E "Drafting": the proposer supports cumulative log-prob, entropy-
guided and hybrid scores; the hybrid weight alpha interpolates between the
two (alpha -> 0: cumulative log-prob, alpha -> inf: entropy only). Reading
used here: a child's score increment is logp - alpha*H_d (hybrid) or -H_d
(entropy only), H_d the entropy of depth d's draft distribution.

Entropy: closed forms (uniform, two-point), scipy's entropy of scipy's
softmax (independent library routines), shift invariance, -inf entries.
Scored expansion: a linear-rescan implementation with the same increments,
the alpha = 0 limit, and the level-order shape of entropy-only scoring.
"""
import numpy as np
import pytest

from test_oracle_expand import random_draft


@pytest.mark.parametrize("V", [1, 2, 7, 1024, 151936])
def test_entropy_uniform(orc, V):
    x = np.full((2, V), 0.25, np.float32)
    np.testing.assert_allclose(orc.row_entropy(x), np.log(V), rtol=0, atol=2e-6 * max(1, np.log(V)))


def test_entropy_two_point(orc):
    V = 4096
    for a, b in [(0.0, 0.0), (3.0, -1.0), (10.0, 0.0), (-2.5, 1.25)]:
        x = np.full((1, V), -np.inf, np.float32)
        x[0, 17], x[0, 4000] = a, b
        p = 1.0 / (1.0 + np.exp(-(a - b)))
        want = -(p * np.log(p) + (1 - p) * np.log(1 - p))
        np.testing.assert_allclose(orc.row_entropy(x)[0], want, rtol=1e-6, atol=1e-7)


def test_entropy_matches_scipy(orc):
    stats = pytest.importorskip("scipy.stats")
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(5)
    for V, sigma in [(1000, 3.0), (151936, 3.0), (50, 0.01), (4096, 30.0)]:
        x = (rng.standard_normal((3, V)) * sigma).astype(np.float32)
        want = stats.entropy(special.softmax(x.astype(np.float64), axis=-1), axis=-1)
        np.testing.assert_allclose(orc.row_entropy(x), want, rtol=2e-6, atol=1e-6)


def test_entropy_invariants(orc):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((4, 3000)) * 2).astype(np.float32)
    h = orc.row_entropy(x)
    np.testing.assert_allclose(orc.row_entropy(x + np.float32(7.0)), h, rtol=1e-5)
    assert (h >= 0).all() and (h <= np.log(3000) + 1e-6).all()
    y = np.concatenate([x, np.full((4, 500), -np.inf, np.float32)], axis=1)
    np.testing.assert_allclose(orc.row_entropy(y), h, rtol=1e-6)
    assert orc.row_entropy(np.full((1, 8), -np.inf, np.float32))[0] == 0.0


def expand_rescan_scored(tok, logp, H, B, mode, alpha):
    """Linear-rescan best-first expansion with the scored increments."""
    N, W = tok.shape
    def inc(d, r):
        if mode == 0:
            return np.float32(logp[d, r])
        if mode == 1:
            return np.float32(np.float32(logp[d, r]) - np.float32(np.float32(alpha) * H[d]))
        return np.float32(-H[d])
    frontier = [(np.float32(0.0), -1, 0)]
    nodes = []
    while len(nodes) < B and frontier:
        best = max(range(len(frontier)), key=lambda i: (frontier[i][0], -frontier[i][1]))
        s, u, d = frontier.pop(best)
        for r in range(W):
            if len(nodes) == B:
                break
            v = len(nodes)
            sc = np.float32(s + inc(d, r))
            nodes.append((u, int(tok[d, r]), d + 1, sc))
            if d + 1 < N:
                frontier.append((sc, v, d + 1))
    return nodes


@pytest.mark.parametrize("mode,alpha", [(1, 0.5), (1, 3.0), (1, 1e-3), (2, 0.0)])
@pytest.mark.parametrize("N,W,B", [(4, 2, 16), (8, 4, 64), (16, 1, 16), (5, 3, 60)])
def test_scored_matches_linear_rescan(orc, mode, alpha, N, W, B):
    rng = np.random.default_rng(N + W + B + mode)
    batch = 5
    tok, logp = random_draft(rng, batch, N, W)
    H = rng.uniform(0.0, 4.0, (batch, N)).astype(np.float32)
    H[0, ::2] = 1.0                              # exact ties across depths
    out = orc.tree_expand(tok, logp, B, entropy=H, mode=mode, alpha=alpha)
    for b in range(batch):
        ref = expand_rescan_scored(tok[b], logp[b], H[b], B, mode, alpha)
        n = len(ref)
        assert out["n_nodes"][b] == n
        assert out["parent"][b, :n].tolist() == [r[0] for r in ref]
        assert out["token"][b, :n].tolist() == [r[1] for r in ref]
        assert np.array_equal(out["score"][b, :n], np.array([r[3] for r in ref], np.float32))


def test_hybrid_alpha_zero_is_cumulative_logp(orc):
    rng = np.random.default_rng(7)
    tok, logp = random_draft(rng, 4, 16, 4)
    H = rng.uniform(0.0, 5.0, (4, 16)).astype(np.float32)
    a = orc.tree_expand(tok, logp, 256)
    b = orc.tree_expand(tok, logp, 256, entropy=H, mode=1, alpha=0.0)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("N,W,B", [(4, 2, 30), (3, 4, 50), (6, 3, 100), (16, 4, 256)])
def test_entropy_only_is_level_order(orc, N, W, B):
    """Entropy-only scores are equal within a depth and fall with depth (H >= 0),
    so ties go to creation order: the tree is the complete W-ary tree in level
    order, node v >= W being a child of node v // W - 1, until the budget or
    depth N ends it."""
    rng = np.random.default_rng(N * W)
    tok, logp = random_draft(rng, 2, N, W)
    H = rng.uniform(0.0, 3.0, (2, N)).astype(np.float32)
    out = orc.tree_expand(tok, logp, B, entropy=H, mode=2)
    full = sum(W ** d for d in range(1, N + 1))
    n = min(B, full)
    for b in range(2):
        assert out["n_nodes"][b] == n
        par = out["parent"][b, :n]
        assert (par[:W] == -1).all()
        assert (par[W:] == np.arange(W, n) // W - 1).all()
        depth = out["depth"][b, :n]
        assert (np.diff(depth) >= 0).all()
        # Score of a depth-d node: the binary32 running sum 0 - H_1 - ... - H_d.
        run = [np.float32(0.0)]
        for d in range(N):
            run.append(np.float32(run[-1] + np.float32(-H[b, d])))
        np.testing.assert_array_equal(out["score"][b, :n], [run[d] for d in depth])
