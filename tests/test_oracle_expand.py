"""Pins for the oracle's best-first tree expansion.

Algorithm: JetSpec summary on paperlayer.ai, App. B "Tree-Drafting Algorithm
Details" (Algorithm 1) and §2 "Tree Construction and Verification"; the
Chinese summary on paper.rainbus.top, "方法步骤详情". Score: cumulative draft
log-probability (JetSpec review on startedourmission.github.io, "How it
works", s(π(v)) equation; paperlayer.ai App. C: the production default).

Independent checks: a linear-rescan implementation (no heap), the "best-first
= top-K of the virtual tree" characterisation by enumeration, closed-form tree
shapes, hand-worked golden cases and ordering invariants.
"""
import itertools
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def expand_rescan(tok, logp, B):
    """Best-first expansion with a plain list and a linear scan for the max."""
    N, W = tok.shape
    frontier = [(np.float32(0.0), -1, 0)]  # (score, id, depth); the root
    nodes = []                              # (parent, token, depth, score)
    while len(nodes) < B and frontier:
        best = max(range(len(frontier)), key=lambda i: (frontier[i][0], -frontier[i][1]))
        s, u, d = frontier.pop(best)
        for r in range(W):
            if len(nodes) == B:
                break
            v = len(nodes)
            sc = np.float32(s + np.float32(logp[d, r]))
            nodes.append((u, int(tok[d, r]), d + 1, sc))
            if d + 1 < N:
                frontier.append((sc, v, d + 1))
    return nodes


def random_draft(rng, batch, N, W, V=1000):
    tok = np.stack([np.stack([rng.choice(V, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    return tok, logp


@pytest.mark.parametrize("N,W,B", [(4, 2, 16), (16, 4, 256), (8, 4, 64), (16, 1, 16), (3, 3, 200),
                                   (16, 4, 128), (5, 7, 100), (2, 8, 3)])
def test_expand_matches_linear_rescan(orc, N, W, B):
    rng = np.random.default_rng(N * 100 + W * 10 + B)
    batch = 6
    tok, logp = random_draft(rng, batch, N, W)
    # Quantised log-probs produce many exact score ties, exercising the id order.
    logp[::2] = np.round(logp[::2] * 4) / 4
    out = orc.tree_expand(tok, logp, B)
    for b in range(batch):
        ref = expand_rescan(tok[b], logp[b], B)
        n = len(ref)
        assert out["n_nodes"][b] == n
        assert out["parent"][b, :n].tolist() == [r[0] for r in ref]
        assert out["token"][b, :n].tolist() == [r[1] for r in ref]
        assert out["depth"][b, :n].tolist() == [r[2] for r in ref]
        assert np.array_equal(out["score"][b, :n], np.array([r[3] for r in ref], np.float32))
        assert (out["parent"][b, n:] == -1).all() and (out["token"][b, n:] == -1).all()
        assert (out["depth"][b, n:] == 0).all() and (out["score"][b, n:] == 0).all()


@pytest.mark.parametrize("N,W,B", [(4, 2, 9), (3, 3, 20), (5, 2, 40), (3, 2, 14), (6, 2, 30)])
def test_expand_is_top_k_of_the_virtual_tree(orc, N, W, B):
    """Best-first pops the virtual tree's expandable nodes in descending score."""
    rng = np.random.default_rng(N + W + B)
    tok, logp = random_draft(rng, 1, N, W)
    out = orc.tree_expand(tok, logp, B)
    n = int(out["n_nodes"][0])
    # Every rank path of length < N (root = empty path) with its fp32 score.
    virt = []
    for d in range(0, N):
        for path in itertools.product(range(W), repeat=d):
            s = np.float32(0.0)
            for i, r in enumerate(path):
                s = np.float32(s + logp[0, i, r])
            virt.append((float(s), path))
    virt.sort(key=lambda e: -e[0])
    # Expected tree: children of the popped paths, in pop order, cut at B.
    want = []
    for _, path in virt:
        if len(want) >= B:
            break
        for r in range(W):
            if len(want) >= B:
                break
            want.append(path + (r,))
    # Rank path of each oracle node.
    par, tk, dp = out["parent"][0], out["token"][0], out["depth"][0]
    got = []
    for v in range(n):
        r = int(np.nonzero(tok[0, dp[v] - 1] == tk[v])[0][0])
        got.append((got[par[v]] if par[v] >= 0 else ()) + (r,))
    assert got == want[:n]


def test_expand_closed_form_shapes(orc):
    rng = np.random.default_rng(5)
    # W = 1: a chain of min(B, N) nodes carrying each depth's rank-0 token.
    for N, B in [(16, 16), (4, 16), (16, 5)]:
        tok, logp = random_draft(rng, 1, N, 1)
        out = orc.tree_expand(tok, logp, B)
        n = min(B, N)
        assert out["n_nodes"][0] == n
        assert out["parent"][0, :n].tolist() == [-1] + list(range(n - 1))
        assert out["token"][0, :n].tolist() == tok[0, :n, 0].tolist()
        assert out["depth"][0, :n].tolist() == list(range(1, n + 1))
    # B >= sum_d W^d: the complete W-ary tree of depth N.
    for N, W in [(3, 3), (4, 2), (2, 8)]:
        tok, logp = random_draft(rng, 1, N, W)
        full = sum(W ** d for d in range(1, N + 1))
        out = orc.tree_expand(tok, logp, full + 7)
        assert out["n_nodes"][0] == full
        counts = np.bincount(out["depth"][0, :full], minlength=N + 1)
        assert counts.tolist() == [0] + [W ** d for d in range(1, N + 1)]
    # B < W: only the root's top-B children.
    tok, logp = random_draft(rng, 1, 4, 8)
    out = orc.tree_expand(tok, logp, 3)
    assert out["parent"][0].tolist() == [-1, -1, -1]
    assert out["token"][0].tolist() == tok[0, 0, :3].tolist()


def test_expand_order_invariants(orc):
    rng = np.random.default_rng(9)
    N, W, B = 16, 4, 256
    tok, logp = random_draft(rng, 8, N, W)
    out = orc.tree_expand(tok, logp, B)
    for b in range(8):
        n = out["n_nodes"][b]
        par, sc, dp = out["parent"][b, :n], out["score"][b, :n], out["depth"][b, :n]
        # Pop order = order in which parents first appear; their scores never rise.
        popped = list(dict.fromkeys(par.tolist()))
        pop_scores = [0.0 if u < 0 else sc[u] for u in popped]
        assert all(a >= c for a, c in zip(pop_scores, pop_scores[1:]))
        # Every popped node scores at least as high as any expandable node left unpopped.
        left = [v for v in range(n) if dp[v] < N and v not in set(popped)]
        if left:
            assert min(pop_scores) >= max(sc[v] for v in left)
        # Score = sum of the path's log-probs (float64 sum, within fp32 rounding).
        for v in range(n):
            s, u = 0.0, v
            while u >= 0:
                r = int(np.nonzero(tok[b, dp[u] - 1] == out["token"][b, u])[0][0])
                s += float(logp[b, dp[u] - 1, r])
                u = par[u]
            assert abs(s - sc[v]) <= 1e-5 * max(1.0, abs(s))


def read_golden():
    cases, cur = [], None
    for raw in open(os.path.join(GOLDEN, "expand_examples.txt")):
        line = raw.split("#")[0].strip()
        if not line:
            continue
        if line.startswith("case"):
            cur = {"rows": []}
            cases.append(cur)
            continue
        cur["rows"].append(line)
    out = []
    for c in cases:
        W, N, B = map(int, c["rows"][0].split())
        tok = np.zeros((1, N, W), np.int32)
        logp = np.zeros((1, N, W), np.float32)
        for d in range(N):
            t, p = c["rows"][1 + d].split("|")
            tok[0, d] = [int(x) for x in t.split()]
            logp[0, d] = [float(x) for x in p.split()]
        exp = {}
        for line in c["rows"][1 + N:]:
            key, *vals = line.split()
            exp[key] = [float(x) if key == "score" else int(x) for x in vals]
        out.append((tok, logp, B, exp))
    return out


def test_expand_golden_examples(orc):
    cases = read_golden()
    assert len(cases) == 5
    for tok, logp, B, exp in cases:
        out = orc.tree_expand(tok, logp, B)
        n = len(exp["parent"])
        assert out["n_nodes"][0] == n
        for key in ("parent", "token", "depth"):
            assert out[key][0, :n].tolist() == exp[key]
        assert out["score"][0, :n].tolist() == exp["score"]
