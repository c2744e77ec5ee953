"""Pins for the oracle's greedy tree acceptance.

Rule: JetSpec summary on paperlayer.ai, §2 "Tree Construction and
Verification" (accept the longest prefix whose draft tokens satisfy the
target's condition); Chinese summary on paper.rainbus.top, "前置知识" (keep the
longest prefix consistent with the target, expected committed tokens
(1-α^{N+1})/(1-α)); JetSpec++ summary on paperlayer.ai, §3 "Preliminaries"
(the accepted prefix plus one bonus token is committed; τ counts committed
tokens per round) and App. E (speculative output equals AR output token by
token).
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_valid_paths(parent, token, n, target):
    """Every root path whose tokens each equal numpy's argmax at the parent."""
    best = None
    am = np.argmax(target, axis=-1)  # first maximum = lowest token id
    children = {u: [v for v in range(n) if parent[v] == u] for u in range(-1, n)}
    stack = [(-1, [])]
    while stack:
        u, path = stack.pop()
        if best is None or len(path) > len(best):
            best = path
        for c in children[u]:
            if token[c] == am[0 if u < 0 else 1 + u]:
                stack.append((c, path + [c]))
    return best, am


def biased_targets(rng, parent, token, n, B, V, p_match=0.7, p_tie=0.2):
    t = rng.standard_normal((B + 1, V)).astype(np.float32)
    for u in range(-1, B):
        row = t[0 if u < 0 else 1 + u]
        kids = [v for v in range(n) if parent[v] == u]
        if kids and rng.random() < p_match:
            row[token[rng.choice(kids)]] = row.max() + 1
        if rng.random() < p_tie:
            j = int(np.argmax(row))
            row[rng.integers(V)] = row[j]
    return t


@pytest.mark.parametrize("N,W,B,V", [(4, 2, 16, 32), (16, 4, 64, 64), (16, 1, 16, 16),
                                     (8, 4, 64, 256), (3, 3, 30, 12)])
def test_accept_is_the_longest_valid_root_path(orc, N, W, B, V):
    rng = np.random.default_rng(N * W + B)
    batch = 40
    tok = np.stack([np.stack([rng.choice(V, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    tree = orc.tree_expand(tok, logp, B)
    target = np.stack([biased_targets(rng, tree["parent"][b], tree["token"][b],
                                      tree["n_nodes"][b], B, V) for b in range(batch)])
    out = orc.tree_accept(target, tree["parent"], tree["token"], tree["n_nodes"], N)
    lens = []
    for b in range(batch):
        path, am = all_valid_paths(tree["parent"][b], tree["token"][b], tree["n_nodes"][b],
                                   target[b])
        k = len(path)
        lens.append(k)
        assert out["acc_len"][b] == k
        assert out["acc_nodes"][b, :k].tolist() == path
        assert (out["acc_nodes"][b, k:] == -1).all() and (out["acc_tokens"][b, k:] == -1).all()
        # AR equivalence: committed tokens are the target's greedy chain along the path.
        chain = [int(am[0])] + [int(am[1 + v]) for v in path]
        assert out["acc_tokens"][b, :k].tolist() == chain[:k]
        assert out["bonus"][b] == chain[k]
    assert max(lens) >= 2  # the biased targets do produce multi-token acceptances


@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.9])
@pytest.mark.parametrize("N", [4, 16])
def test_expected_committed_tokens_closed_form(orc, alpha, N):
    """Chains with i.i.d. Bernoulli(alpha) agreement: E[acc_len + 1] = (1-α^{N+1})/(1-α)."""
    rng = np.random.default_rng(int(alpha * 10) + N)
    trials, V = 20000, 8
    parent = np.tile(np.array([-1] + list(range(N - 1)), np.int32), (trials, 1))
    token = rng.integers(0, V, (trials, N)).astype(np.int32)
    target = np.zeros((trials, N + 1, V), np.float32)
    agree = rng.random((trials, N + 1)) < alpha
    nxt = np.concatenate([token, np.zeros((trials, 1), np.int32)], 1)  # row d predicts token d
    other = (nxt + 1 + rng.integers(0, V - 1, nxt.shape)) % V          # any token but the next
    choice = np.where(agree, nxt, other)
    choice[:, N] = rng.integers(0, V, trials)                          # below the leaf: free
    np.put_along_axis(target, choice[..., None], 1.0, axis=-1)
    out = orc.tree_accept(target, parent, token, np.full(trials, N, np.int32), N)
    committed = out["acc_len"].astype(np.float64) + 1
    expect = (1 - alpha ** (N + 1)) / (1 - alpha)
    se = committed.std() / np.sqrt(trials)
    assert abs(committed.mean() - expect) <= 4 * se + 1e-12


def test_accept_golden_examples(orc):
    lines = [l.split("#")[0].strip() for l in open(os.path.join(GOLDEN, "accept_examples.txt"))]
    lines = [l for l in lines if l]
    par_s, tok_s = lines[0][len("tree"):].split("|")
    parent = np.array([int(x) for x in par_s.split()], np.int32)
    token = np.array([int(x) for x in tok_s.split()], np.int32)
    B, V, N = len(parent), 64, 4
    cases = lines[1:]
    assert len(cases) == 5
    for line in cases:
        fields = [f.strip() for f in line[len("case"):].split("|")]
        target = np.zeros((B + 1, V), np.float32)
        for spec in fields[0].split()[1:]:
            r, toks = spec.split(":")
            for t in toks.split(","):
                target[int(r), int(t)] = 1.0
        exp_len = int(fields[1].split()[1])
        exp_nodes = [int(x) for x in fields[2].split()[1:]]
        exp_tokens = [int(x) for x in fields[3].split()[1:]]
        exp_bonus = int(fields[4].split()[1])
        out = orc.tree_accept(target[None], parent[None], token[None], np.array([B], np.int32), N)
        assert out["acc_len"][0] == exp_len
        assert out["acc_nodes"][0, :exp_len].tolist() == exp_nodes
        assert out["acc_tokens"][0, :exp_len].tolist() == exp_tokens
        assert out["bonus"][0] == exp_bonus


def test_accept_rejects_bad_tree(orc):
    target = np.zeros((1, 3, 8), np.float32)
    with pytest.raises(orc.OracleError):
        orc.tree_accept(target, np.array([[0, -1]], np.int32), np.array([[1, 2]], np.int32),
                        np.array([2], np.int32), 2)
    with pytest.raises(orc.OracleError):
        orc.tree_accept(target, np.array([[-1, 0]], np.int32), np.array([[1, 9]], np.int32),
                        np.array([2], np.int32), 2)
