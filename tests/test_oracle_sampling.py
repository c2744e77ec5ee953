"""Pins for the oracle's temperature-T acceptance (no GPU).

"JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
summary), App. F.1 (worked example P(1, b) = 0.24) and App. F.3 (point-mass
proposals: every committed token is the target's own draw).

The generator (SplitMix64, Steele, Lea and Flood 2014) is pinned by its
reference outputs; the log by fp64 log; the Gumbel-max draw by the softmax
frequencies; the walk by the pages' worked example and by the T -> 0 limit
(greedy acceptance).
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampled_accept_example.txt")


def test_splitmix64_reference_outputs(orc):
    # First five outputs of the reference splitmix64.c generator seeded with 1234567.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    got = orc.splitmix64(1234567, np.arange(1, 6, dtype=np.uint64))
    assert [int(v) for v in got] == want


def test_series_ln_accuracy(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([np.exp(rng.uniform(-16.7, 2.9, 200000)),
                        [5.96e-8, 1.0 - 2 ** -24, 1.0, 2.0, 0.5, np.sqrt(2.0), 17.0]])
    x = x.astype(np.float32)
    got = orc.series_ln(x).astype(np.float64)
    ref = np.log(x.astype(np.float64))
    err = np.abs(got - ref)
    assert (err <= 4e-7 * np.maximum(np.abs(ref), 1e-30) + 2e-7).all(), err.max()


def test_uniform_and_gumbel_moments(orc):
    k = np.arange(1, 400001, dtype=np.uint64)
    g = orc.gumbel(99, k).astype(np.float64)
    # Gumbel(0,1): mean = Euler-Mascheroni constant, variance = pi^2 / 6.
    n = g.size
    assert abs(g.mean() - 0.5772156649) < 4 * np.sqrt(np.pi ** 2 / 6 / n)
    assert abs(g.var() - np.pi ** 2 / 6) < 0.02
    u = np.exp(-np.exp(-g))                       # back to the uniform
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / n)
    hist = np.histogram(u, bins=20, range=(0, 1))[0]
    assert (np.abs(hist - n / 20) < 5 * np.sqrt(n / 20)).all()


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_draw_frequencies_match_softmax(orc, T):
    """Root draws (acc_len 0 when no child matches) follow softmax(x / T)."""
    V, trials = 8, 20000
    x = np.array([1.0, 0.0, -1.0, 2.0, 0.5, -np.inf, 1.5, -0.5], np.float32)
    p = np.exp(np.where(np.isinf(x), -np.inf, x / T))
    p = p / p.sum()
    counts = np.zeros(V)
    parent = np.full((1, 1), -1, np.int32)
    token = np.full((1, 1), 0, np.int32)
    n0 = np.zeros(1, np.int32)                    # no tree nodes: the draw is the bonus
    target = np.tile(x, (1, 2, 1))
    for s in range(trials):
        r = orc.tree_accept_sampled(target, parent, token, n0, 1, T, seed=s)
        counts[r["bonus"][0]] += 1
    freq = counts / trials
    assert counts[5] == 0                          # a -inf logit is never drawn
    assert (np.abs(freq - p) <= 4.5 * np.sqrt(p * (1 - p) / trials) + 1e-12).all(), (freq, p)


def read_golden():
    d = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if line:
            d[line[0]] = float(line[1])
    return d


def test_worked_example_outcome_probability(orc):
    """Chain d1 -> d2 with the pages' target probabilities: the frequency of
    outcome (1 accepted, bonus b) converges to 0.24, and the other outcomes
    to their products."""
    g = read_golden()
    V, d1, d2, b_tok = 6, 1, 2, 3
    logits = lambda probs: np.log(np.asarray(probs, np.float64)).astype(np.float32)
    root = [0.05, g["p_d1"], 0.05, 0.05, 0.025, 0.025]                  # p(d1) = 0.8
    after_d1 = [0.05, 0.05, g["p_d2_after_d1"], g["p_b_after_d1"], 0.05, 0.05]
    after_d2 = [1 / 6] * 6
    target = np.stack([logits(root), logits(after_d1), logits(after_d2)])[None]
    parent = np.array([[-1, 0]], np.int32)
    token = np.array([[d1, d2]], np.int32)
    n = np.array([2], np.int32)
    trials = 20000
    hits_1b = len0 = len1 = len2 = 0
    for s in range(trials):
        r = orc.tree_accept_sampled(target, parent, token, n, 2, 1.0, seed=1000 + s)
        L, bonus = int(r["acc_len"][0]), int(r["bonus"][0])
        len0 += L == 0
        len1 += L == 1
        len2 += L == 2
        hits_1b += (L == 1 and bonus == b_tok)
    se = lambda p: 4 * np.sqrt(p * (1 - p) / trials)
    assert abs(hits_1b / trials - g["P_1_b"]) < se(g["P_1_b"])
    assert abs(len0 / trials - (1 - g["p_d1"])) < se(0.2)
    assert abs(len1 / trials - g["p_d1"] * (1 - g["p_d2_after_d1"])) < se(0.4)
    assert abs(len2 / trials - g["p_d1"] * g["p_d2_after_d1"]) < se(0.4)


def test_low_temperature_is_greedy(orc):
    rng = np.random.default_rng(3)
    batch, B, N, V = 6, 20, 6, 512
    parent = np.full((batch, B), -1, np.int32)
    token = np.zeros((batch, B), np.int32)
    for b in range(batch):
        for v in range(B):
            parent[b, v] = rng.integers(-1, v) if v else -1
        for v in range(B):   # distinct tokens among siblings
            sib = [u for u in range(v) if parent[b, u] == parent[b, v]]
            choices = [t for t in range(V) if t not in token[b, sib]]
            token[b, v] = rng.choice(choices)
    n = np.full(batch, B, np.int32)
    target = rng.standard_normal((batch, B + 1, V)).astype(np.float32)
    for b in range(batch):   # steer rows towards children so walks go deep
        for u in range(-1, B):
            kids = [v for v in range(B) if parent[b, v] == u]
            if kids:
                target[b, 0 if u < 0 else 1 + u, token[b, rng.choice(kids)]] += 5.0
    g = orc.tree_accept(target, parent, token, n, N)
    for seed in (1, 2, 3):
        s = orc.tree_accept_sampled(target, parent, token, n, N, 1e-4, seed=seed)
        for k in g:
            assert np.array_equal(g[k], s[k]), k
