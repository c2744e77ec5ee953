"""GPU temperature-T acceptance (jt_tree_accept_sampled) vs the oracle.

"JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
summary), App. F.1 and F.3. Both sides draw from the same counter-based
stream with the same binary32 steps, so the walks match bit for bit: chains
and small trees (per-row draws + warp walk), wide trees (cluster path walk),
vocabularies up to 151936, several temperatures and seeds. Also the pages'
worked example as a frequency over many independent sequences.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity_util import to_np
from test_oracle_sampling import read_golden
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def random_tree_tokens(rng, batch, B, V, n):
    parent = np.full((batch, B), -1, np.int32)
    token = np.full((batch, B), -1, np.int32)
    for b in range(batch):
        for v in range(n[b]):
            parent[b, v] = rng.integers(-1, v) if v else -1
            sib = {int(token[b, u]) for u in range(v) if parent[b, u] == parent[b, v]}
            t = int(rng.integers(0, V))
            while t in sib:
                t = int(rng.integers(0, V))
            token[b, v] = t
    return parent, token


def steer(rng, target, parent, token, n, T):
    """Raise a child's token in each row so that walks often go deep."""
    for b in range(target.shape[0]):
        for u in range(-1, n[b]):
            kids = [v for v in range(n[b]) if parent[b, v] == u]
            if kids:
                row = target[b, 0 if u < 0 else 1 + u]
                row[token[b, rng.choice(kids)]] = row.max() + 2.0 * T


@pytest.mark.parametrize("batch,B,N,V,T", [
    (6, 16, 16, 1024, 1.0), (3, 16, 16, 151936, 0.7), (8, 8, 4, 4096, 2.0),
    (4, 128, 16, 8192, 1.0), (2, 200, 8, 151936, 1.0), (5, 64, 4, 2048, 0.3)])
def test_sampled_accept_parity(batch, B, N, V, T):
    rng = np.random.default_rng(B * 7 + N + V % 97)
    n = np.full(batch, B, np.int32)
    n[-1] = max(1, B // 3)
    parent, token = random_tree_tokens(rng, batch, B, V, n)
    target = (rng.standard_normal((batch, B + 1, V)) * 2).astype(np.float32)
    steer(rng, target, parent, token, n, T)
    d = lambda a: torch.from_numpy(a).to(DEV)
    for seed in (0, 12345, 2 ** 63 + 17):
        ref = oracle.tree_accept_sampled(target, parent, token, n, N, T, seed)
        got = jtree.jt_tree_accept(d(target), d(parent), d(token), d(n), N, temperature=T,
                                   seed=seed)
        for k in ("acc_len", "acc_tokens", "acc_nodes", "bonus"):
            assert np.array_equal(to_np(got[k]), ref[k]), (k, seed)


def test_sampled_worked_example_frequency():
    """The pages' chain: P(accept d1, reject d2, bonus b) = 0.24 over 40000
    independent sequences of one call (draws differ by sequence index)."""
    g = read_golden()
    V, d1, d2, b_tok, batch = 8, 1, 2, 3, 40000
    lg = lambda p: np.log(np.asarray(p, np.float64)).astype(np.float32)
    root = [0.05, g["p_d1"], 0.05, 0.05, 0.0125, 0.0125, 0.0125, 0.0125]
    after_d1 = [0.05, 0.05, g["p_d2_after_d1"], g["p_b_after_d1"], 0.025, 0.025, 0.025, 0.025]
    rows = np.stack([lg(root), lg(after_d1), lg([1 / 8] * 8)])
    target = np.broadcast_to(rows, (batch, 3, V)).copy()
    parent = np.broadcast_to(np.array([-1, 0], np.int32), (batch, 2)).copy()
    token = np.broadcast_to(np.array([d1, d2], np.int32), (batch, 2)).copy()
    n = np.full(batch, 2, np.int32)
    d = lambda a: torch.from_numpy(a).to(DEV)
    got = jtree.jt_tree_accept(d(target), d(parent), d(token), d(n), 2, temperature=1.0, seed=7)
    L, bonus = to_np(got["acc_len"]), to_np(got["bonus"])
    se = lambda p: 4 * np.sqrt(p * (1 - p) / batch)
    assert abs(np.mean((L == 1) & (bonus == b_tok)) - g["P_1_b"]) < se(g["P_1_b"])
    assert abs(np.mean(L == 2) - g["p_d1"] * g["p_d2_after_d1"]) < se(0.4)
    # And the oracle agrees draw for draw on a slice of it.
    ref = oracle.tree_accept_sampled(target[:500], parent[:500], token[:500], n[:500], 2, 1.0, 7)
    assert np.array_equal(L[:500], ref["acc_len"]) and np.array_equal(bonus[:500], ref["bonus"])


def test_sampled_host_checks():
    lib = jtree.load()
    z = torch.zeros(256, dtype=torch.int32, device=DEV)
    f = torch.zeros(256, dtype=torch.float32, device=DEV)
    ex = jtree.Exec(DEV).c()
    for T in (0.0, -1.0, float("nan"), float("inf")):
        rc = lib.jt_tree_accept_sampled(f.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                        1, 4, 4, 16, ctypes.c_float(T), ctypes.c_uint64(1),
                                        z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr(),
                                        ctypes.byref(ex))
        assert rc == 1, T
