"""Pins for the oracle's accepted-path K/V commit (no GPU).

"JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
summary), §3 "Preliminaries": a round commits the accepted prefix plus a bonus
token. Pinned by a hand-worked example, by the verification semantics (the
committed cache is exactly what a causal decoder would attend to: prefix plus
the accepted path), and by invariants on random paged caches.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "commit_example.txt")


def bf16_bits(x):
    """float array -> bf16 bit patterns (values chosen exactly representable)."""
    u = np.asarray(x, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "golden values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def from_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def parse_golden():
    seqs, expects = {}, {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        if line[0] == "seq":
            b = int(line[1])
            seqs[b] = dict(L=int(line[3]), a=int(line[5]), nodes=[int(t) for t in line[7:]])
        elif line[0] == "expect":
            b = int(line[1])
            i = line.index("len")
            expects[b] = dict(src=line[2:i], len=int(line[i + 1]), rejected="rejected" in line)
    return seqs, expects


def test_commit_golden(orc):
    seqs, expects = parse_golden()
    batch, B, n_depth, hkv, D, Lmax = 3, 4, 3, 1, 8, 5
    e = np.arange(D) / 2.0
    kt = np.zeros((batch, B, hkv, D), np.float32)
    for b in range(batch):
        for v in range(B):
            kt[b, v, 0] = b * 32 + v * 4 + e
    kc = np.zeros((batch, Lmax, hkv, D), np.float32)
    for b in range(batch):
        for j in range(Lmax):
            kc[b, j] = -(100 + 10 * b + j)
    L = np.array([seqs[b]["L"] for b in range(batch)], np.int32)
    a = np.array([seqs[b]["a"] for b in range(batch)], np.int32)
    nodes = np.array([seqs[b]["nodes"] for b in range(batch)], np.int32)
    k2, v2, new_len, rc = orc.tree_commit_kv(bf16_bits(kt), bf16_bits(-kt), bf16_bits(kc),
                                             bf16_bits(-kc), L, a, nodes, check=False)
    assert rc != 0  # sequence 2 is rejected
    k2, v2 = from_bits(k2), from_bits(v2)
    for b in range(batch):
        ex = expects[b]
        assert new_len[b] == ex["len"]
        for j, src in enumerate(ex["src"]):
            want = kc[b, j] if src == "keep" else kt[b, int(src[4:])]
            np.testing.assert_array_equal(k2[b, j], want)
            np.testing.assert_array_equal(v2[b, j], -want)


def plain_attention(q, K, V, scale):
    """Textbook softmax attention of one query row over keys K / values V (fp64)."""
    s = (K @ q) * scale
    p = np.exp(s - s.max())
    return (p / p.sum()) @ V


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_commit_matches_tree_attention(orc, seed):
    """After committing the path to node v, plain causal attention of v's query
    over the committed cache equals the tree attention output of v (prefix plus
    ancestors plus itself): [PL] §2 "Architecture" and [PP] App. E."""
    rng = np.random.default_rng(seed)
    batch, B, N, W, hq, hkv, D = 2, 12, 5, 3, 4, 2, 16
    g = hq // hkv
    tok = np.stack([np.stack([rng.choice(50, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    tree = orc.tree_expand(tok, logp, B)
    mask = orc.tree_mask(tree["parent"], tree["n_nodes"])
    Lmax = 40
    L = rng.integers(0, 20, batch).astype(np.int32)
    bits = lambda shape: (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16
                          ).astype(np.uint16)
    q, kt, vt = bits((batch, B, hq, D)), bits((batch, B, hkv, D)), bits((batch, B, hkv, D))
    kc, vc = bits((batch, Lmax, hkv, D)), bits((batch, Lmax, hkv, D))
    # Accepted path: root -> ... -> the deepest node of a random leaf's ancestry.
    acc_len = np.zeros(batch, np.int32)
    acc_nodes = -np.ones((batch, N), np.int32)
    last = np.zeros(batch, np.int64)
    for b in range(batch):
        v = int(rng.integers(0, tree["n_nodes"][b]))
        path = []
        while v >= 0:
            path.append(v)
            v = int(tree["parent"][b, v])
        path = path[::-1]
        acc_len[b] = len(path)
        acc_nodes[b, : len(path)] = path
        last[b] = path[-1]
    k2, v2, new_len, _ = orc.tree_commit_kv(kt, vt, kc, vc, L, acc_len, acc_nodes)
    np.testing.assert_array_equal(new_len, L + acc_len)
    ref = orc.tree_attn(q, kt, vt, kc, vc, L, tree["n_nodes"], mask, hq=hq, hkv=hkv)
    scale = 1.0 / np.sqrt(D)
    for b in range(batch):
        n_keys = int(new_len[b])
        for h in range(hq):
            K = from_bits(k2[b, :n_keys, h // g]).astype(np.float64)
            V = from_bits(v2[b, :n_keys, h // g]).astype(np.float64)
            qv = from_bits(q[b, last[b], h]).astype(np.float64)
            np.testing.assert_allclose(plain_attention(qv, K, V, scale), ref[b, last[b], h],
                                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [3, 4])
def test_commit_paged_invariants(orc, seed):
    """Only the committed slots change; each holds its tree row; rejected
    sequences (bad node, overflow, bad page) are untouched and keep their length."""
    rng = np.random.default_rng(seed)
    batch, B, N, hkv, D, P = 6, 20, 8, 2, 8, 16
    max_pages = 4
    n_pool = batch * max_pages + 5
    table = rng.permutation(n_pool)[: batch * max_pages].reshape(batch, max_pages).astype(np.int32)
    kt = rng.integers(0, 2 ** 16, (batch, B, hkv, D)).astype(np.uint16)
    vt = rng.integers(0, 2 ** 16, (batch, B, hkv, D)).astype(np.uint16)
    kc = rng.integers(0, 2 ** 16, (n_pool, P, hkv, D)).astype(np.uint16)
    vc = rng.integers(0, 2 ** 16, (n_pool, P, hkv, D)).astype(np.uint16)
    L = rng.integers(0, max_pages * P - N, batch).astype(np.int32)
    acc_len = rng.integers(0, N + 1, batch).astype(np.int32)
    acc_nodes = np.stack([rng.permutation(B)[:N] for _ in range(batch)]).astype(np.int32)
    acc_len[0] = 0                                   # nothing to commit
    acc_len[1], acc_nodes[1, 0] = max(acc_len[1], 1), B   # bad node -> rejected
    L[2], acc_len[2] = max_pages * P - 2, 3          # overflow -> rejected
    L[3], acc_len[3] = 5, 4
    table[3, 0] = n_pool + 7                         # bad page on the committed slots -> rejected
    bad = {1, 2, 3}
    k2, v2, new_len, rc = orc.tree_commit_kv(kt, vt, kc, vc, L, acc_len, acc_nodes,
                                             block_table=table, check=False)
    assert rc != 0
    written = np.zeros((n_pool, P), bool)
    for b in range(batch):
        if b in bad:
            assert new_len[b] == L[b]
            continue
        assert new_len[b] == L[b] + acc_len[b]
        for i in range(acc_len[b]):
            pos = L[b] + i
            page, slot = table[b, pos // P], pos % P
            np.testing.assert_array_equal(k2[page, slot], kt[b, acc_nodes[b, i]])
            np.testing.assert_array_equal(v2[page, slot], vt[b, acc_nodes[b, i]])
            written[page, slot] = True
    np.testing.assert_array_equal(k2[~written], kc[~written])
    np.testing.assert_array_equal(v2[~written], vc[~written])
