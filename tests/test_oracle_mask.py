"""Pins for the oracle's tree-causal mask.

Definition pinned: M[v,u] = 0 iff u ∈ Anc(v) ∪ {v} (JetSpec review on
startedourmission.github.io, "How it works", mask equation; JetSpec summary
on paperlayer.ai, §2 "Architecture": a node sees its ancestors and itself,
never descendants or unrelated siblings).
"""
import itertools
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_parent_arrays(n):
    """Every valid parent array of n nodes: parent[v] in [-1, v)."""
    return itertools.product(*[range(-1, v) for v in range(n)])


def closure_reference(parents, n_nodes, B):
    """Ancestor-or-self relation by boolean matrix iteration (no parent walk).

    step[v,u] = 1 iff u == parent[v]; reach = I, then reach |= reach @ step until
    fixed. reach[v,u] = 1 iff u is reachable from v by following parent links.
    """
    batch = parents.shape[0]
    step = np.zeros((batch, B, B), np.int64)
    bi, vi = np.nonzero(parents >= 0)
    step[bi, vi, parents[bi, vi]] = 1
    alive = (np.arange(B)[None, :] < n_nodes[:, None])
    reach = np.broadcast_to(np.eye(B, dtype=np.int64), (batch, B, B)).copy()
    reach *= alive[:, :, None]
    for _ in range(B):
        nxt = ((reach + reach @ step) > 0).astype(np.int64)
        if np.array_equal(nxt, reach):
            break
        reach = nxt
    return reach.astype(bool)


def unpack(mask, B):
    bits = np.zeros(mask.shape[:-1] + (B,), bool)
    for u in range(B):
        bits[..., u] = (mask[..., u >> 5] >> np.uint32(u & 31)) & 1
    return bits


def test_mask_bruteforce_all_trees_up_to_8(orc):
    B = 8
    parents, sizes = [], []
    for n in range(0, B + 1):
        for p in all_parent_arrays(n):
            row = list(p) + [-1] * (B - n)
            parents.append(row)
            sizes.append(n)
    parents = np.array(parents, np.int32)
    sizes = np.array(sizes, np.int32)
    assert parents.shape[0] == sum(__import__("math").factorial(n) for n in range(B + 1))
    mask = orc.tree_mask(parents, sizes)
    got = unpack(mask, B)
    want = closure_reference(parents, sizes, B)
    assert np.array_equal(got, want)


def test_mask_recurrence_and_depth(orc):
    # mask[v] = mask[parent[v]] | bit(v), popcount(mask[v]) = depth(v) (root depth 0).
    rng = np.random.default_rng(1)
    B = 256
    batch = 16
    parents = np.full((batch, B), -1, np.int32)
    n_nodes = rng.integers(0, B + 1, batch).astype(np.int32)
    for b in range(batch):
        for v in range(1, B):
            parents[b, v] = rng.integers(-1, v)
    mask = orc.tree_mask(parents, n_nodes)
    bits = unpack(mask, B)
    for b in range(batch):
        n = n_nodes[b]
        depth = np.zeros(B, np.int64)
        for v in range(n):
            p = parents[b, v]
            expect = bits[b, p].copy() if p >= 0 else np.zeros(B, bool)
            expect[v] = True
            assert np.array_equal(bits[b, v], expect)
            depth[v] = (depth[p] if p >= 0 else 0) + 1
            assert bits[b, v].sum() == depth[v]
        assert not bits[b, n:].any()


def test_mask_word_layout(orc):
    # u -> word u >> 5, bit u & 31: a 40-node chain sets bit 7 of word 1 for node 39.
    B = 40
    parents = np.array([[-1] + list(range(B - 1))], np.int32)
    mask = orc.tree_mask(parents, np.array([B], np.int32))
    assert mask.shape == (1, B, 2)
    assert mask[0, 39, 0] == 0xFFFFFFFF
    assert mask[0, 39, 1] == 0xFF
    assert mask[0, 0, 0] == 1 and mask[0, 0, 1] == 0


def test_mask_golden_example(orc):
    """Hand-worked 6-node example (tests/golden/mask_example.txt)."""
    lines = [l.split("#")[0].strip() for l in open(os.path.join(GOLDEN, "mask_example.txt"))]
    lines = [l for l in lines if l]
    parents = np.array([[int(x) for x in lines[0].split()]], np.int32)
    B = parents.shape[1]
    want = np.array([[int(c) for c in l.split()] for l in lines[1:]], bool)
    got = unpack(orc.tree_mask(parents, np.array([B], np.int32)), B)[0]
    assert np.array_equal(got, want)


@pytest.mark.parametrize("bad", [[0, -1], [-1, 1], [-1, -2], [-1, 5]])
def test_mask_rejects_bad_parent(orc, bad):
    with pytest.raises(orc.OracleError):
        orc.tree_mask(np.array([bad], np.int32), np.array([2], np.int32))
