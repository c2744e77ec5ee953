"""GPU accepted-path K/V commit (jt_tree_commit_kv) vs the oracle.

"JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
summary), §3 "Preliminaries": a round commits the accepted prefix plus a bonus
token. Bit-exact on whole caches: the hand-worked example, random contiguous
and paged caches with rejected sequences (bad node, overflow, bad page, bad
acc_len), in-place lengths, and the host-side argument checks.
"""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_commit import bf16_bits, parse_golden
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_dev_bf16(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).to(DEV).view(torch.bfloat16)


def to_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(kt, vt, kc, vc, L, a, nodes, table=None, in_place=False):
    ex = jtree.Exec(DEV)
    kc_d, vc_d = to_dev_bf16(kc), to_dev_bf16(vc)
    L_d = torch.from_numpy(L).to(DEV)
    new_len = jtree.jt_tree_commit_kv(
        to_dev_bf16(kt), to_dev_bf16(vt), kc_d, vc_d, L_d, torch.from_numpy(a).to(DEV),
        torch.from_numpy(nodes).to(DEV), new_prefix_len=L_d if in_place else None,
        block_table=None if table is None else torch.from_numpy(table).to(DEV), exec=ex)
    flags = ex.read_error()
    return to_bits(kc_d), to_bits(vc_d), new_len.cpu().numpy(), flags


def test_commit_golden_gpu():
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
    args = (bf16_bits(kt), bf16_bits(-kt), bf16_bits(kc), bf16_bits(-kc), L, a, nodes)
    k2, v2, new_len, flags = run_gpu(*args)
    ko, vo, len_o, _ = oracle.tree_commit_kv(*args, check=False)
    assert np.array_equal(k2, ko) and np.array_equal(v2, vo)
    assert list(new_len) == [expects[b]["len"] for b in range(batch)]
    assert flags == jtree.JT_DEVERR_PREFIX   # sequence 2 overflows its cache


def random_case(rng, batch, B, N, hkv, D, paged, P=16, max_pages=6, Lmax=90):
    kt = rng.integers(0, 2 ** 16, (batch, B, hkv, D)).astype(np.uint16)
    vt = rng.integers(0, 2 ** 16, (batch, B, hkv, D)).astype(np.uint16)
    acc_len = rng.integers(0, N + 1, batch).astype(np.int32)
    acc_nodes = -np.ones((batch, N), np.int32)
    for b in range(batch):
        acc_nodes[b, : acc_len[b]] = rng.permutation(B)[: acc_len[b]]
    if paged:
        n_pool = batch * max_pages + 3
        table = rng.permutation(n_pool)[: batch * max_pages].reshape(batch, max_pages)
        table = table.astype(np.int32)
        kc = rng.integers(0, 2 ** 16, (n_pool, P, hkv, D)).astype(np.uint16)
        vc = rng.integers(0, 2 ** 16, (n_pool, P, hkv, D)).astype(np.uint16)
        cap = max_pages * P
    else:
        table = None
        kc = rng.integers(0, 2 ** 16, (batch, Lmax, hkv, D)).astype(np.uint16)
        vc = rng.integers(0, 2 ** 16, (batch, Lmax, hkv, D)).astype(np.uint16)
        cap = Lmax
    L = rng.integers(0, cap - N + 1, batch).astype(np.int32)
    return kt, vt, kc, vc, L, acc_len, acc_nodes, table, cap


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("batch,B,N,hkv,D", [(1, 16, 16, 8, 128), (5, 64, 8, 8, 128),
                                             (9, 256, 64, 1, 64), (17, 33, 7, 4, 8),
                                             (3, 1, 1, 2, 16)])
def test_commit_random(paged, batch, B, N, hkv, D):
    rng = np.random.default_rng(batch * 100 + B + N + paged)
    kt, vt, kc, vc, L, a, nodes, table, cap = random_case(rng, batch, B, N, hkv, D, paged)
    want_flags = 0
    if batch >= 5:
        # One rejected sequence of each kind.
        a[0], nodes[0, 0] = max(a[0], 1), B                      # node outside [0, B)
        L[1], a[1] = cap - 1, 2                                  # past the cache
        nodes[1, :2] = [0, 0]
        a[2] = N + 1                                             # acc_len > n_depth
        want_flags = jtree.JT_DEVERR_PATH | jtree.JT_DEVERR_PREFIX
        if paged:
            L[3], a[3] = 0, max(a[3], 1)
            nodes[3, : a[3]] = np.arange(a[3]) % B
            table[3, 0] = 10 ** 6                                # page outside the pool
            want_flags |= jtree.JT_DEVERR_PAGE
    for in_place in (False, True):
        k2, v2, new_len, flags = run_gpu(kt, vt, kc, vc, L, a, nodes, table, in_place)
        ko, vo, len_o, rc = oracle.tree_commit_kv(kt, vt, kc, vc, L, a, nodes,
                                                  block_table=table, check=False)
        assert np.array_equal(k2, ko), "K cache"
        assert np.array_equal(v2, vo), "V cache"
        assert np.array_equal(new_len, len_o)
        assert flags == want_flags
        assert (rc != 0) == (want_flags != 0)


def test_commit_host_checks():
    lib = jtree.load()
    kt = torch.zeros((1, 4, 1, 12), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((1, 8, 1, 12), dtype=torch.bfloat16, device=DEV)
    i1 = torch.zeros((1,), dtype=torch.int32, device=DEV)
    nodes = torch.zeros((1, 2), dtype=torch.int32, device=DEV)
    args = jtree.commit_args(kt, kt, kc, kc, i1, i1, nodes, i1.clone())
    ex = jtree.Exec(DEV).c()
    import ctypes
    assert lib.jt_tree_commit_kv(ctypes.byref(args), ctypes.byref(ex)) == 2   # head_dim % 8
    args.head_dim = 16
    args.k_tree = None
    assert lib.jt_tree_commit_kv(ctypes.byref(args), ctypes.byref(ex)) == 1   # null pointer
    assert lib.jt_tree_commit_kv(None, ctypes.byref(ex)) == 1
