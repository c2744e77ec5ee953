"""Pins for the oracle's tree-causal attention.

What the pages fix (JetSpec summary on paperlayer.ai, §2 "Architecture" and
App. D "Draft-head training"; JetSpec review on startedourmission.github.io,
"How it works", mask and factorisation equations):
  * a node attends to the prefix, its ancestors and itself only;
  * with a chain tree this is ordinary causal attention over prefix + chain
    (the block-causal training mask is the chain special case);
  * the branch factorisation: node v's output is plain attention of its query
    over the gathered sequence prefix ++ path(v).
The references below use torch's scaled_dot_product_attention in float64 —
a library routine, independent of the oracle's loops.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F


def bf16(shape, gen):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def random_tree(B, rng, n=None):
    n = B if n is None else n
    parent = np.full(B, -1, np.int32)
    for v in range(1, n):
        parent[v] = rng.integers(-1, v)
    return parent, n


def path_of(parent, v):
    p = []
    while v != -1:
        p.append(v)
        v = parent[v]
    return p[::-1]


def sdpa64(q, k, v, causal=False):
    return F.scaled_dot_product_attention(q.double(), k.double(), v.double(), is_causal=causal)


def make(batch, B, hq, hkv, D, L, seed):
    g = torch.Generator().manual_seed(seed)
    return dict(
        q=bf16((batch, B, hq, D), g), k_tree=bf16((batch, B, hkv, D), g),
        v_tree=bf16((batch, B, hkv, D), g), k_cache=bf16((batch, L, hkv, D), g),
        v_cache=bf16((batch, L, hkv, D), g))


@pytest.mark.parametrize("L,n,hq,hkv,D", [(37, 9, 4, 1, 64), (128, 16, 8, 2, 128), (0, 5, 2, 2, 64)])
def test_chain_equals_causal_attention(orc, L, n, hq, hkv, D):
    t = make(1, n, hq, hkv, D, max(L, 1), seed=L + n)
    parent = np.array([[-1] + list(range(n - 1))], np.int32)
    nn = np.array([n], np.int32)
    mask = orc.tree_mask(parent, nn)
    got = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                        np.array([L], np.int32), nn, mask, hq=hq, hkv=hkv)
    # Textbook causal attention over the full sequence prefix ++ chain; the
    # prefix positions get arbitrary queries and their outputs are dropped.
    g = torch.Generator().manual_seed(99)
    q_pre = bf16((L, hq, D), g)
    qs = torch.cat([q_pre, t["q"][0]], 0).permute(1, 0, 2)[None]             # [1,hq,S,D]
    k = torch.cat([t["k_cache"][0, :L], t["k_tree"][0]], 0).permute(1, 0, 2)[None]
    v = torch.cat([t["v_cache"][0, :L], t["v_tree"][0]], 0).permute(1, 0, 2)[None]
    grp = hq // hkv
    k = k.repeat_interleave(grp, dim=1)
    v = v.repeat_interleave(grp, dim=1)
    ref = sdpa64(qs, k, v, causal=True)[0, :, L:, :].permute(1, 0, 2).numpy()  # [n,hq,D]
    np.testing.assert_allclose(got[0], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L,B,hq,hkv,D,seed", [(50, 24, 4, 1, 64, 1), (0, 33, 4, 2, 64, 2),
                                               (200, 64, 8, 2, 128, 3)])
def test_each_node_equals_attention_over_its_gathered_path(orc, L, B, hq, hkv, D, seed):
    rng = np.random.default_rng(seed)
    t = make(1, B, hq, hkv, D, max(L, 1), seed)
    parent, n = random_tree(B, rng, n=B - 3)
    nn = np.array([n], np.int32)
    mask = orc.tree_mask(parent[None], nn)
    got = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                        np.array([L], np.int32), nn, mask, hq=hq, hkv=hkv)
    grp = hq // hkv
    for v in range(n):
        path = path_of(parent, v)
        for h in range(hq):
            kh = h // grp
            keys = torch.cat([t["k_cache"][0, :L, kh], t["k_tree"][0, path, kh]], 0)
            vals = torch.cat([t["v_cache"][0, :L, kh], t["v_tree"][0, path, kh]], 0)
            ref = sdpa64(t["q"][0, v, h][None, None], keys[None], vals[None])[0, 0].numpy()
            np.testing.assert_allclose(got[0, v, h], ref, rtol=0, atol=1e-12)
    assert not got[0, n:].any()


def test_non_ancestor_perturbation_leaves_output_bit_identical(orc):
    rng = np.random.default_rng(7)
    B, hq, hkv, D, L = 40, 4, 2, 64, 30
    t = make(1, B, hq, hkv, D, L, seed=7)
    parent, n = random_tree(B, rng)
    nn = np.array([n], np.int32)
    mask = orc.tree_mask(parent[None], nn)
    args = dict(hq=hq, hkv=hkv)
    base = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                         np.array([L], np.int32), nn, mask, **args)
    g = torch.Generator().manual_seed(8)
    for v in [0, 5, 17, 39]:
        hidden = [u for u in range(n) if u not in path_of(parent, v)]
        kt, vt = t["k_tree"].clone(), t["v_tree"].clone()
        kt[0, hidden] = bf16((len(hidden), hkv, D), g) * 50
        vt[0, hidden] = bf16((len(hidden), hkv, D), g) * 50
        out = orc.tree_attn(t["q"], kt, vt, t["k_cache"], t["v_cache"],
                            np.array([L], np.int32), nn, mask, **args)
        assert np.array_equal(out[0, v], base[0, v])
        assert not np.array_equal(out, base)  # the perturbation did reach other nodes


def test_paged_layout_equals_contiguous(orc):
    rng = np.random.default_rng(11)
    batch, B, hq, hkv, D, Lmax, P = 3, 16, 4, 2, 64, 100, 16
    t = make(batch, B, hq, hkv, D, Lmax, seed=11)
    lens = np.array([100, 33, 0], np.int32)
    parents = np.stack([random_tree(B, rng)[0] for _ in range(batch)])
    nn = np.array([16, 9, 16], np.int32)
    mask = orc.tree_mask(parents, nn)
    ref = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"], lens, nn,
                        mask, hq=hq, hkv=hkv)
    max_pages = (Lmax + P - 1) // P
    n_pages = batch * max_pages
    perm = rng.permutation(n_pages).astype(np.int32)
    bt = perm.reshape(batch, max_pages)
    kp = torch.zeros((n_pages, P, hkv, D), dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    for b in range(batch):
        for j in range(Lmax):
            kp[bt[b, j // P], j % P] = t["k_cache"][b, j]
            vp[bt[b, j // P], j % P] = t["v_cache"][b, j]
    got = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], kp, vp, lens, nn, mask, hq=hq, hkv=hkv,
                        block_table=bt)
    assert np.array_equal(got, ref)
    # Selected rows equal the matching rows of the full computation.
    rows = np.array([[0, 3, 1], [1, 8, 3], [2, 15, 0], [1, 12, 2]], np.int32)
    sel = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], kp, vp, lens, nn, mask, hq=hq, hkv=hkv,
                        block_table=bt, rows=rows)
    for i, (b, v, h) in enumerate(rows):
        assert np.array_equal(sel[i], ref[b, v, h])
    assert not sel[3].any()  # node 12 >= n_nodes[1] = 9


def test_scale_argument(orc):
    t = make(1, 4, 2, 1, 64, 8, seed=5)
    parent = np.array([[-1, 0, 1, 2]], np.int32)
    nn = np.array([4], np.int32)
    mask = orc.tree_mask(parent, nn)
    a = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                      np.array([8], np.int32), nn, mask, hq=2, hkv=1)
    b = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                      np.array([8], np.int32), nn, mask, hq=2, hkv=1, scale=1 / 8.0)
    assert np.array_equal(a, b)  # 0 means 1/sqrt(64)
    c = orc.tree_attn(t["q"], t["k_tree"], t["v_tree"], t["k_cache"], t["v_cache"],
                      np.array([8], np.int32), nn, mask, hq=2, hkv=1, scale=0.5)
    assert not np.allclose(a, c)
