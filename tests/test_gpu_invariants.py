"""Properties the pages fix, checked on the CUDA path itself.

* Non-ancestor invariance (JetSpec summary on paperlayer.ai, §2
  "Architecture"; Korean review on startedourmission.github.io, "How it
  works", mask equation M[v,u] = 0 iff u is v or an ancestor of v): node v
  attends to the prefix and to its own root path only, so rewriting the K/V
  of every other tree node must leave v's output unchanged. The kernel
  masks those keys before the row maximum and multiplies their values by an
  exact zero, so the output must be bit-identical, not merely close.
* A chain is causal attention (JetSpec summary, App. A.1: a depth-N chain
  reduces to ordinary causal attention): the chain workload's tree
  attention equals torch's scaled_dot_product_attention(is_causal=True)
  over prefix ++ chain, evaluated in fp64 on the CPU.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from parity_util import check_attn
from tree_causal_verification_gb300 import jtree, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def bf16(shape, g):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def deep_tree(rng, B):
    """Random tree with long paths: each node hangs below its predecessor
    half of the time, else below a uniformly drawn earlier node (or the root)."""
    parent = np.full(B, -1, np.int32)
    for v in range(1, B):
        parent[v] = v - 1 if rng.random() < 0.5 else rng.integers(-1, v)
    return parent


def path_of(parent, v):
    out = []
    while v >= 0:
        out.append(v)
        v = parent[v]
    return out


@pytest.mark.parametrize("batch,B,hq,hkv,paged,Lmax", [
    (3, 128, 32, 4, True, 3000),     # MoE shape, paged prefix
    (2, 256, 32, 8, False, 1100),    # high-budget shape, contiguous prefix
    (4, 64, 32, 8, True, 2050),      # mid-batch shape, paged prefix
    (40, 64, 32, 8, True, 700),      # enough units for the length-ordered schedule
])
def test_non_ancestor_kv_leaves_output_bit_identical(batch, B, hq, hkv, paged, Lmax):
    rng = np.random.default_rng(B + batch)
    g = torch.Generator().manual_seed(B * 3 + batch)
    D = 128
    n = np.full(batch, B, np.int32)
    n[-1] = B - 5
    parent = np.stack([deep_tree(rng, B) for _ in range(batch)])
    mask = oracle.tree_mask(parent, n)
    lens = rng.integers(Lmax // 2, Lmax + 1, batch).astype(np.int32)
    q = bf16((batch, B, hq, D), g)
    kt, vt = bf16((batch, B, hkv, D), g), bf16((batch, B, hkv, D), g)
    if paged:
        max_pages = (Lmax + 15) // 16
        n_pages = batch * max_pages
        bt = rng.permutation(n_pages).reshape(batch, max_pages).astype(np.int32)
        kc, vc = bf16((n_pages, 16, hkv, D), g), bf16((n_pages, 16, hkv, D), g)
    else:
        bt = None
        kc, vc = bf16((batch, Lmax, hkv, D), g), bf16((batch, Lmax, hkv, D), g)
    # Chosen nodes per sequence: the deepest, the last live one and one at random.
    chosen, keep = [], np.zeros((batch, B), bool)
    for b in range(batch):
        depth = [len(path_of(parent[b], v)) for v in range(n[b])]
        vs = {int(np.argmax(depth)), int(n[b]) - 1, int(rng.integers(0, n[b]))}
        for v in vs:
            chosen.append((b, v))
            keep[b, path_of(parent[b], v)] = True
    assert (~keep[:, : int(n.min())]).any()   # something is left to perturb
    # Every other node's K and V, times 50.
    scale = torch.from_numpy(np.where(keep, 1.0, 50.0).astype(np.float32)).view(batch, B, 1, 1)
    kt2 = (kt.float() * scale).to(torch.bfloat16)
    vt2 = (vt.float() * scale).to(torch.bfloat16)
    d = lambda t: t.to(DEV)
    ex = jtree.Exec(DEV)

    def run(k_tree, v_tree):
        out = torch.full((batch, B, hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        jtree.jt_tree_attn(d(q), d(k_tree), d(v_tree), d(kc), d(vc), d(torch.from_numpy(lens)),
                           d(torch.from_numpy(n)), d(torch.from_numpy(mask.view(np.int32))),
                           out=out, block_table=None if bt is None else d(torch.from_numpy(bt)),
                           exec=ex)
        assert ex.read_error() == 0
        return out.view(torch.int16).cpu().numpy()

    base, pert = run(kt, vt), run(kt2, vt2)
    for b, v in chosen:
        assert np.array_equal(base[b, v], pert[b, v]), (b, v)
    # The perturbation did reach the nodes that see a perturbed key.
    assert not np.array_equal(base, pert)


def test_chain_equals_causal_attention():
    w = synth.WORKLOADS["qwen3-8b-chain"]
    kv = synth.kv_inputs(w, 3, "cpu")
    L, n, g = int(kv["prefix_len"][0]), w.B, w.hq // w.hkv
    parent = np.arange(-1, n - 1, dtype=np.int32)[None]          # node v below v - 1
    nn = np.array([n], np.int32)
    d = lambda t: t.to(DEV)
    ex = jtree.Exec(DEV)
    mask = jtree.jt_tree_mask(d(torch.from_numpy(parent)), d(torch.from_numpy(nn)), exec=ex)
    out = jtree.jt_tree_attn(d(kv["q"]), d(kv["k_tree"]), d(kv["v_tree"]), d(kv["k_cache"]),
                             d(kv["v_cache"]), d(kv["prefix_len"]), d(torch.from_numpy(nn)),
                             mask, exec=ex)
    assert ex.read_error() == 0
    got = out[0].float().cpu().numpy()                            # [n][hq][D]
    # Textbook causal attention over the L + n positions prefix ++ chain; the
    # prefix positions' queries are zeros (their rows are not compared).
    K = torch.cat([kv["k_cache"][0, :L], kv["k_tree"][0]], 0).double()   # [L+n][hkv][D]
    V = torch.cat([kv["v_cache"][0, :L], kv["v_tree"][0]], 0).double()
    Q = torch.cat([torch.zeros((L, w.hq, w.D), dtype=torch.float64), kv["q"][0].double()], 0)
    ref = np.zeros_like(got, dtype=np.float64)
    for kh in range(w.hkv):
        qh = Q[:, kh * g:(kh + 1) * g].permute(1, 0, 2)                 # [g][L+n][D]
        kk = K[:, kh].unsqueeze(0).expand(g, -1, -1)
        vv = V[:, kh].unsqueeze(0).expand(g, -1, -1)
        o = F.scaled_dot_product_attention(qh, kk, vv, is_causal=True)
        ref[:, kh * g:(kh + 1) * g] = o[:, L:].permute(1, 0, 2).numpy()
    check_attn(got.reshape(-1, w.D), ref.reshape(-1, w.D), "chain vs causal")
