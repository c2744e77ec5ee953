"""GPU vs oracle on small random and edge cases, and the device-side checks.

Covers budgets that straddle mask words (1, 31, 32, 33, 255, 256), widths
1..32, depths 1..64, ragged prefixes around page and tile boundaries (0, 1,
15, 16, 17, ...), n_nodes < B, paged and contiguous caches, GQA groups 1..16,
head_dim 64 and 128, ties and -inf logits, and bad device data (parent,
token, page, prefix length, n_nodes) that must raise a flag, never fault.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import LOGP_ABS, check_attn, to_np, u32
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def bf16(shape, g):
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def random_tree(rng, B, n):
    parent = np.full(B, -1, np.int32)
    for v in range(1, n):
        parent[v] = rng.integers(-1, v)
    return parent


@pytest.mark.parametrize("batch,N,V,W,sigma", [
    (1, 4, 1024, 2, 3.0), (3, 5, 4096, 1, 3.0), (2, 3, 256, 32, 1.0), (1, 16, 151936, 4, 3.0),
    (7, 2, 8192, 8, 0.01), (1, 1, 4, 3, 1.0), (2, 2, 20000, 16, 5.0), (33, 3, 2048, 4, 3.0)])
def test_topw_random(batch, N, V, W, sigma):
    rng = np.random.default_rng(V + W)
    x = (rng.standard_normal((batch, N, V)) * sigma).astype(np.float32)
    tok_o, logp_o = oracle.topw(x, W)
    tok, logp = jtree.jt_topw(torch.from_numpy(x).to(DEV), W)
    assert np.array_equal(to_np(tok), tok_o)
    assert np.abs(to_np(logp) - logp_o).max() <= LOGP_ABS


@pytest.mark.parametrize("rows,V,W,ent", [
    (4, 60004, 4, False), (4, 60004, 4, True), (3, 151936, 32, True), (1, 28672, 1, False),
    (2, 100000, 8, True), (5, 49156, 16, False), (640, 16384, 16, True), (600, 12292, 2, False)])
def test_topw_streaming_shapes(rows, V, W, ent):
    """Segments longer than the register-resident scan holds.

    Few rows take the shared-memory ring, many rows the register double
    buffer; the segment lengths leave ragged last batches (down to one
    float4 in one lane). Row 0 starts with a run of -inf, row 1 holds
    integer values (ties everywhere).
    """
    rng = np.random.default_rng(rows * 7 + V + W)
    x = (rng.standard_normal((rows, 1, V)) * 3.0).astype(np.float32)
    x[0, 0, : V // 5] = -np.inf
    if rows > 1:
        x[1, 0] = rng.integers(-4, 4, V).astype(np.float32)
    tok_o, logp_o = oracle.topw(x, W)
    xd = torch.from_numpy(x).to(DEV)
    if ent:
        tok, logp, h = jtree.jt_topw(xd, W, with_entropy=True)
        assert np.abs(to_np(h) - oracle.row_entropy(x)).max() <= 2e-4
    else:
        tok, logp = jtree.jt_topw(xd, W)
    assert np.array_equal(to_np(tok), tok_o)
    assert np.abs(to_np(logp) - logp_o).max() <= LOGP_ABS


def test_topw_ties_and_neg_inf():
    V = 4096
    x = np.zeros((4, 1, V), np.float32)
    x[0, 0, ::7] = 1.0                       # many exact ties at the top
    x[1] = -np.inf
    x[1, 0, [5, 4000, 17]] = [0.5, 0.5, -3.0]  # -inf everywhere else
    x[2, 0] = np.float32(-0.0)
    x[2, 0, 1::2] = 0.0                       # -0 == +0: lower id first
    x[3] = np.random.default_rng(0).integers(-3, 3, V).astype(np.float32)  # integer ties
    for W in (1, 4, 8, 32):
        tok_o, logp_o = oracle.topw(x, W)
        tok, logp = jtree.jt_topw(torch.from_numpy(x).to(DEV), W)
        assert np.array_equal(to_np(tok), tok_o), W
        got = to_np(logp)
        fin = np.isfinite(logp_o)
        assert np.array_equal(np.isfinite(got), fin)
        assert np.abs(got[fin] - logp_o[fin]).max() <= LOGP_ABS


@pytest.mark.parametrize("batch,N,W,B", [(1, 4, 2, 16), (5, 16, 4, 256), (3, 64, 1, 64),
                                         (9, 8, 4, 64), (2, 16, 32, 255), (4, 3, 3, 33),
                                         (1, 1, 8, 5), (6, 2, 2, 31), (2, 64, 2, 256),
                                         # width 1: chains cut by the budget or by the depth
                                         (2, 20, 1, 7), (3, 5, 1, 40), (1, 1, 1, 1)])
def test_expand_and_mask_random(batch, N, W, B):
    rng = np.random.default_rng(batch * 1000 + N * 10 + W + B)
    tok = rng.integers(0, 50000, (batch, N, W)).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    logp[::2] = np.round(logp[::2] * 2) / 2  # exact ties in half the sequences
    ref = oracle.tree_expand(tok, logp, B)
    tree = jtree.jt_tree_expand(torch.from_numpy(tok).to(DEV), torch.from_numpy(logp).to(DEV), B)
    for k in ("parent", "token", "depth", "n_nodes"):
        assert np.array_equal(to_np(tree[k]), ref[k]), k
    assert np.array_equal(to_np(tree["score"]).view(np.uint32), ref["score"].view(np.uint32))
    mask = jtree.jt_tree_mask(tree["parent"], tree["n_nodes"])
    assert np.array_equal(u32(mask), oracle.tree_mask(ref["parent"], ref["n_nodes"]))


def _increments(kind, rng, shape):
    """Candidate score increments of one shape family (binary32)."""
    if kind == "unsorted":          # ranks not in increment order
        x = -rng.exponential(1.0, shape)
    elif kind == "near-zero":       # many rounds; exact zeros tie with their parents
        x = -np.sort(rng.exponential(0.05, shape), axis=-1)
        x[..., 0] = np.where(rng.random(shape[:-1]) < 0.3, 0.0, x[..., 0])
    elif kind == "equal":           # every node of a depth ties: level order by id
        x = np.broadcast_to(-rng.exponential(1.0, shape[:-1])[..., None], shape).copy()
    elif kind == "positive":        # increments above 0: children outscore parents
        x = rng.normal(0.0, 1.0, shape)
    elif kind == "neg-inf":         # -inf candidates (a row with fewer finite tokens than W)
        x = -np.sort(rng.exponential(1.0, shape), axis=-1)
        x[..., -1] = -np.inf
        x[:, ::3, 1:] = -np.inf
    else:                           # one dominant token per depth
        x = -np.sort(rng.exponential(4.0, shape), axis=-1)
        x[..., 0] = -rng.exponential(0.01, shape[:-1])
    return x.astype(np.float32)


@pytest.mark.parametrize("kind", ["unsorted", "near-zero", "equal", "positive", "neg-inf",
                                  "dominant"])
@pytest.mark.parametrize("batch,N,W,B", [(3, 16, 4, 256), (5, 8, 4, 64), (2, 64, 2, 255),
                                         (4, 6, 32, 200), (7, 3, 3, 33),
                                         # more than 16 pops (rounds): depth 1 and 2 only,
                                         # width 8 over 64 depths, width 15 (one warp a block)
                                         (2, 1, 4, 100), (3, 2, 2, 200), (2, 64, 8, 256),
                                         (2, 40, 15, 256)])
def test_expand_increment_shapes(kind, batch, N, W, B):
    """Expansion is the heap's best-first order whatever the increments look like."""
    rng = np.random.default_rng(B * 31 + N * 7 + W + len(kind))
    tok = rng.integers(0, 50000, (batch, N, W)).astype(np.int32)
    logp = _increments(kind, rng, (batch, N, W))
    ref = oracle.tree_expand(tok, logp, B)
    tree = jtree.jt_tree_expand(torch.from_numpy(tok).to(DEV), torch.from_numpy(logp).to(DEV), B)
    for k in ("parent", "token", "depth", "n_nodes"):
        assert np.array_equal(to_np(tree[k]), ref[k]), k
    assert np.array_equal(to_np(tree["score"]).view(np.uint32), ref["score"].view(np.uint32))


@pytest.mark.parametrize("B", [1, 2, 31, 32, 33, 100, 255, 256])
def test_mask_random_trees(B):
    rng = np.random.default_rng(B)
    batch = 7
    n = rng.integers(0, B + 1, batch).astype(np.int32)
    n[0] = B
    parent = np.stack([random_tree(rng, B, B) for _ in range(batch)])
    mask = jtree.jt_tree_mask(torch.from_numpy(parent).to(DEV), torch.from_numpy(n).to(DEV))
    assert np.array_equal(u32(mask), oracle.tree_mask(parent, n))


ATTN_CASES = [
    # batch, B, n_nodes, hq, hkv, D, prefix lengths, paged
    (1, 16, [16], 4, 1, 64, [128], False),
    (2, 33, [33, 7], 8, 2, 128, [0, 1], False),
    (3, 64, [64, 40, 1], 32, 8, 128, [15, 16, 17], True),
    (2, 256, [256, 129], 16, 1, 64, [300, 0], True),
    (1, 1, [1], 2, 2, 128, [1000], False),
    (4, 48, [48, 48, 0, 20], 32, 4, 128, [127, 128, 129, 513], True),
    (2, 128, [128, 77], 8, 8, 64, [2049, 31], False),
    # Few units and >= 16 key tiles: 16-CTA split, ragged live rows, ranks
    # without a tile (the short second sequence).
    (2, 24, [19, 5], 16, 2, 128, [2000, 100], False),
    (1, 40, [37], 8, 1, 64, [2100], True),
]


@pytest.mark.parametrize("batch,B,n_list,hq,hkv,D,lens,paged", ATTN_CASES)
def test_attention_random(batch, B, n_list, hq, hkv, D, lens, paged):
    rng = np.random.default_rng(B + hq + D)
    g = torch.Generator().manual_seed(B * 7 + D)
    n = np.array(n_list, np.int32)
    parent = np.stack([random_tree(rng, B, int(n[b])) for b in range(batch)])
    mask = oracle.tree_mask(parent, n)
    Lmax = max(max(lens), 1)
    q = bf16((batch, B, hq, D), g)
    kt, vt = bf16((batch, B, hkv, D), g), bf16((batch, B, hkv, D), g)
    lens_np = np.array(lens, np.int32)
    if paged:
        max_pages = (Lmax + 15) // 16
        n_pages = batch * max_pages + 3
        bt = rng.permutation(n_pages)[: batch * max_pages].reshape(batch, max_pages).astype(np.int32)
        kc, vc = bf16((n_pages, 16, hkv, D), g), bf16((n_pages, 16, hkv, D), g)
    else:
        bt = None
        kc, vc = bf16((batch, Lmax, hkv, D), g), bf16((batch, Lmax, hkv, D), g)
    ref = oracle.tree_attn(q, kt, vt, kc, vc, lens_np, n, mask, hq=hq, hkv=hkv, block_table=bt)
    d = lambda t: t.to(DEV)
    ex = jtree.Exec(DEV)
    # NaN-filled: a row the kernels never write fails the comparison.
    out = torch.full((batch, B, hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    jtree.jt_tree_attn(d(q), d(kt), d(vt), d(kc), d(vc), d(torch.from_numpy(lens_np)),
                       d(torch.from_numpy(n)), d(torch.from_numpy(mask.view(np.int32))), out=out,
                       block_table=None if bt is None else d(torch.from_numpy(bt)), exec=ex)
    assert ex.read_error() == 0
    check_attn(out.float().cpu().numpy(), ref)


@pytest.mark.parametrize("batch,N,W,B,V", [(4, 4, 2, 16, 64), (3, 16, 4, 256, 1024),
                                           (5, 8, 1, 8, 4096), (2, 64, 2, 200, 512),
                                           (17, 16, 4, 128, 2048),
                                           # all-rows argmax over long, streamed segments
                                           # (136 and 104 rows, 4 and 2 segments per row)
                                           (3, 16, 1, 16, 151936), (2, 8, 2, 12, 100000)])
def test_accept_random(batch, N, W, B, V):
    rng = np.random.default_rng(N * W * B)
    batch = max(batch, 8)
    tok = np.stack([np.stack([rng.choice(V, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    tree = oracle.tree_expand(tok, logp, B)
    target = rng.standard_normal((batch, B + 1, V)).astype(np.float32)
    # Bias rows towards a child's token so that acceptance walks several levels.
    for b in range(batch):
        for u in range(-1, int(tree["n_nodes"][b])):
            kids = [v for v in range(tree["n_nodes"][b]) if tree["parent"][b, v] == u]
            row = target[b, 0 if u < 0 else 1 + u]
            if kids and rng.random() < 0.95:
                row[tree["token"][b, rng.choice(kids)]] = row.max() + 1
            if rng.random() < 0.25:  # an exact tie at the maximum, either side of the argmax
                row[rng.integers(V)] = row.max()
    ref = oracle.tree_accept(target, tree["parent"], tree["token"], tree["n_nodes"], N)
    d = lambda a: torch.from_numpy(a).to(DEV)
    got = jtree.jt_tree_accept(d(target), d(tree["parent"]), d(tree["token"]), d(tree["n_nodes"]),
                               N)
    for k in ref:
        assert np.array_equal(to_np(got[k]), ref[k]), k
    assert ref["acc_len"].max() >= 2


def test_device_checks_raise_flags_without_faulting():
    ex = jtree.Exec(DEV)
    # Bad parent (points forward) -> JT_DEVERR_PARENT, zero mask rows.
    parent = torch.tensor([[-1, 2, 0]], dtype=torch.int32, device=DEV)
    nn = torch.tensor([3], dtype=torch.int32, device=DEV)
    mask = jtree.jt_tree_mask(parent, nn, exec=ex)
    assert ex.read_error() & jtree.JT_DEVERR_PARENT
    assert not mask.any()
    # n_nodes > B -> JT_DEVERR_NNODES.
    jtree.jt_tree_mask(parent, torch.tensor([9], dtype=torch.int32, device=DEV), exec=ex)
    assert ex.read_error() & jtree.JT_DEVERR_NNODES
    # Token outside the vocabulary in acceptance -> JT_DEVERR_TOKEN, acc_len 0, bonus -1.
    target = torch.zeros((1, 4, 8), dtype=torch.float32, device=DEV)
    good_parent = torch.tensor([[-1, 0, 1]], dtype=torch.int32, device=DEV)
    token = torch.tensor([[0, 99, 1]], dtype=torch.int32, device=DEV)
    acc = jtree.jt_tree_accept(target, good_parent, token, nn, 3, exec=ex)
    assert ex.read_error() & jtree.JT_DEVERR_TOKEN
    assert int(acc["acc_len"][0]) == 0 and int(acc["bonus"][0]) == -1
    # Page id outside the pool and prefix longer than the table -> flags, zero output.
    B, hq, hkv, D = 4, 4, 1, 64
    g = torch.Generator().manual_seed(1)
    q = bf16((2, B, hq, D), g).to(DEV)
    kt, vt = bf16((2, B, hkv, D), g).to(DEV), bf16((2, B, hkv, D), g).to(DEV)
    kc, vc = bf16((4, 16, hkv, D), g).to(DEV), bf16((4, 16, hkv, D), g).to(DEV)
    bt = torch.tensor([[0, 7], [1, 2]], dtype=torch.int32, device=DEV)   # page 7 does not exist
    lens = torch.tensor([20, 40], dtype=torch.int32, device=DEV)         # 40 > 2 pages * 16
    nn2 = torch.tensor([4, 4], dtype=torch.int32, device=DEV)
    m = jtree.jt_tree_mask(torch.tensor([[-1, 0, 1, 2]] * 2, dtype=torch.int32, device=DEV), nn2)
    out = jtree.jt_tree_attn(q, kt, vt, kc, vc, lens, nn2, m, block_table=bt, exec=ex)
    err = ex.read_error()
    assert err & jtree.JT_DEVERR_PAGE and err & jtree.JT_DEVERR_PREFIX
    assert not out.float().abs().sum().item()
    assert ex.read_error() == 0  # reading cleared the word


def test_empty_batch_and_host_validation():
    ex = jtree.Exec(DEV)
    z = torch.zeros((0, 4, 1024), dtype=torch.float32, device=DEV)
    tok, logp = jtree.jt_topw(z, 2, exec=ex)
    assert tok.shape == (0, 4, 2)
    with pytest.raises(jtree.JtError):
        jtree.jt_topw(torch.zeros((1, 1, 8), dtype=torch.float32, device=DEV), 9)
    with pytest.raises(jtree.JtError):
        jtree.jt_topw(torch.zeros((1, 1, 6), dtype=torch.float32, device=DEV), 2)  # V % 4
    with pytest.raises(jtree.JtError):
        jtree.jt_tree_expand(torch.zeros((1, 2, 2), dtype=torch.int32, device=DEV),
                             torch.zeros((1, 2, 2), dtype=torch.float32, device=DEV), 300)
    assert ex.read_error() == 0


# Many units (sequence x KV head x 256-row block): the length-ordered schedule.
# 96 units -> up to 4 chunks per unit merged by the last chunk to finish;
# 320 units -> one CTA per unit, longest first. Ragged prefixes (0, 1, page
# and tile edges, long), n_nodes 0 / 1 / B, paged and contiguous; all rows
# of a few sequences plus a random sample of the rest are compared.
@pytest.mark.parametrize("batch,hq,hkv,B,paged,Lmax", [(24, 16, 4, 64, True, 3000),
                                                       (24, 16, 4, 64, False, 2100),
                                                       (80, 8, 4, 16, True, 1500)])
def test_attention_balanced_schedule(batch, hq, hkv, B, paged, Lmax):
    rng = np.random.default_rng(batch + hq + B + paged)
    g = torch.Generator().manual_seed(batch * 3 + B)
    D = 128
    n = rng.integers(0, B + 1, batch).astype(np.int32)
    n[:3] = [B, 0, 1]
    lens = rng.integers(0, Lmax + 1, batch).astype(np.int32)
    lens[:6] = [Lmax, 0, 1, 127, 128, 129]
    parent = np.stack([random_tree(rng, B, int(n[b])) for b in range(batch)])
    mask = oracle.tree_mask(parent, n)
    q = bf16((batch, B, hq, D), g)
    kt, vt = bf16((batch, B, hkv, D), g), bf16((batch, B, hkv, D), g)
    if paged:
        max_pages = (Lmax + 15) // 16
        n_pages = batch * max_pages + 3
        bt = rng.permutation(n_pages)[: batch * max_pages].reshape(batch, max_pages).astype(np.int32)
        kc, vc = bf16((n_pages, 16, hkv, D), g), bf16((n_pages, 16, hkv, D), g)
    else:
        bt = None
        kc, vc = bf16((batch, Lmax, hkv, D), g), bf16((batch, Lmax, hkv, D), g)
    d = lambda t: t.to(DEV)
    ex = jtree.Exec(DEV)
    out = torch.full((batch, B, hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    jtree.jt_tree_attn(d(q), d(kt), d(vt), d(kc), d(vc), d(torch.from_numpy(lens)),
                       d(torch.from_numpy(n)), d(torch.from_numpy(mask.view(np.int32))), out=out,
                       block_table=None if bt is None else d(torch.from_numpy(bt)), exec=ex)
    assert ex.read_error() == 0
    rows = [(b, v, h) for b in (0, 1, 2) for v in range(B) for h in range(hq)]
    rows += [(int(b), int(v), int(h)) for b, v, h in
             zip(rng.integers(0, batch, 1500), rng.integers(0, B, 1500), rng.integers(0, hq, 1500))]
    rows = np.array(rows, np.int32)
    ref = oracle.tree_attn(q, kt, vt, kc, vc, lens, n, mask, hq=hq, hkv=hkv, block_table=bt,
                           rows=rows)
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    check_attn(got, ref)
    # Rows of unused budget slots are exactly zero.
    o = out.float().cpu().numpy()
    for b in range(batch):
        assert not o[b, n[b]:].any()
