"""GPU vs oracle on the five step workloads, at their full sizes.

Bit-exact: top-W indices, tree topology (parent/token/depth/n_nodes), masks,
acceptance. Within tolerance: log-probs (1e-5 abs) and bf16 attention
(max-abs 2e-2, mean-abs 2e-3 against the fp64 oracle). Attention is checked
on every row of the batch-1 workloads (all 8192 (node, head) rows of the
256-node tree). For the batched workloads every row of four whole sequences
(the longest prefix, the shortest and two drawn at random: every KV head,
tile pair and key-split chunk of those sequences) plus sampled rows of all
the others, always through the same C-ABI calls bench.py times.
"""
import numpy as np
import pytest
import torch

from parity_util import LOGP_ABS, Case, check_attn, gather_rows, to_np, u32
from tree_causal_verification_gb300 import jtree, synth
from tree_causal_verification_gb300.step import StepBuffers, run_step

pytestmark = pytest.mark.gpu

FULL_ATTN = {"tiny", "qwen3-8b-chain", "high-budget"}


def attn_rows(case):
    """Rows compared for a workload (see the module docstring)."""
    w = case.w
    if w.name in FULL_ATTN:
        return case.whole_sequences(range(w.batch))
    L = to_np(case.kv["prefix_len"])
    rng = np.random.default_rng(7)
    seqs = {int(np.argmax(L)), int(np.argmin(L))}
    rest = [b for b in range(w.batch) if b not in seqs]
    seqs |= set(rng.choice(rest, 2, replace=False).tolist())
    whole = case.whole_sequences(sorted(seqs))
    sampled = case.sample_rows(case.tree["n_nodes"])
    sampled = sampled[~np.isin(sampled[:, 0], sorted(seqs))]
    return np.concatenate([whole, sampled])


@pytest.fixture(scope="module", params=synth.WORKLOAD_ORDER)
def case(request):
    torch.cuda.set_device(0)
    c = Case(synth.WORKLOADS[request.param], seed=0, device="cuda:0")
    yield c
    del c
    torch.cuda.empty_cache()


def test_topw(case):
    w = case.w
    ex = jtree.Exec(case.dev)
    tok, logp = jtree.jt_topw(case.inp["draft"], w.W, exec=ex)
    assert ex.read_error() == 0
    assert np.array_equal(to_np(tok), case.tok)
    assert np.abs(to_np(logp) - case.logp).max() <= LOGP_ABS


def test_expand_on_oracle_candidates(case):
    """Same tok/logp bytes on both sides: the whole tree must be bit-identical."""
    w = case.w
    ex = jtree.Exec(case.dev)
    tree = jtree.jt_tree_expand(torch.from_numpy(case.tok).to(case.dev),
                                torch.from_numpy(case.logp).to(case.dev), w.B, exec=ex)
    assert ex.read_error() == 0
    for k in ("parent", "token", "depth", "n_nodes"):
        assert np.array_equal(to_np(tree[k]), case.tree[k]), k
    assert np.array_equal(to_np(tree["score"]).view(np.uint32), case.tree["score"].view(np.uint32))


def test_step_end_to_end(case):
    """The five calls chained on the device (bench.py's launch sequence)."""
    w = case.w
    ex = jtree.Exec(case.dev)
    buf = StepBuffers(w, case.dev)
    buf.attn_out.fill_(float("nan"))   # a row the kernels never write fails below
    buf = run_step(w, case.inp, buf, ex)
    torch.cuda.synchronize()
    assert ex.read_error() == 0
    for k in ("parent", "token", "depth", "n_nodes"):
        assert np.array_equal(to_np(buf.tree[k]), case.tree[k]), k
    np.testing.assert_allclose(to_np(buf.tree["score"]), case.tree["score"], rtol=0, atol=1e-4)
    assert np.array_equal(u32(buf.mask), case.mask)
    rows = attn_rows(case)
    ref = case.oracle_attn(rows)
    check_attn(gather_rows(buf.attn_out, rows), ref, w.name)
    acc = case.oracle_accept()
    for k in acc:
        assert np.array_equal(to_np(buf.acc[k]), acc[k]), k
    # Rows of unused budget slots are zero.
    n = case.tree["n_nodes"]
    out = buf.attn_out.float().cpu().numpy()
    for b in range(w.batch):
        assert not out[b, n[b]:].any()
