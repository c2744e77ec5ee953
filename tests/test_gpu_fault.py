"""Failure detection without a GPU fault: bounded waits that run out.

Every wait of the tcgen05 kernels (tree attention, LM head + top-W) on an
mbarrier gives up after a cycle budget, raises JT_DEVERR_TIMEOUT in the
device error word, waits (with the default budget) for the TMA loads and
tensor-core operations its CTA already issued, frees its tensor memory and
finishes. These tests shrink the budget to one cycle through the library's
test hook, so the first wait on a phase that is not already complete gives
up; nothing is left waiting. They then restore the default and check that
the next call on the same context is correct.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import LOGP_ABS, check_attn, to_np
from tree_causal_verification_gb300 import jtree, synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def tiny_inputs():
    w = synth.WORKLOADS["tiny"]
    kv = synth.kv_inputs(w, 5, "cpu")
    draft = synth.draft_logits(w, 5, "cpu")[:, : w.N].contiguous()
    tok, logp = oracle.topw(draft.numpy(), w.W)
    tree = oracle.tree_expand(tok, logp, w.B)
    mask = oracle.tree_mask(tree["parent"], tree["n_nodes"])
    return w, kv, tree, mask


def run_attn(w, kv, tree, mask, ex):
    d = lambda t: t.to(DEV)
    out = torch.full((w.batch, w.B, w.hq, w.D), float("nan"), dtype=torch.bfloat16, device=DEV)
    jtree.jt_tree_attn(d(kv["q"]), d(kv["k_tree"]), d(kv["v_tree"]), d(kv["k_cache"]),
                       d(kv["v_cache"]), d(kv["prefix_len"]), d(torch.from_numpy(tree["n_nodes"])),
                       d(torch.from_numpy(mask.view(np.int32))), out=out, exec=ex)
    return out


def test_attention_wait_timeout_then_recovers():
    w, kv, tree, mask = tiny_inputs()
    ex = jtree.Exec(DEV)
    jtree.jt_set_wait_budget(1)
    try:
        run_attn(w, kv, tree, mask, ex)
        err = ex.read_error()
    finally:
        jtree.jt_set_wait_budget(0)
    assert err & jtree.JT_DEVERR_TIMEOUT, err
    # Default budget again: the same context gives the oracle's result.
    out = run_attn(w, kv, tree, mask, ex)
    assert ex.read_error() == 0
    ref = oracle.tree_attn(kv["q"], kv["k_tree"], kv["v_tree"], kv["k_cache"], kv["v_cache"],
                           kv["prefix_len"].numpy(), tree["n_nodes"], mask, hq=w.hq, hkv=w.hkv)
    check_attn(out.float().cpu().numpy(), ref, "after timeout")


def test_lmhead_wait_timeout_then_recovers():
    rows, d, V, W = 16, 256, 1024, 4
    rng = np.random.default_rng(11)
    h = rng.integers(-2, 3, (rows, d)) / 4.0
    wl = rng.integers(-4, 5, (V, d)) / 8.0
    hd = torch.from_numpy(h.astype(np.float32)).to(DEV).to(torch.bfloat16)
    wd = torch.from_numpy(wl.astype(np.float32)).to(DEV).to(torch.bfloat16)
    ex = jtree.Exec(DEV)
    jtree.jt_set_wait_budget(1)
    try:
        jtree.jt_lmhead_topw(hd, wd, W, exec=ex)
        err = ex.read_error()
    finally:
        jtree.jt_set_wait_budget(0)
    assert err & jtree.JT_DEVERR_TIMEOUT, err
    tok, logp = jtree.jt_lmhead_topw(hd, wd, W, exec=ex)
    assert ex.read_error() == 0
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    tok_o, logp_o, _ = oracle.lmhead_topw(bits(hd), bits(wd), W)
    assert np.array_equal(to_np(tok), tok_o)
    assert np.abs(to_np(logp) - logp_o).max() <= LOGP_ABS
