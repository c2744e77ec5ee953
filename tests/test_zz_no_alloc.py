"""jt_tree_accept_noalloc: acceptance for callers that cannot allocate.

Such callers (runtimes whose device memory belongs to another allocator,
plain C hosts with no device allocator, code that must not call cudaMalloc
because it synchronises the device) cannot hand the library a workspace;
this entry point uses a fixed device array inside the library instead. Its
results must equal the oracle's and jt_tree_accept's (which takes a caller
workspace) bit for bit, call after call, even though every call reuses the
same array. Collected last (file name) so that a stop-at-first-failure run
has already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tree_causal_verification_gb300 import jtree

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def make_case(seed, batch, N, W, B, V):
    rng = np.random.default_rng(seed)
    tok = np.stack([np.stack([rng.choice(V, W, replace=False) for _ in range(N)])
                    for _ in range(batch)]).astype(np.int32)
    logp = -np.sort(rng.exponential(1.0, (batch, N, W)), axis=-1).astype(np.float32)
    tree = oracle.tree_expand(tok, logp, B)
    target = rng.standard_normal((batch, B + 1, V)).astype(np.float32)
    for b in range(batch):  # make acceptance walk several levels
        for u in range(-1, int(tree["n_nodes"][b])):
            kids = [v for v in range(tree["n_nodes"][b]) if tree["parent"][b, v] == u]
            if kids and rng.random() < 0.9:
                row = target[b, 0 if u < 0 else 1 + u]
                row[tree["token"][b, rng.choice(kids)]] = row.max() + 1
    ref = oracle.tree_accept(target, tree["parent"], tree["token"], tree["n_nodes"], N)
    d = lambda a: torch.from_numpy(a).to(DEV)
    return (d(target), d(tree["parent"]), d(tree["token"]), d(tree["n_nodes"]), N), ref


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    torch.cuda.set_device(0)
    ex = jtree.Exec(DEV)
    # Two different shapes in a row that both keep per-row argmaxes in the
    # library's array (chains and trees not much wider than a root path): the
    # second call reuses, and must not be confused by, what the first left
    # there. A third, wide tree walks the path and needs no array at all.
    for seed, shape in ((1, (12, 16, 1, 16, 4096)), (2, (5, 8, 2, 24, 151936)),
                        (3, (16, 16, 4, 128, 2048))):
        args, ref = make_case(seed, *shape)
        want = jtree.jt_tree_accept(*args, exec=ex)
        got = jtree.jt_tree_accept_noalloc(*args, exec=ex)
        torch.cuda.synchronize()
        assert ex.read_error() == 0
        for k in want:
            assert np.array_equal(got[k].cpu().numpy(), ref[k]), (seed, k)
            assert torch.equal(got[k], want[k]), (seed, k)
        assert int(ref["acc_len"].max()) >= 2


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = jtree.load()
    ex = jtree.jt_exec()
    # batch * (B + 1) = 300 * 257 > 65536: refused before any launch.
    rc = lib.jt_tree_accept_noalloc(None, None, None, None, 300, 256, 16, 1024, None, None, None,
                                    None, ctypes.byref(ex))
    assert rc == 2  # JT_ERR_UNSUPPORTED
