"""The C-ABI library loads and exports every symbol include/jtree.h declares.

Runs without a GPU: only symbol lookup, the status strings, the workspace
size queries and argument checks that fail before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from tree_causal_verification_gb300 import build, jtree

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "jtree.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"JT_API\s+[\w\s\*]+?\b(jt_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return jtree.load()


def test_header_declares_the_five_calls():
    syms = declared_symbols()
    for name in ("jt_topw", "jt_tree_expand", "jt_tree_mask", "jt_tree_attn", "jt_tree_accept"):
        assert name in syms
    assert set(syms) <= set(jtree.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in jtree.STATUS_NAMES.items():
        assert lib.jt_status_str(code).decode().startswith(name)


def test_host_validation_needs_no_gpu(lib):
    ex = jtree.jt_exec()
    # W = 0, B = 300, bad head_dim: rejected before any CUDA call.
    assert lib.jt_topw(None, 1, 1, 8, 0, None, None, ctypes.byref(ex)) == 1
    assert lib.jt_tree_expand(None, None, 1, 4, 2, 300, None, None, None, None, None,
                              ctypes.byref(ex)) == 1
    assert lib.jt_tree_mask(None, None, 1, 0, None, ctypes.byref(ex)) == 1
    args = jtree.jt_attn_args(1, 16, 32, 8, 96, 0.0)
    assert lib.jt_tree_attn(ctypes.byref(args), ctypes.byref(ex)) == 2
    args = jtree.jt_attn_args(1, 16, 30, 8, 128, 0.0)  # hq % hkv != 0
    assert lib.jt_tree_attn(ctypes.byref(args), ctypes.byref(ex)) == 1
    assert lib.jt_tree_accept(None, None, None, None, 1, 16, 0, 1024, None, None, None, None,
                              ctypes.byref(ex)) == 1
    assert lib.jt_read_device_error(None, None) == 1


def test_workspace_queries(lib):
    # Chains / small trees: per-row argmax scratch; wide trees walk the path and need none.
    assert lib.jt_tree_accept_workspace_bytes(64, 16, 16, 151936) >= 64 * 17 * 4
    assert lib.jt_tree_accept_workspace_bytes(64, 16, 16, 151936) % 256 == 0
    assert lib.jt_tree_accept_workspace_bytes(64, 128, 16, 151936) == 0
    assert lib.jt_topw_workspace_bytes(1, 16, 151936, 4) == 0


def _attn_args(batch, B, hq, hkv, D, max_prefix):
    a = jtree.jt_attn_args(batch, B, hq, hkv, D, 0.0)
    for f in ("q", "k_tree", "v_tree", "k_cache", "v_cache", "prefix_len", "n_nodes", "mask",
              "out"):
        setattr(a, f, 4096)  # never dereferenced by the query
    a.max_prefix = max_prefix
    return a


def test_attn_workspace_query(lib):
    # Few work units (one sequence, 8 KV heads, one 256-row block each): the key
    # range is split over a cluster and the fp32 partials need scratch, bounded
    # by one partial per SM. Many units (64 sequences x 4 KV heads x 4 blocks
    # of 32 nodes x 8 heads) cover the SMs more than twice: no split, only the
    # length order of the units (8 bytes per unit).
    small = lib.jt_tree_attn_workspace_bytes(ctypes.byref(_attn_args(1, 16, 32, 8, 128, 2048)))
    assert small > 0 and small % 256 == 0
    assert small <= 1024 * (256 * 128 + 1024) * 4
    assert lib.jt_tree_attn_workspace_bytes(
        ctypes.byref(_attn_args(64, 128, 32, 4, 128, 16384))) == 64 * 4 * 4 * 8
    # In between (96 units), long units are cut into chunks: one partial per
    # chunk slot on top of the order.
    mid = lib.jt_tree_attn_workspace_bytes(ctypes.byref(_attn_args(24, 64, 16, 4, 128, 3000)))
    assert mid >= 96 * 8 + 96 * 2 * (256 * 128 + 512) * 4
    # A single key tile cannot be split.
    assert lib.jt_tree_attn_workspace_bytes(ctypes.byref(_attn_args(1, 16, 32, 8, 128, 0))) == 0
