"""CPU oracle for the tree-drafting hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` legs may import this package. The product library never
does: it shares no code with the oracle and must not fall back to it.

The arithmetic lives in ``jtree_oracle.cpp`` (plain single-threaded C++17);
this module builds it with g++ and wraps it with ctypes over numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jtree_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libjtree_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u64p = ctypes.POINTER(ctypes.c_uint64)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (plain g++, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_tree_mask.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, _u32p]
            lib.orc_tree_attn.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                _u16p, _u16p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, _i32p, _i32p, _u32p, _i32p, ctypes.c_int, _f64p]
            lib.orc_topw.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     _i32p, _f32p]
            lib.orc_tree_expand.argtypes = [_i32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, _i32p, _i32p, _i32p, _f32p, _i32p]
            lib.orc_tree_accept.argtypes = [_f32p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, _i32p, _i32p, _i32p, _i32p]
            lib.orc_row_entropy.argtypes = [_f32p, ctypes.c_long, ctypes.c_int, _f32p]
            lib.orc_tree_accept_sampled.argtypes = [
                _f32p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_float, ctypes.c_uint64, _i32p, _i32p, _i32p, _i32p]
            lib.orc_series_ln.argtypes = [_f32p, ctypes.c_long, _f32p]
            lib.orc_splitmix64.argtypes = [ctypes.c_uint64, _u64p, ctypes.c_long, _u64p]
            lib.orc_gumbel.argtypes = [ctypes.c_uint64, _u64p, ctypes.c_long, _f32p]
            lib.orc_tree_expand_scored.argtypes = [
                _i32p, _f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_float, _i32p, _i32p, _i32p, _f32p, _i32p]
            lib.orc_tree_commit_kv.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                _u16p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, _i32p, _i32p, _i32p, _i32p]
            for f in (lib.orc_tree_mask, lib.orc_tree_attn, lib.orc_topw, lib.orc_tree_expand,
                      lib.orc_tree_accept, lib.orc_tree_commit_kv, lib.orc_row_entropy,
                      lib.orc_tree_expand_scored, lib.orc_tree_accept_sampled):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctype) if a is not None else None


def _check(rc, name):
    if rc != 0:
        raise OracleError(f"{name} returned {rc}")


def tree_mask(parent, n_nodes):
    """parent [batch][B] int32, n_nodes [batch] -> mask uint32 [batch][B][ceil(B/32)]."""
    parent = _arr(parent, np.int32)
    n_nodes = _arr(n_nodes, np.int32)
    batch, B = parent.shape
    mask = np.zeros((batch, B, (B + 31) // 32), np.uint32)
    _check(_load().orc_tree_mask(_ptr(parent, _i32p), _ptr(n_nodes, _i32p), batch, B,
                                 _ptr(mask, _u32p)), "orc_tree_mask")
    return mask


def _bf16_bits(a):
    """Accept uint16 bit patterns (numpy) or a torch bf16 tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return _arr(a, np.uint16)


def tree_attn(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, mask, *,
              hq, hkv, block_table=None, page_size=16, scale=0.0, rows=None):
    """Tree-causal GQA attention in double precision.

    q [batch][B][hq][D], k/v_tree [batch][B][hkv][D] (bf16 bits),
    k/v_cache contiguous [batch][Lmax][hkv][D] or paged [pages][page_size][hkv][D].
    rows: optional int array [n][3] of (b, v, h); returns [n][D] float64, else
    [batch][B][hq][D].
    """
    q, k_tree, v_tree = _bf16_bits(q), _bf16_bits(k_tree), _bf16_bits(v_tree)
    k_cache, v_cache = _bf16_bits(k_cache), _bf16_bits(v_cache)
    prefix_len = _arr(prefix_len, np.int32)
    n_nodes = _arr(n_nodes, np.int32)
    mask = _arr(mask, np.uint32)
    batch, B = q.shape[0], q.shape[1]
    D = q.shape[-1]
    if block_table is not None:
        block_table = _arr(block_table, np.int32)
        max_pages = block_table.shape[1]
        max_prefix = 0
        n_pool_pages = k_cache.shape[0]
        page_size = k_cache.shape[1]
    else:
        max_pages = 0
        max_prefix = k_cache.shape[1]
        n_pool_pages = 0
    if rows is not None:
        rows = _arr(rows, np.int32).reshape(-1, 3)
        out = np.zeros((rows.shape[0], D), np.float64)
        n_rows = rows.shape[0]
    else:
        out = np.zeros((batch, B, hq, D), np.float64)
        n_rows = 0
    rc = _load().orc_tree_attn(batch, B, hq, hkv, D, float(scale),
                               _ptr(q, _u16p), _ptr(k_tree, _u16p), _ptr(v_tree, _u16p),
                               _ptr(k_cache, _u16p), _ptr(v_cache, _u16p),
                               _ptr(block_table, _i32p), page_size, max_pages, max_prefix,
                               n_pool_pages, _ptr(prefix_len, _i32p), _ptr(n_nodes, _i32p),
                               _ptr(mask, _u32p), _ptr(rows, _i32p), n_rows, _ptr(out, _f64p))
    _check(rc, "orc_tree_attn")
    return out


def topw(logits, W):
    """logits fp32 [batch][N][V] -> (tok int32 [batch][N][W], logp fp32 [batch][N][W])."""
    logits = _arr(logits, np.float32)
    batch, n_depth, vocab = logits.shape
    tok = np.zeros((batch, n_depth, W), np.int32)
    logp = np.zeros((batch, n_depth, W), np.float32)
    _check(_load().orc_topw(_ptr(logits, _f32p), batch, n_depth, vocab, W, _ptr(tok, _i32p),
                            _ptr(logp, _f32p)), "orc_topw")
    return tok, logp


def tree_expand(tok, logp, B, entropy=None, mode=0, alpha=0.0):
    """Best-first expansion -> dict(parent, token, depth, score, n_nodes).

    mode 0: cumulative log-prob; 1: hybrid (increment logp - alpha*H_d);
    2: entropy only (increment -H_d). entropy: fp32 [batch][n_depth]."""
    tok = _arr(tok, np.int32)
    logp = _arr(logp, np.float32)
    batch, n_depth, W = tok.shape
    if entropy is not None:
        entropy = _arr(entropy, np.float32)
        assert entropy.shape == (batch, n_depth)
    parent = np.zeros((batch, B), np.int32)
    token = np.zeros((batch, B), np.int32)
    depth = np.zeros((batch, B), np.int32)
    score = np.zeros((batch, B), np.float32)
    n_nodes = np.zeros((batch,), np.int32)
    _check(_load().orc_tree_expand_scored(_ptr(tok, _i32p), _ptr(logp, _f32p),
                                          _ptr(entropy, _f32p), batch, n_depth, W, B, int(mode),
                                          float(alpha), _ptr(parent, _i32p), _ptr(token, _i32p),
                                          _ptr(depth, _i32p), _ptr(score, _f32p),
                                          _ptr(n_nodes, _i32p)), "orc_tree_expand_scored")
    return dict(parent=parent, token=token, depth=depth, score=score, n_nodes=n_nodes)


def row_entropy(rows):
    """Shannon entropy (nats) of softmax over the last axis, fp64 -> fp32."""
    rows = _arr(rows, np.float32)
    V = rows.shape[-1]
    out = np.zeros(rows.shape[:-1], np.float32)
    _check(_load().orc_row_entropy(_ptr(rows, _f32p), int(np.prod(rows.shape[:-1])), V,
                                   _ptr(out, _f32p)), "orc_row_entropy")
    return out


def tree_accept(target, parent, token, n_nodes, n_depth):
    """Greedy acceptance -> dict(acc_len, acc_tokens, acc_nodes, bonus)."""
    target = _arr(target, np.float32)
    parent = _arr(parent, np.int32)
    token = _arr(token, np.int32)
    n_nodes = _arr(n_nodes, np.int32)
    batch, B = parent.shape
    vocab = target.shape[-1]
    assert target.shape == (batch, B + 1, vocab)
    acc_len = np.zeros((batch,), np.int32)
    acc_tokens = np.zeros((batch, n_depth), np.int32)
    acc_nodes = np.zeros((batch, n_depth), np.int32)
    bonus = np.zeros((batch,), np.int32)
    _check(_load().orc_tree_accept(_ptr(target, _f32p), _ptr(parent, _i32p), _ptr(token, _i32p),
                                   _ptr(n_nodes, _i32p), batch, B, n_depth, vocab,
                                   _ptr(acc_len, _i32p), _ptr(acc_tokens, _i32p),
                                   _ptr(acc_nodes, _i32p), _ptr(bonus, _i32p)),
           "orc_tree_accept")
    return dict(acc_len=acc_len, acc_tokens=acc_tokens, acc_nodes=acc_nodes, bonus=bonus)


def tree_accept_sampled(target, parent, token, n_nodes, n_depth, temperature, seed):
    """Temperature-T acceptance (one Gumbel-max target draw per visited node)
    -> dict(acc_len, acc_tokens, acc_nodes, bonus). The binary32 reciprocal
    of the temperature is what both sides multiply by."""
    target = _arr(target, np.float32)
    parent = _arr(parent, np.int32)
    token = _arr(token, np.int32)
    n_nodes = _arr(n_nodes, np.int32)
    batch, B = parent.shape
    vocab = target.shape[-1]
    assert target.shape == (batch, B + 1, vocab)
    inv_t = float(np.float32(1.0) / np.float32(temperature))
    acc_len = np.zeros((batch,), np.int32)
    acc_tokens = np.zeros((batch, n_depth), np.int32)
    acc_nodes = np.zeros((batch, n_depth), np.int32)
    bonus = np.zeros((batch,), np.int32)
    _check(_load().orc_tree_accept_sampled(_ptr(target, _f32p), _ptr(parent, _i32p),
                                           _ptr(token, _i32p), _ptr(n_nodes, _i32p), batch, B,
                                           n_depth, vocab, inv_t, int(seed) & (2 ** 64 - 1),
                                           _ptr(acc_len, _i32p), _ptr(acc_tokens, _i32p),
                                           _ptr(acc_nodes, _i32p), _ptr(bonus, _i32p)),
           "orc_tree_accept_sampled")
    return dict(acc_len=acc_len, acc_tokens=acc_tokens, acc_nodes=acc_nodes, bonus=bonus)


def series_ln(x):
    x = _arr(x, np.float32)
    out = np.zeros_like(x)
    _load().orc_series_ln(_ptr(x, _f32p), x.size, _ptr(out, _f32p))
    return out


def splitmix64(seed, k):
    k = _arr(k, np.uint64)
    out = np.zeros_like(k)
    _load().orc_splitmix64(int(seed) & (2 ** 64 - 1), _ptr(k, _u64p), k.size, _ptr(out, _u64p))
    return out


def gumbel(seed, k):
    k = _arr(k, np.uint64)
    out = np.zeros(k.shape, np.float32)
    _load().orc_gumbel(int(seed) & (2 ** 64 - 1), _ptr(k, _u64p), k.size, _ptr(out, _f32p))
    return out


def tree_commit_kv(k_tree, v_tree, k_cache, v_cache, prefix_len, acc_len, acc_nodes,
                   block_table=None, check=True):
    """Append the accepted path's tree K/V rows to the prefix cache.

    k/v_tree [batch][B][hkv][D] and k/v_cache (contiguous [batch][Lmax][hkv][D]
    or paged [pages][page_size][hkv][D]) as bf16 bit patterns (uint16) or
    torch bf16. Returns (k_cache', v_cache', new_prefix_len, rc) on copies;
    the inputs are not modified. check=False returns the oracle's status
    instead of raising on rejected sequences.
    """
    k_tree, v_tree = _bf16_bits(k_tree), _bf16_bits(v_tree)
    k_out, v_out = _bf16_bits(k_cache).copy(), _bf16_bits(v_cache).copy()
    prefix_len = _arr(prefix_len, np.int32)
    acc_len = _arr(acc_len, np.int32)
    acc_nodes = _arr(acc_nodes, np.int32)
    batch, B, hkv, D = k_tree.shape
    n_depth = acc_nodes.shape[1]
    if block_table is not None:
        block_table = _arr(block_table, np.int32)
        max_pages, page_size, n_pool, max_prefix = block_table.shape[1], k_out.shape[1], k_out.shape[0], 0
    else:
        max_pages, page_size, n_pool, max_prefix = 0, 0, 0, k_out.shape[1]
    new_len = np.zeros((batch,), np.int32)
    rc = _load().orc_tree_commit_kv(batch, B, n_depth, hkv, D, _ptr(k_tree, _u16p),
                                    _ptr(v_tree, _u16p), _ptr(k_out, _u16p), _ptr(v_out, _u16p),
                                    _ptr(block_table, _i32p), page_size, max_pages, n_pool,
                                    max_prefix, _ptr(prefix_len, _i32p), _ptr(acc_len, _i32p),
                                    _ptr(acc_nodes, _i32p), _ptr(new_len, _i32p))
    if check:
        _check(rc, "orc_tree_commit_kv")
    return k_out, v_out, new_len, rc


def lmhead_logits(hidden, w_lm):
    """Draft logits through the LM head: hidden bf16 [rows][d] times w_lm bf16
    [vocab][d] transposed, every product and sum in float64 from the exactly
    widened bf16 values (a library matmul is the step), returned in float64."""
    h = _widen_bf16(hidden)
    w = _widen_bf16(w_lm)
    return h @ w.T


def lmhead_topw(hidden, w_lm, W):
    """Top-W tokens and log-probs of softmax(hidden @ w_lm^T) per row, with the
    logits rounded once to binary32 before the top-W step (orc_topw).
    Returns (tok [rows][W], logp [rows][W], logits float64 [rows][vocab])."""
    logits = lmhead_logits(hidden, w_lm)
    tok, logp = topw(logits.astype(np.float32)[None], W)
    return tok[0], logp[0], logits


def _widen_bf16(a):
    bits = _bf16_bits(a)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
