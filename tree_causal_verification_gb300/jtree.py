"""Python binding for libjtree's C ABI (include/jtree.h).

Argument marshalling only: every function here checks tensor shapes/dtypes,
passes ``data_ptr()`` values and the current CUDA stream to the C call of the
same name, and raises ``JtError`` on a non-OK status. All computation runs in
the CUDA kernels of libjtree.so. There is no fallback: if the library is not
built, or no CUDA device is present, the calls raise.

Output tensors and the workspace are allocated here with torch (the caller
side of the ABI); the library itself never allocates.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libjtree.so")

JT_OK = 0
JT_DEVERR_PARENT = 0x01
JT_DEVERR_TOKEN = 0x02
JT_DEVERR_NNODES = 0x04
JT_DEVERR_PAGE = 0x08
JT_DEVERR_PREFIX = 0x10
JT_DEVERR_TIMEOUT = 0x20
JT_DEVERR_PATH = 0x40
STATUS_NAMES = {0: "JT_OK", 1: "JT_ERR_INVALID_ARG", 2: "JT_ERR_UNSUPPORTED", 3: "JT_ERR_CUDA",
                4: "JT_ERR_DEVICE_DATA", 5: "JT_ERR_TIMEOUT", 6: "JT_ERR_WORKSPACE"}

EXPORTED = ["jt_status_str", "jt_read_device_error", "jt_topw_workspace_bytes", "jt_topw",
            "jt_tree_expand", "jt_tree_mask", "jt_tree_attn_workspace_bytes", "jt_tree_attn",
            "jt_tree_accept_workspace_bytes", "jt_tree_accept", "jt_tree_accept_noalloc",
            "jt_tree_commit_kv", "jt_topw_entropy", "jt_tree_expand_scored",
            "jt_tree_accept_sampled", "jt_lmhead_topw_workspace_bytes", "jt_lmhead_topw",
            "jt_set_wait_budget"]
JT_SCORE_LOGP, JT_SCORE_HYBRID, JT_SCORE_ENTROPY = 0, 1, 2


class JtError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib_status_str(status) if _lib is not None else STATUS_NAMES.get(status, "?")
        super().__init__(f"{where}: {msg}")


class jt_exec(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("d_err", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class jt_attn_args(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("B", ctypes.c_int), ("hq", ctypes.c_int),
                ("hkv", ctypes.c_int), ("head_dim", ctypes.c_int), ("scale", ctypes.c_float),
                ("q", ctypes.c_void_p), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int),
                ("max_pages", ctypes.c_int), ("n_pages", ctypes.c_int),
                ("max_prefix", ctypes.c_int), ("prefix_len", ctypes.c_void_p),
                ("n_nodes", ctypes.c_void_p), ("mask", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class jt_commit_args(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("B", ctypes.c_int), ("n_depth", ctypes.c_int),
                ("hkv", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int),
                ("max_pages", ctypes.c_int), ("n_pages", ctypes.c_int),
                ("max_prefix", ctypes.c_int), ("prefix_len", ctypes.c_void_p),
                ("acc_len", ctypes.c_void_p), ("acc_nodes", ctypes.c_void_p),
                ("new_prefix_len", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()
_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_pexec = ctypes.POINTER(jt_exec)


def load(path: str = LIB_PATH):
    """Loads libjtree.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libjtree.so is not built ({path}); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            lib.jt_status_str.restype = ctypes.c_char_p
            lib.jt_status_str.argtypes = [_c_int]
            lib.jt_read_device_error.argtypes = [_pexec, ctypes.POINTER(ctypes.c_int32)]
            lib.jt_topw_workspace_bytes.restype = _c_size
            lib.jt_topw_workspace_bytes.argtypes = [_c_int] * 4
            lib.jt_topw.argtypes = [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _pexec]
            lib.jt_tree_expand.argtypes = [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp,
                                           _vp, _vp, _vp, _pexec]
            lib.jt_tree_mask.argtypes = [_vp, _vp, _c_int, _c_int, _vp, _pexec]
            lib.jt_topw_entropy.argtypes = [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                            _pexec]
            lib.jt_tree_expand_scored.argtypes = [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                                  _c_int, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
                                                  _pexec]
            lib.jt_tree_attn_workspace_bytes.restype = _c_size
            lib.jt_tree_attn_workspace_bytes.argtypes = [ctypes.POINTER(jt_attn_args)]
            lib.jt_tree_attn.argtypes = [ctypes.POINTER(jt_attn_args), _pexec]
            lib.jt_tree_accept_workspace_bytes.restype = _c_size
            lib.jt_tree_accept_workspace_bytes.argtypes = [_c_int] * 4
            lib.jt_tree_accept.argtypes = [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                           _vp, _vp, _vp, _vp, _pexec]
            lib.jt_tree_accept_noalloc.argtypes = lib.jt_tree_accept.argtypes
            lib.jt_tree_accept_sampled.argtypes = [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                                   _c_int, ctypes.c_float, ctypes.c_uint64, _vp,
                                                   _vp, _vp, _vp, _pexec]
            lib.jt_tree_commit_kv.argtypes = [ctypes.POINTER(jt_commit_args), _pexec]
            lib.jt_lmhead_topw_workspace_bytes.restype = _c_size
            lib.jt_lmhead_topw_workspace_bytes.argtypes = [_c_int] * 4
            lib.jt_lmhead_topw.argtypes = [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp,
                                           _pexec]
            lib.jt_set_wait_budget.argtypes = [ctypes.c_longlong]
            for name in ("jt_read_device_error", "jt_topw", "jt_tree_expand", "jt_tree_mask",
                         "jt_tree_attn", "jt_tree_accept", "jt_tree_accept_noalloc",
                         "jt_tree_commit_kv", "jt_topw_entropy", "jt_tree_expand_scored",
                         "jt_tree_accept_sampled", "jt_lmhead_topw", "jt_set_wait_budget"):
                getattr(lib, name).restype = _c_int
            _lib = lib
    return _lib


def _lib_status_str(status: int) -> str:
    return _lib.jt_status_str(status).decode()


def _check(status: int, where: str):
    if status != JT_OK:
        raise JtError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


class Exec:
    """Stream, device error word and workspace for a sequence of calls.

    The workspace grows on demand (a torch allocation on the caller side) and
    is reused; calls on one Exec must not overlap on the GPU.
    """

    def __init__(self, device=None, stream=None, error_word=True):
        self.device = torch.device(device if device is not None else "cuda")
        self.stream = stream
        self.d_err = torch.zeros(1, dtype=torch.int32, device=self.device) if error_word else None
        self.workspace = None

    def reserve(self, nbytes: int):
        if nbytes and (self.workspace is None or self.workspace.numel() < nbytes):
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self

    def c(self) -> jt_exec:
        s = self.stream if self.stream is not None else torch.cuda.current_stream(self.device)
        ws = self.workspace
        return jt_exec(ctypes.c_void_p(s.cuda_stream), _ptr(self.d_err), _ptr(ws),
                       0 if ws is None else ws.numel())

    def read_error(self) -> int:
        """Synchronises the stream; returns and clears the device error word."""
        if self.d_err is None:
            return 0
        out = ctypes.c_int32(0)
        ex = self.c()
        st = load().jt_read_device_error(ctypes.byref(ex), ctypes.byref(out))
        if st not in (0, 4, 5):
            _check(st, "jt_read_device_error")
        return out.value


def jt_set_wait_budget(cycles: int = 0):
    """Test hook: cycle budget of the kernels' bounded waits for later
    launches (0 restores the default of about 2 s)."""
    _check(load().jt_set_wait_budget(int(cycles)), "jt_set_wait_budget")


_default_execs = {}


def _exec(ex):
    if ex is not None:
        return ex
    dev = torch.cuda.current_device()
    if dev not in _default_execs:
        _default_execs[dev] = Exec(device=f"cuda:{dev}")
    return _default_execs[dev]


def jt_topw(logits, W, tok=None, logp=None, exec=None, entropy=None, with_entropy=False):
    """Top-W tokens and log-probs per row: logits fp32 [batch][N][V].

    with_entropy (or an entropy buffer) also returns the per-row entropy
    fp32 [batch][N] (jt_topw_entropy)."""
    batch, N, V = logits.shape
    dev = logits.device
    tok = torch.empty((batch, N, W), dtype=torch.int32, device=dev) if tok is None else tok
    logp = torch.empty((batch, N, W), dtype=torch.float32, device=dev) if logp is None else logp
    _need(logits, torch.float32, (batch, N, V), "logits")
    _need(tok, torch.int32, (batch, N, W), "tok")
    _need(logp, torch.float32, (batch, N, W), "logp")
    lib = load()
    ex = _exec(exec).reserve(lib.jt_topw_workspace_bytes(batch, N, V, W))
    c = ex.c()
    if entropy is None and not with_entropy:
        _check(lib.jt_topw(_ptr(logits), batch, N, V, W, _ptr(tok), _ptr(logp), ctypes.byref(c)),
               "jt_topw")
        return tok, logp
    if entropy is None:
        entropy = torch.empty((batch, N), dtype=torch.float32, device=dev)
    _need(entropy, torch.float32, (batch, N), "entropy")
    _check(lib.jt_topw_entropy(_ptr(logits), batch, N, V, W, _ptr(tok), _ptr(logp),
                               _ptr(entropy), ctypes.byref(c)), "jt_topw_entropy")
    return tok, logp, entropy


def jt_tree_expand(tok, logp, B, out=None, exec=None, entropy=None, mode=JT_SCORE_LOGP,
                   alpha=0.0):
    """Best-first expansion; returns dict(parent, token, depth, score, n_nodes).

    mode / entropy / alpha select the branch score (jt_tree_expand_scored):
    0 cumulative log-prob, 1 hybrid logp - alpha*H_d, 2 entropy only -H_d."""
    batch, N, W = tok.shape
    dev = tok.device
    if out is None:
        out = dict(parent=torch.empty((batch, B), dtype=torch.int32, device=dev),
                   token=torch.empty((batch, B), dtype=torch.int32, device=dev),
                   depth=torch.empty((batch, B), dtype=torch.int32, device=dev),
                   score=torch.empty((batch, B), dtype=torch.float32, device=dev),
                   n_nodes=torch.empty((batch,), dtype=torch.int32, device=dev))
    _need(tok, torch.int32, (batch, N, W), "tok")
    _need(logp, torch.float32, (batch, N, W), "logp")
    for k in ("parent", "token", "depth"):
        _need(out[k], torch.int32, (batch, B), k)
    _need(out["score"], torch.float32, (batch, B), "score")
    _need(out["n_nodes"], torch.int32, (batch,), "n_nodes")
    c = _exec(exec).c()
    outs = (_ptr(out["parent"]), _ptr(out["token"]), _ptr(out["depth"]), _ptr(out["score"]),
            _ptr(out["n_nodes"]))
    if mode == JT_SCORE_LOGP and entropy is None:
        _check(load().jt_tree_expand(_ptr(tok), _ptr(logp), batch, N, W, B, *outs,
                                     ctypes.byref(c)), "jt_tree_expand")
        return out
    if entropy is not None:
        _need(entropy, torch.float32, (batch, N), "entropy")
    _check(load().jt_tree_expand_scored(_ptr(tok), _ptr(logp), _ptr(entropy), batch, N, W, B,
                                        int(mode), float(alpha), *outs, ctypes.byref(c)),
           "jt_tree_expand_scored")
    return out


def jt_tree_mask(parent, n_nodes, mask=None, exec=None):
    """Ancestor bitmasks: uint32 words as int32 [batch][B][ceil(B/32)]."""
    batch, B = parent.shape
    words = (B + 31) // 32
    mask = torch.empty((batch, B, words), dtype=torch.int32, device=parent.device) \
        if mask is None else mask
    _need(parent, torch.int32, (batch, B), "parent")
    _need(n_nodes, torch.int32, (batch,), "n_nodes")
    _need(mask, torch.int32, (batch, B, words), "mask")
    c = _exec(exec).c()
    _check(load().jt_tree_mask(_ptr(parent), _ptr(n_nodes), batch, B, _ptr(mask), ctypes.byref(c)),
           "jt_tree_mask")
    return mask


def attn_args(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, mask, out,
              block_table=None, scale=0.0, max_prefix=None) -> jt_attn_args:
    batch, B, hq, D = q.shape
    hkv = k_tree.shape[2]
    _need(q, torch.bfloat16, (batch, B, hq, D), "q")
    _need(k_tree, torch.bfloat16, (batch, B, hkv, D), "k_tree")
    _need(v_tree, torch.bfloat16, (batch, B, hkv, D), "v_tree")
    _need(prefix_len, torch.int32, (batch,), "prefix_len")
    _need(n_nodes, torch.int32, (batch,), "n_nodes")
    _need(mask, torch.int32, (batch, B, (B + 31) // 32), "mask")
    _need(out, torch.bfloat16, (batch, B, hq, D), "out")
    if block_table is not None:
        n_pages, page_size = k_cache.shape[0], k_cache.shape[1]
        _need(k_cache, torch.bfloat16, (n_pages, page_size, hkv, D), "k_cache")
        _need(v_cache, torch.bfloat16, (n_pages, page_size, hkv, D), "v_cache")
        _need(block_table, torch.int32, (batch, block_table.shape[1]), "block_table")
        max_pages = block_table.shape[1]
        mp = 0 if max_prefix is None else max_prefix
    else:
        Lmax = k_cache.shape[1]
        _need(k_cache, torch.bfloat16, (batch, Lmax, hkv, D), "k_cache")
        _need(v_cache, torch.bfloat16, (batch, Lmax, hkv, D), "v_cache")
        n_pages, page_size, max_pages = 0, 0, 0
        mp = Lmax
    return jt_attn_args(batch, B, hq, hkv, D, float(scale), _ptr(q), _ptr(k_tree), _ptr(v_tree),
                        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), page_size, max_pages,
                        n_pages, mp, _ptr(prefix_len), _ptr(n_nodes), _ptr(mask), _ptr(out))


def jt_tree_attn_workspace_bytes(args: jt_attn_args) -> int:
    return load().jt_tree_attn_workspace_bytes(ctypes.byref(args))


def jt_tree_attn(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, mask, out=None,
                 block_table=None, scale=0.0, exec=None):
    """Tree-causal GQA attention -> bf16 [batch][B][hq][D]."""
    out = torch.empty_like(q) if out is None else out
    args = attn_args(q, k_tree, v_tree, k_cache, v_cache, prefix_len, n_nodes, mask, out,
                     block_table, scale)
    lib = load()
    ex = _exec(exec).reserve(lib.jt_tree_attn_workspace_bytes(ctypes.byref(args)))
    c = ex.c()
    _check(lib.jt_tree_attn(ctypes.byref(args), ctypes.byref(c)), "jt_tree_attn")
    return out


def jt_tree_accept(target, parent, token, n_nodes, n_depth, out=None, exec=None,
                   temperature=0.0, seed=0):
    """Acceptance; returns dict(acc_len, acc_tokens, acc_nodes, bonus).

    temperature 0: greedy (jt_tree_accept); > 0: one target draw per visited
    node from the counter-based stream `seed` (jt_tree_accept_sampled)."""
    batch, B = parent.shape
    V = target.shape[-1]
    dev = target.device
    if out is None:
        out = dict(acc_len=torch.empty((batch,), dtype=torch.int32, device=dev),
                   acc_tokens=torch.empty((batch, n_depth), dtype=torch.int32, device=dev),
                   acc_nodes=torch.empty((batch, n_depth), dtype=torch.int32, device=dev),
                   bonus=torch.empty((batch,), dtype=torch.int32, device=dev))
    _need(target, torch.float32, (batch, B + 1, V), "target")
    _need(parent, torch.int32, (batch, B), "parent")
    _need(token, torch.int32, (batch, B), "token")
    _need(n_nodes, torch.int32, (batch,), "n_nodes")
    lib = load()
    ex = _exec(exec).reserve(lib.jt_tree_accept_workspace_bytes(batch, B, n_depth, V))
    c = ex.c()
    outs = (_ptr(out["acc_len"]), _ptr(out["acc_tokens"]), _ptr(out["acc_nodes"]),
            _ptr(out["bonus"]))
    if temperature == 0.0:
        _check(lib.jt_tree_accept(_ptr(target), _ptr(parent), _ptr(token), _ptr(n_nodes), batch,
                                  B, n_depth, V, *outs, ctypes.byref(c)), "jt_tree_accept")
    else:
        _check(lib.jt_tree_accept_sampled(_ptr(target), _ptr(parent), _ptr(token), _ptr(n_nodes),
                                          batch, B, n_depth, V, ctypes.c_float(temperature),
                                          ctypes.c_uint64(int(seed) & (2 ** 64 - 1)), *outs,
                                          ctypes.byref(c)), "jt_tree_accept_sampled")
    return out


def jt_tree_accept_noalloc(target, parent, token, n_nodes, n_depth, out=None, exec=None):
    """jt_tree_accept without a workspace: for callers that cannot allocate
    device scratch. The library uses its own fixed device array instead, so
    calls on one device must not overlap on the GPU (they share that array).
    Limit: batch * (B + 1) <= 65536."""
    batch, B = parent.shape
    V = target.shape[-1]
    dev = target.device
    if out is None:
        out = dict(acc_len=torch.empty((batch,), dtype=torch.int32, device=dev),
                   acc_tokens=torch.empty((batch, n_depth), dtype=torch.int32, device=dev),
                   acc_nodes=torch.empty((batch, n_depth), dtype=torch.int32, device=dev),
                   bonus=torch.empty((batch,), dtype=torch.int32, device=dev))
    _need(target, torch.float32, (batch, B + 1, V), "target")
    _need(parent, torch.int32, (batch, B), "parent")
    _need(token, torch.int32, (batch, B), "token")
    _need(n_nodes, torch.int32, (batch,), "n_nodes")
    c = _exec(exec).c()
    _check(load().jt_tree_accept_noalloc(_ptr(target), _ptr(parent), _ptr(token), _ptr(n_nodes),
                                         batch, B, n_depth, V, _ptr(out["acc_len"]),
                                         _ptr(out["acc_tokens"]), _ptr(out["acc_nodes"]),
                                         _ptr(out["bonus"]), ctypes.byref(c)),
           "jt_tree_accept_noalloc")
    return out


def commit_args(k_tree, v_tree, k_cache, v_cache, prefix_len, acc_len, acc_nodes, new_prefix_len,
                block_table=None) -> jt_commit_args:
    batch, B, hkv, D = k_tree.shape
    n_depth = acc_nodes.shape[1]
    _need(k_tree, torch.bfloat16, (batch, B, hkv, D), "k_tree")
    _need(v_tree, torch.bfloat16, (batch, B, hkv, D), "v_tree")
    _need(prefix_len, torch.int32, (batch,), "prefix_len")
    _need(acc_len, torch.int32, (batch,), "acc_len")
    _need(acc_nodes, torch.int32, (batch, n_depth), "acc_nodes")
    _need(new_prefix_len, torch.int32, (batch,), "new_prefix_len")
    if block_table is not None:
        n_pages, page_size = k_cache.shape[0], k_cache.shape[1]
        _need(k_cache, torch.bfloat16, (n_pages, page_size, hkv, D), "k_cache")
        _need(v_cache, torch.bfloat16, (n_pages, page_size, hkv, D), "v_cache")
        _need(block_table, torch.int32, (batch, block_table.shape[1]), "block_table")
        max_pages, mp = block_table.shape[1], 0
    else:
        Lmax = k_cache.shape[1]
        _need(k_cache, torch.bfloat16, (batch, Lmax, hkv, D), "k_cache")
        _need(v_cache, torch.bfloat16, (batch, Lmax, hkv, D), "v_cache")
        n_pages, page_size, max_pages, mp = 0, 0, 0, Lmax
    return jt_commit_args(batch, B, n_depth, hkv, D, _ptr(k_tree), _ptr(v_tree), _ptr(k_cache),
                          _ptr(v_cache), _ptr(block_table), page_size, max_pages, n_pages, mp,
                          _ptr(prefix_len), _ptr(acc_len), _ptr(acc_nodes), _ptr(new_prefix_len))


def jt_tree_commit_kv(k_tree, v_tree, k_cache, v_cache, prefix_len, acc_len, acc_nodes,
                      new_prefix_len=None, block_table=None, exec=None):
    """Writes the accepted path's tree K/V rows into k_cache / v_cache (in place)
    after each sequence's prefix; returns new_prefix_len (int32 [batch])."""
    if new_prefix_len is None:
        new_prefix_len = torch.empty_like(prefix_len)
    args = commit_args(k_tree, v_tree, k_cache, v_cache, prefix_len, acc_len, acc_nodes,
                       new_prefix_len, block_table)
    c = _exec(exec).c()
    _check(load().jt_tree_commit_kv(ctypes.byref(args), ctypes.byref(c)), "jt_tree_commit_kv")
    return new_prefix_len


def jt_lmhead_topw(hidden, w_lm, W, tok=None, logp=None, entropy=None, with_entropy=False,
                   exec=None):
    """Top-W of softmax(hidden @ w_lm^T) per row without materialising the
    logits: hidden bf16 [rows][d], w_lm bf16 [vocab][d] -> (tok, logp[, entropy])."""
    rows, d = hidden.shape
    V = w_lm.shape[0]
    dev = hidden.device
    _need(hidden, torch.bfloat16, (rows, d), "hidden")
    _need(w_lm, torch.bfloat16, (V, d), "w_lm")
    tok = torch.empty((rows, W), dtype=torch.int32, device=dev) if tok is None else tok
    logp = torch.empty((rows, W), dtype=torch.float32, device=dev) if logp is None else logp
    _need(tok, torch.int32, (rows, W), "tok")
    _need(logp, torch.float32, (rows, W), "logp")
    if with_entropy and entropy is None:
        entropy = torch.empty((rows,), dtype=torch.float32, device=dev)
    if entropy is not None:
        _need(entropy, torch.float32, (rows,), "entropy")
    lib = load()
    ex = _exec(exec).reserve(lib.jt_lmhead_topw_workspace_bytes(rows, d, V, W))
    c = ex.c()
    _check(lib.jt_lmhead_topw(_ptr(hidden), _ptr(w_lm), rows, d, V, W, _ptr(tok), _ptr(logp),
                              _ptr(entropy), ctypes.byref(c)), "jt_lmhead_topw")
    return (tok, logp) if entropy is None else (tok, logp, entropy)
