"""Seeded synthetic inputs for one tree-drafting decode step.

This module only draws random tensors with the shapes, sizes and value
distributions of the workloads below; it contains none of the method's
arithmetic. The same bytes feed the CUDA library and the CPU oracle.

Every tensor has its own ``torch.Generator`` seeded from (seed, tensor name),
so a tensor's values do not depend on which other tensors were drawn or in
which order. Values drawn on a CUDA generator differ from those drawn on the
CPU one; tests therefore always hand both sides the same materialised bytes.

Shapes stand in for a Qwen3-8B verification step (32 query / 8 KV heads,
head_dim 128, vocabulary 151936; JetSpec summary on paperlayer.ai, App. D
"Model implementation", and the Korean review on startedourmission.github.io,
"How it works") and for the MoE target's attention shape (32 / 4 heads).
No dataset, tokenizer or trained weight is used.
"""
from __future__ import annotations

import dataclasses
import zlib

import torch

PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    prefix_lo: int          # prefix lengths ~ U[prefix_lo, prefix_hi] (inclusive)
    prefix_hi: int
    B: int                  # tree budget (draft nodes, root excluded)
    N: int                  # maximum depth
    W: int                  # width (children per expansion)
    hq: int
    hkv: int
    D: int
    V: int
    paged: bool
    draft_sigma: float = 3.0      # draft logits ~ N(0, draft_sigma^2)
    target_sigma: float = 1.0     # target row = draft row + N(0, target_sigma^2)
    temp_slope: float = 0.0       # draft logits divided by 1 + temp_slope * depth

    @property
    def max_prefix(self) -> int:
        return self.prefix_hi

    @property
    def max_pages(self) -> int:
        return (self.prefix_hi + PAGE_SIZE - 1) // PAGE_SIZE

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["workload"] = d.pop("name")
        return d


# The five step shapes this library is built and measured on.
WORKLOADS = {
    w.name: w for w in [
        Workload("tiny", 1, 128, 128, B=16, N=4, W=2, hq=4, hkv=1, D=64, V=1024, paged=False,
                 target_sigma=1.0),
        Workload("qwen3-8b-chain", 1, 2048, 2048, B=16, N=16, W=1, hq=32, hkv=8, D=128,
                 V=151936, paged=False, target_sigma=0.5),
        Workload("high-budget", 1, 4096, 4096, B=256, N=16, W=4, hq=32, hkv=8, D=128,
                 V=151936, paged=False, target_sigma=1.0, temp_slope=0.1),
        Workload("mid-batch-paged", 16, 1024, 8192, B=64, N=8, W=4, hq=32, hkv=8, D=128,
                 V=151936, paged=True, target_sigma=1.0),
        Workload("moe-paged", 64, 2048, 16384, B=128, N=16, W=4, hq=32, hkv=4, D=128,
                 V=151936, paged=True, target_sigma=1.5),
    ]
}
WORKLOAD_ORDER = ["tiny", "qwen3-8b-chain", "high-budget", "mid-batch-paged", "moe-paged"]


def _gen(seed: int, name: str, device) -> torch.Generator:
    s = (seed * 0x9E3779B97F4A7C15 + zlib.crc32(name.encode())) & 0x7FFFFFFFFFFFFFFF
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def randn(shape, seed, name, device="cpu", sigma=1.0):
    g = _gen(seed, name, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x


def randn_bf16(shape, seed, name, device="cpu"):
    return randn(shape, seed, name, device).to(torch.bfloat16)


def prefix_lengths(w: Workload, seed: int = 0) -> torch.Tensor:
    if w.prefix_lo == w.prefix_hi:
        return torch.full((w.batch,), w.prefix_lo, dtype=torch.int32)
    g = _gen(seed, "prefix_len", "cpu")
    return torch.randint(w.prefix_lo, w.prefix_hi + 1, (w.batch,), generator=g,
                         dtype=torch.int64).to(torch.int32)


def draft_logits(w: Workload, seed: int = 0, device="cpu") -> torch.Tensor:
    """Draft logits for depths 1..N+1, fp32 [batch][N+1][V].

    Depths 1..N feed the proposer; the extra depth N+1 row stands in for the
    target's prediction below a depth-N node. With temp_slope > 0 the row for
    depth d is divided by 1 + temp_slope * d.
    """
    x = randn((w.batch, w.N + 1, w.V), seed, "draft", device, sigma=w.draft_sigma)
    if w.temp_slope:
        d = torch.arange(1, w.N + 2, device=device, dtype=torch.float32)
        x.div_((1.0 + w.temp_slope * d).view(1, -1, 1))
    return x


def kv_inputs(w: Workload, seed: int = 0, device="cpu", prefix_len=None) -> dict:
    """Query, tree K/V and prefix KV cache (bf16 ~ N(0,1)), plus the paging.

    Contiguous prefix: k/v_cache [batch][max_prefix][hkv][D].
    Paged prefix: a pool of exactly sum(ceil(L_b/16)) pages [pages][16][hkv][D];
    sequence b's pages are a seeded random permutation of the pool, so its
    block table is not contiguous. Unused block-table entries are -1.
    """
    if prefix_len is None:
        prefix_len = prefix_lengths(w, seed)
    out = {
        "prefix_len": prefix_len.to(device),
        "q": randn_bf16((w.batch, w.B, w.hq, w.D), seed, "q", device),
        "k_tree": randn_bf16((w.batch, w.B, w.hkv, w.D), seed, "k_tree", device),
        "v_tree": randn_bf16((w.batch, w.B, w.hkv, w.D), seed, "v_tree", device),
    }
    if w.paged:
        pages_per = [(int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in prefix_len.tolist()]
        total = sum(pages_per)
        g = _gen(seed, "page_perm", "cpu")
        perm = torch.randperm(total, generator=g).to(torch.int32)
        bt = torch.full((w.batch, w.max_pages), -1, dtype=torch.int32)
        off = 0
        for b, p in enumerate(pages_per):
            bt[b, :p] = perm[off:off + p]
            off += p
        out["block_table"] = bt.to(device)
        out["k_cache"] = randn_bf16((total, PAGE_SIZE, w.hkv, w.D), seed, "k_cache", device)
        out["v_cache"] = randn_bf16((total, PAGE_SIZE, w.hkv, w.D), seed, "v_cache", device)
    else:
        out["block_table"] = None
        out["k_cache"] = randn_bf16((w.batch, w.max_prefix, w.hkv, w.D), seed, "k_cache", device)
        out["v_cache"] = randn_bf16((w.batch, w.max_prefix, w.hkv, w.D), seed, "v_cache", device)
    return out


def target_logits(w: Workload, draft_ext: torch.Tensor, depth: torch.Tensor,
                  n_nodes: torch.Tensor, seed: int = 0) -> torch.Tensor:
    """Target logits fp32 [batch][B+1][V] for a given tree.

    Row 0 (the root, depth 0) and row 1+v (node v at depth d_v) are the draft
    row of depth d+1 plus fresh N(0, target_sigma^2) noise, so the target
    agrees with the draft often but not always. Rows of unused budget slots
    (v >= n_nodes) are noise only. ``depth`` / ``n_nodes`` describe the tree
    the rows are drawn for; they select rows and do not enter any arithmetic.
    """
    device = draft_ext.device
    x = randn((w.batch, w.B + 1, w.V), seed, "target_noise", device, sigma=w.target_sigma)
    depth = depth.to(device=device, dtype=torch.int64)
    n_nodes = n_nodes.to(device=device, dtype=torch.int64)
    slot = torch.arange(w.B, device=device).view(1, -1)
    used = slot < n_nodes.view(-1, 1)
    d_row = torch.where(used, depth, torch.zeros_like(depth))       # depth of node v
    src = torch.cat([torch.zeros((w.batch, 1), dtype=torch.int64, device=device), d_row], 1)
    for b in range(w.batch):
        rows = draft_ext[b].index_select(0, src[b])                     # depth d -> draft row d+1
        keep = torch.cat([torch.ones(1, dtype=torch.bool, device=device), used[b]])
        x[b][keep] += rows[keep]
        del rows
    return x


__all__ = ["Workload", "WORKLOADS", "WORKLOAD_ORDER", "PAGE_SIZE", "randn", "randn_bf16",
           "prefix_lengths", "draft_logits", "kv_inputs", "target_logits"]
