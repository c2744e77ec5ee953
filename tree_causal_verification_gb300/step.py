"""The hot path of one decode step, run through libjtree's five calls.

top-W per depth -> best-first expansion -> tree mask -> tree attention ->
greedy acceptance, every intermediate kept on the device in buffers that
are allocated once (``StepBuffers``) so that a step launches kernels only.
"""
from __future__ import annotations

import torch

from . import jtree
from .synth import Workload


class StepBuffers:
    """Device outputs of every step of the path for one workload shape."""

    def __init__(self, w: Workload, device="cuda"):
        dev = torch.device(device)
        i32, f32 = torch.int32, torch.float32
        b, N, W, B = w.batch, w.N, w.W, w.B
        self.w = w
        self.tok = torch.empty((b, N, W), dtype=i32, device=dev)
        self.logp = torch.empty((b, N, W), dtype=f32, device=dev)
        self.tree = dict(parent=torch.empty((b, B), dtype=i32, device=dev),
                         token=torch.empty((b, B), dtype=i32, device=dev),
                         depth=torch.empty((b, B), dtype=i32, device=dev),
                         score=torch.empty((b, B), dtype=f32, device=dev),
                         n_nodes=torch.empty((b,), dtype=i32, device=dev))
        self.mask = torch.empty((b, B, (B + 31) // 32), dtype=i32, device=dev)
        self.attn_out = torch.empty((b, B, w.hq, w.D), dtype=torch.bfloat16, device=dev)
        self.acc = dict(acc_len=torch.empty((b,), dtype=i32, device=dev),
                        acc_tokens=torch.empty((b, N), dtype=i32, device=dev),
                        acc_nodes=torch.empty((b, N), dtype=i32, device=dev),
                        bonus=torch.empty((b,), dtype=i32, device=dev))


def run_step(w: Workload, inp: dict, buf: StepBuffers, ex: jtree.Exec):
    """Enqueues the five calls on the current stream. ``inp`` holds device
    tensors: draft [b][N][V], q, k_tree, v_tree, k_cache, v_cache,
    block_table (or None), prefix_len, target [b][B+1][V]."""
    jtree.jt_topw(inp["draft"], w.W, buf.tok, buf.logp, exec=ex)
    jtree.jt_tree_expand(buf.tok, buf.logp, w.B, out=buf.tree, exec=ex)
    jtree.jt_tree_mask(buf.tree["parent"], buf.tree["n_nodes"], buf.mask, exec=ex)
    jtree.jt_tree_attn(inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                       inp["prefix_len"], buf.tree["n_nodes"], buf.mask, out=buf.attn_out,
                       block_table=inp["block_table"], exec=ex)
    jtree.jt_tree_accept(inp["target"], buf.tree["parent"], buf.tree["token"],
                         buf.tree["n_nodes"], w.N, out=buf.acc, exec=ex)
    return buf
