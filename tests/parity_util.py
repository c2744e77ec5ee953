"""Shared helpers for the GPU parity tests: a workload's inputs (drawn once,
the same bytes for both sides) and the oracle's results on them."""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
from tree_causal_verification_gb300 import jtree, synth

ATTN_MAX_ABS = 2e-2     # bf16 output vs fp64 oracle, per element
ATTN_MEAN_ABS = 2e-3    # mean over the compared elements
LOGP_ABS = 1e-5


def to_np(t):
    return t.detach().cpu().numpy()


def u32(t):
    return to_np(t).view(np.uint32)


class Case:
    """One workload: device inputs, host copies and the oracle tree."""

    def __init__(self, w: synth.Workload, seed=0, device="cuda", topw_rows=None):
        self.w = w
        dev = torch.device(device)
        gen = dev if w.V * w.batch * (w.N + 1) > 4_000_000 else torch.device("cpu")
        self.draft_ext = synth.draft_logits(w, seed, gen)
        self.draft = self.draft_ext[:, : w.N].contiguous()
        self.kv = synth.kv_inputs(w, seed, gen)
        self.draft_h = to_np(self.draft)
        # Oracle top-W over every row (the oracle tree needs all of them).
        self.tok, self.logp = oracle.topw(self.draft_h, w.W)
        self.tree = oracle.tree_expand(self.tok, self.logp, w.B)
        self.mask = oracle.tree_mask(self.tree["parent"], self.tree["n_nodes"])
        self.target = synth.target_logits(w, self.draft_ext.to(gen),
                                          torch.from_numpy(self.tree["depth"]),
                                          torch.from_numpy(self.tree["n_nodes"]), seed)
        self.dev = dev
        self.inp = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in self.kv.items()}
        self.inp["draft"] = self.draft.to(dev)
        self.inp["target"] = self.target.to(dev)

    def oracle_accept(self, tree=None):
        t = self.tree if tree is None else tree
        return oracle.tree_accept(to_np(self.target), t["parent"], t["token"], t["n_nodes"],
                                  self.w.N)

    def sample_rows(self, n_nodes, per_seq=24, seed=0):
        rng = np.random.default_rng(seed)
        rows = []
        g = self.w.hq
        for b in range(self.w.batch):
            n = int(n_nodes[b])
            vs = {0, max(n - 1, 0), min(n, self.w.B - 1)}
            vs |= set(rng.integers(0, self.w.B, 4).tolist())
            for v in sorted(vs):
                hs = {0, g - 1} | set(rng.integers(0, g, 2).tolist())
                for h in sorted(hs):
                    rows.append((b, v, h))
        rows = np.array(rows, np.int32)
        if len(rows) > per_seq * max(self.w.batch, 8):
            rows = rows[rng.choice(len(rows), per_seq * max(self.w.batch, 8), replace=False)]
        return rows

    def whole_sequences(self, seqs):
        """Every (sequence, node, head) row of the given sequences."""
        w = self.w
        return np.array([(b, v, h) for b in seqs for v in range(w.B) for h in range(w.hq)],
                        np.int32)

    def host_kv(self):
        """Host copies (bf16 bit patterns) of the attention inputs, made once."""
        if not hasattr(self, "_host_kv"):
            hk = {}
            for k in ("q", "k_tree", "v_tree", "k_cache", "v_cache"):
                hk[k] = self.kv[k].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            hk["prefix_len"] = to_np(self.kv["prefix_len"])
            hk["block_table"] = None if self.kv["block_table"] is None \
                else to_np(self.kv["block_table"])
            self._host_kv = hk
        return self._host_kv

    def oracle_attn(self, rows, mask=None, n_nodes=None):
        """The oracle on the given rows, split over the host's cores: every
        worker runs the unchanged single-threaded oracle on its own slice of
        the rows (the oracle keeps no shared state)."""
        kv = self.host_kv()
        nn = self.tree["n_nodes"] if n_nodes is None else n_nodes
        mk = self.mask if mask is None else mask
        rows = np.ascontiguousarray(rows, np.int32).reshape(-1, 3)

        def part(r):
            return oracle.tree_attn(kv["q"], kv["k_tree"], kv["v_tree"], kv["k_cache"],
                                    kv["v_cache"], kv["prefix_len"], nn, mk, hq=self.w.hq,
                                    hkv=self.w.hkv, block_table=kv["block_table"], rows=r)

        workers = max(1, min(len(os.sched_getaffinity(0)), 64))
        if len(rows) < 64 or workers == 1:
            return part(rows)
        chunks = np.array_split(rows, min(workers * 4, len(rows)))
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            return np.concatenate(list(ex.map(part, chunks)))


def check_attn(got_bf16, ref, what=""):
    got = got_bf16.astype(np.float64)
    err = np.abs(got - ref)
    assert err.max() <= ATTN_MAX_ABS, f"{what} attention max-abs {err.max():.3e}"
    assert err.mean() <= ATTN_MEAN_ABS, f"{what} attention mean-abs {err.mean():.3e}"
    return err.max(), err.mean()


def gather_rows(out, rows):
    o = out.float().cpu().numpy()
    return o[rows[:, 0], rows[:, 1], rows[:, 2]]


def new_exec(dev):
    return jtree.Exec(dev)
