#!/usr/bin/env python3
"""Benchmark: tree nodes verified per second for one decode step's hot path.

A step is the whole path through libjtree's C ABI on inputs resident in HBM:
top-W per depth -> best-first expansion -> tree mask -> tree attention ->
greedy acceptance. Default workload: batch 1, prefix 2048, a 16-node chain
(N=16, W=1), 32/8 heads, head_dim 128, vocabulary 151936 (Qwen3-8B shapes).

Timing: W eager warm-up steps, then EXACTLY K steps captured into one CUDA
graph and launched once, bracketed by a barrier and a device synchronise on
both sides, timed by CUDA events recorded on the launching stream at the two
ends. Each call's average duration comes from a further timed region per
call: one graph of K launches of that call alone on the same input sets
(events at its two ends); those feed the roofline figures. Steps rotate
through enough independent input sets that the inputs exceed the 129 MB L2.
SM clocks and throttle reasons are sampled through NVML during that region.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path shards by sequence with no exchange: weak scaling); value = nodes of all
ranks / the slowest rank's time.

--impl reference times the CPU oracle (the plain C++ reference, untuned) on
the host cores: each step is a one-node sample of the same workload.

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree nodes verified/sec per step (attn+top-W+accept); % of GB300 HBM/tensor roofline"
UNIT = "nodes/s"
DEFAULT_WORKLOAD = "qwen3-8b-chain"
L2_BYTES = 129e6
CALLS = ["jt_topw", "jt_tree_expand", "jt_tree_mask", "jt_tree_attn", "jt_tree_accept"]
# Kernels each call launches (the acceptance call runs an argmax pass and a walk).
KERNELS_PER_CALL = {"jt_topw": 1, "jt_tree_expand": 1, "jt_tree_mask": 1, "jt_tree_attn": 1,
                    "jt_tree_accept": 2}
# Sources whose change invalidates a committed DRAM-traffic figure.
CALL_SOURCES = {
    "jt_topw": ["jt_topw.cu", "jt_rowscan.cuh"],
    "jt_tree_expand": ["jt_expand.cu"],
    "jt_tree_mask": ["jt_mask.cu"],
    "jt_tree_attn": ["jt_attn.cu", "jt_sm100.cuh"],
    "jt_tree_accept": ["jt_accept.cu", "jt_rowscan.cuh"],
}


# --------------------------------------------------------------------------
# CUDA runtime (the one torch loaded) for graph capture and external events.
# --------------------------------------------------------------------------
def _cudart():
    path = None
    with open("/proc/self/maps") as f:
        for line in f:
            if "libcudart.so" in line:
                path = line.split()[-1]
                break
    lib = ctypes.CDLL(path or "libcudart.so")
    vp = ctypes.c_void_p
    lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
    lib.cudaEventRecordWithFlags.argtypes = [vp, vp, ctypes.c_uint]
    lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), vp, vp]
    lib.cudaEventDestroy.argtypes = [vp]
    lib.cudaStreamBeginCapture.argtypes = [vp, ctypes.c_int]
    lib.cudaStreamEndCapture.argtypes = [vp, ctypes.POINTER(vp)]
    lib.cudaGraphInstantiate.argtypes = [ctypes.POINTER(vp), vp, ctypes.c_ulonglong]
    lib.cudaGraphUpload.argtypes = [vp, vp]
    lib.cudaGraphLaunch.argtypes = [vp, vp]
    lib.cudaGraphGetNodes.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    lib.cudaGraphNodeGetType.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.cudaGraphDestroy.argtypes = [vp]
    lib.cudaGraphExecDestroy.argtypes = [vp]
    lib.cudaDeviceGetPCIBusId.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_int]
    return lib


def _ok(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with cudaError {rc}")


class Graph:
    """A stream capture of Python-side launches, instantiated once."""

    def __init__(self, rt, stream):
        self.rt, self.stream = rt, stream
        self.graph = ctypes.c_void_p()
        self.exec = ctypes.c_void_p()

    def __enter__(self):
        _ok(self.rt.cudaStreamBeginCapture(ctypes.c_void_p(self.stream.cuda_stream), 2),
            "cudaStreamBeginCapture")
        return self

    def __exit__(self, et, ev, tb):
        rc = self.rt.cudaStreamEndCapture(ctypes.c_void_p(self.stream.cuda_stream),
                                          ctypes.byref(self.graph))
        if et is None:
            _ok(rc, "cudaStreamEndCapture")
            _ok(self.rt.cudaGraphInstantiate(ctypes.byref(self.exec), self.graph, 0),
                "cudaGraphInstantiate")
        return False

    def kernel_nodes(self):
        n = ctypes.c_size_t(0)
        _ok(self.rt.cudaGraphGetNodes(self.graph, None, ctypes.byref(n)), "cudaGraphGetNodes")
        nodes = (ctypes.c_void_p * n.value)()
        _ok(self.rt.cudaGraphGetNodes(self.graph, nodes, ctypes.byref(n)), "cudaGraphGetNodes")
        count = 0
        for i in range(n.value):
            t = ctypes.c_int(-1)
            _ok(self.rt.cudaGraphNodeGetType(nodes[i], ctypes.byref(t)), "cudaGraphNodeGetType")
            count += (t.value == 0)  # cudaGraphNodeTypeKernel
        return count

    def upload(self):
        _ok(self.rt.cudaGraphUpload(self.exec, ctypes.c_void_p(self.stream.cuda_stream)),
            "cudaGraphUpload")

    def launch(self):
        _ok(self.rt.cudaGraphLaunch(self.exec, ctypes.c_void_p(self.stream.cuda_stream)),
            "cudaGraphLaunch")

    def close(self):
        if self.exec:
            self.rt.cudaGraphExecDestroy(self.exec)
        if self.graph:
            self.rt.cudaGraphDestroy(self.graph)


# --------------------------------------------------------------------------
# Clock sampling (NVML through ctypes; read-only).
# --------------------------------------------------------------------------
REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle",
           0x2: "applications_clocks_setting"}


class ClockSampler:
    def __init__(self, pci_bus_id: str):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.error = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) != 0:
                raise RuntimeError(f"no NVML handle for {pci_bus_id}")
            self.nv, self.h = nv, h
            mx = ctypes.c_uint(0)
            nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # reported in the JSON line, never fatal
            self.nv = None
            self.error = str(e)

    def _run(self):
        mhz = ctypes.c_uint(0)
        reasons = ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz))
            self._reasons_fn(self.h, ctypes.byref(reasons))
            self.samples.append((mhz.value, reasons.value))
            time.sleep(0.002)

    def __enter__(self):
        if self.nv is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._thread:
            self._thread.join()
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "error": self.error}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        names = sorted(n for b, n in REASONS.items() if bits & b)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples), "sm_mhz_min": min(mhz)}


# --------------------------------------------------------------------------
# Workload accounting (algorithmic bytes / flops per call).
# --------------------------------------------------------------------------
def algorithmic_work(w, prefix_len, n_nodes, depth_sum, path_rows):
    """Bytes (and attention flops) each call must move or do at minimum."""
    b = w.batch
    V4 = 4 * w.V
    kv_bytes = 2 * 2 * w.hkv * w.D * sum(prefix_len)                  # K and V, bf16
    tree_kv = 2 * 2 * w.hkv * w.D * sum(n_nodes)
    q_out = 2 * 2 * w.hq * w.D * sum(n_nodes)                          # q in, o out
    attn_flops = 4 * w.hq * w.D * sum(n * L for n, L in zip(n_nodes, prefix_len)) + \
        4 * w.hq * w.D * depth_sum
    return {
        "jt_topw": {"bytes": b * w.N * V4 + b * w.N * w.W * 8, "flops": None},
        "jt_tree_expand": {"bytes": b * w.N * w.W * 8 + b * w.B * 16, "flops": None},
        "jt_tree_mask": {"bytes": b * w.B * 4 + b * w.B * ((w.B + 31) // 32) * 4, "flops": None},
        "jt_tree_attn": {"bytes": kv_bytes + tree_kv + q_out, "flops": attn_flops},
        # Rows on the accepted paths (acc_len + 1 per sequence) must be read.
        "jt_tree_accept": {"bytes": path_rows * V4 + b * w.B * 8, "flops": None},
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_sha(call):
    h = hashlib.sha1()
    for f in CALL_SOURCES[call]:
        h.update(open(os.path.join(ROOT, "tree_causal_verification_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def committed_traffic(call, workload):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(call, {}).get(workload)
    if not d or d.get("sha1") != source_sha(call):
        return None
    return d.get("bytes_per_launch")


# --------------------------------------------------------------------------
# Inputs.
# --------------------------------------------------------------------------
def make_set(w, seed, dev):
    import torch
    from tree_causal_verification_gb300 import jtree, synth
    draft_ext = synth.draft_logits(w, seed, dev)
    draft = draft_ext[:, : w.N].contiguous()
    kv = synth.kv_inputs(w, seed, dev)
    # The target rows are drawn for the tree this step builds (an input, not an
    # expected value), so run the first two calls once to learn its depths.
    ex = jtree.Exec(dev)
    tok, logp = jtree.jt_topw(draft, w.W, exec=ex)
    tree = jtree.jt_tree_expand(tok, logp, w.B, exec=ex)
    target = synth.target_logits(w, draft_ext, tree["depth"], tree["n_nodes"], seed)
    del draft_ext
    inp = dict(kv)
    inp["draft"], inp["target"] = draft, target
    torch.cuda.synchronize(dev)
    meta = {"n_nodes": tree["n_nodes"].cpu().tolist(),
            "depth_sum": int(tree["depth"].sum().item()),
            "prefix_len": kv["prefix_len"].cpu().tolist()}
    return inp, meta


def set_bytes(inp):
    return sum(t.numel() * t.element_size() for t in inp.values() if t is not None)


# --------------------------------------------------------------------------
# CPU oracle legs.
# --------------------------------------------------------------------------
def oracle_host_inputs(inp):
    import numpy as np
    h = {}
    for k, t in inp.items():
        h[k] = None if t is None else t.cpu()
    h["draft_np"] = h["draft"].numpy()
    h["target_np"] = h["target"].numpy()
    h["prefix_np"] = h["prefix_len"].numpy()
    h["bt_np"] = None if h["block_table"] is None else h["block_table"].numpy()
    return h, np


def oracle_node_sample(w, h, v, full):
    """One node's share of a step, by the oracle: its depth's top-W row, the
    sequence's expansion and mask, the node's attention over every head, and
    the sequence's acceptance walk. ``full`` = (tok, logp) of sequence 0."""
    import oracle
    tree = oracle.tree_expand(full[0], full[1], w.B)
    d = max(int(tree["depth"][0, v]), 1)
    oracle.topw(h["draft_np"][0:1, d - 1:d], w.W)
    mask = oracle.tree_mask(tree["parent"], tree["n_nodes"])
    rows = [(0, v, hh) for hh in range(w.hq)]
    oracle.tree_attn(h["q"][0:1], h["k_tree"][0:1], h["v_tree"][0:1],
                     h["k_cache"] if w.paged else h["k_cache"][0:1],
                     h["v_cache"] if w.paged else h["v_cache"][0:1],
                     h["prefix_np"][0:1], tree["n_nodes"], mask, hq=w.hq, hkv=w.hkv,
                     block_table=None if h["bt_np"] is None else h["bt_np"][0:1], rows=rows)
    oracle.tree_accept(h["target_np"][0:1], tree["parent"], tree["token"], tree["n_nodes"], w.N)
    return tree


def oracle_leg(w, inp, steps=None, warmup=0, budget_s=12.0):
    """Times the oracle on one-node samples (rank 0, host cores, 1 thread)."""
    import oracle
    oracle.build()
    h, _ = oracle_host_inputs(inp)
    full = oracle.topw(h["draft_np"][0:1], w.W)
    tree = oracle.tree_expand(full[0], full[1], w.B)
    n0 = int(tree["n_nodes"][0])
    for i in range(warmup):
        oracle_node_sample(w, h, i % n0, full)
    t0 = time.perf_counter()
    done = 0
    while True:
        oracle_node_sample(w, h, done % n0, full)
        done += 1
        el = time.perf_counter() - t0
        if steps is not None and done >= steps:
            break
        if steps is None and el >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} one-node samples of sequence 0 ({w.name}): the node's depth row "
                      f"top-W (V={w.V}), the sequence's expansion, mask and acceptance walk, and "
                      f"the node's attention over all {w.hq} heads and "
                      f"{int(h['prefix_np'][0])}+tree keys; single thread, {el:.1f} s",
            "seconds": el, "samples": done}


# --------------------------------------------------------------------------
# Main.
# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="jtree", choices=["jtree", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    import torch
    from tree_causal_verification_gb300 import jtree, synth
    from tree_causal_verification_gb300.dist import job_throughput, max_over_ranks, rank_world

    rank, world, local = rank_world()
    from tree_causal_verification_gb300.step import StepBuffers, run_step

    w = synth.WORKLOADS[args.workload]
    wdesc = {"workload": w.name, "batch": w.batch, "prefix": [w.prefix_lo, w.prefix_hi],
             "B": w.B, "N": w.N, "W": w.W, "hq": w.hq, "hkv": w.hkv, "head_dim": w.D,
             "vocab": w.V, "paged": w.paged}

    if args.impl == "reference":
        if rank != 0:
            return
        # CPU oracle on the host cores; inputs drawn on the CPU generator.
        inp, meta = {}, None
        draft_ext = synth.draft_logits(w, 0, "cpu")
        kv = synth.kv_inputs(w, 0, "cpu")
        import oracle
        oracle.build()
        tok, logp = oracle.topw(draft_ext[:1, : w.N].contiguous().numpy(), w.W)
        t1 = oracle.tree_expand(tok, logp, w.B)
        # Only sequence 0 is sampled; draw its target rows for its tree.
        w1 = synth.Workload(**{**w.__dict__, "batch": 1})
        target = synth.target_logits(w1, draft_ext[:1], torch.from_numpy(t1["depth"]),
                                     torch.from_numpy(t1["n_nodes"]), 0)
        inp = dict(kv)
        inp["draft"] = draft_ext[:, : w.N].contiguous()
        inp["target"] = target
        r = oracle_leg(w, inp, steps=args.steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * r["seconds"] / r["samples"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": wdesc,
                "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    rt = _cudart()

    # Independent input sets, rotated so that the step's inputs exceed L2.
    # Each rank is an independent replica with its own sequences (seeds).
    seed0 = 1000 * rank
    first, meta0 = make_set(w, seed0, dev)
    nbytes = set_bytes(first)
    R = max(1, min(16, math.ceil(2.0 * L2_BYTES / nbytes)))
    sets, metas = [first], [meta0]
    for s in range(1, R):
        i, m = make_set(w, seed0 + s, dev)
        sets.append(i)
        metas.append(m)
    nodes = [sum(m["n_nodes"]) for m in metas]

    stream = torch.cuda.Stream(dev)
    ex = jtree.Exec(dev)
    bufs = [StepBuffers(w, dev) for _ in range(R)]   # each set keeps its own tree / mask
    K, Wm = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(max(Wm, R)):
            run_step(w, sets[i % R], bufs[i % R], ex)
    stream.synchronize()
    if ex.read_error() != 0:
        raise RuntimeError("device error flag set during warm-up")
    acc_rows = [int(b_.acc["acc_len"].sum().item()) + w.batch for b_ in bufs]  # rows on the paths

    sptr = ctypes.c_void_p(stream.cuda_stream)

    def call_fns(inp, bf):
        return {
            "jt_topw": lambda: jtree.jt_topw(inp["draft"], w.W, bf.tok, bf.logp, exec=ex),
            "jt_tree_expand": lambda: jtree.jt_tree_expand(bf.tok, bf.logp, w.B, out=bf.tree,
                                                           exec=ex),
            "jt_tree_mask": lambda: jtree.jt_tree_mask(bf.tree["parent"], bf.tree["n_nodes"],
                                                       bf.mask, exec=ex),
            "jt_tree_attn": lambda: jtree.jt_tree_attn(
                inp["q"], inp["k_tree"], inp["v_tree"], inp["k_cache"], inp["v_cache"],
                inp["prefix_len"], bf.tree["n_nodes"], bf.mask, out=bf.attn_out,
                block_table=inp["block_table"], exec=ex),
            "jt_tree_accept": lambda: jtree.jt_tree_accept(inp["target"], bf.tree["parent"],
                                                           bf.tree["token"], bf.tree["n_nodes"],
                                                           w.N, out=bf.acc, exec=ex),
        }

    def capture(only=None):
        """K steps (only=None) or K launches of one call, events at the two ends."""
        events = [ctypes.c_void_p(), ctypes.c_void_p()]
        for ev in events:
            _ok(rt.cudaEventCreateWithFlags(ctypes.byref(ev), 0), "cudaEventCreateWithFlags")
        g = Graph(rt, stream)
        with torch.cuda.stream(stream):
            with g:
                _ok(rt.cudaEventRecordWithFlags(events[0], sptr, 1), "cudaEventRecordWithFlags")
                for i in range(K):
                    fns = call_fns(sets[i % R], bufs[i % R])
                    for c in CALLS:
                        if only is None or c == only:
                            fns[c]()
                _ok(rt.cudaEventRecordWithFlags(events[1], sptr, 1), "cudaEventRecordWithFlags")
        g.upload()
        return g, events

    def capture_fn(fn_of_step):
        """K launches of fn_of_step(i)(), events at the two ends."""
        events = [ctypes.c_void_p(), ctypes.c_void_p()]
        for ev in events:
            _ok(rt.cudaEventCreateWithFlags(ctypes.byref(ev), 0), "cudaEventCreateWithFlags")
        g = Graph(rt, stream)
        with torch.cuda.stream(stream):
            with g:
                _ok(rt.cudaEventRecordWithFlags(events[0], sptr, 1), "cudaEventRecordWithFlags")
                for i in range(K):
                    fn_of_step(i)()
                _ok(rt.cudaEventRecordWithFlags(events[1], sptr, 1), "cudaEventRecordWithFlags")
        g.upload()
        return g, events

    def elapsed(events):
        ms = ctypes.c_float(0)
        _ok(rt.cudaEventElapsedTime(ctypes.byref(ms), events[0], events[1]), "cudaEventElapsedTime")
        return ms.value

    def release(g_, evs):
        g_.close()
        for ev in evs:
            rt.cudaEventDestroy(ev)

    g_plain, ev_plain = capture()
    gpu_launches = g_plain.kernel_nodes()
    stream.synchronize()

    # ---- timed region (headline): K whole steps ------------------------------
    bus = ctypes.create_string_buffer(64)
    rt.cudaDeviceGetPCIBusId(bus, 64, local)
    sampler = ClockSampler(bus.value.decode())
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        g_plain.launch()
        stream.synchronize()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    # --------------------------------------------------------------------------
    total_ms = elapsed(ev_plain)
    release(g_plain, ev_plain)
    # ---- timed regions (per call): K launches of each call alone --------------
    per_call = {}
    for c in CALLS:
        g_c, ev_c = capture(only=c)
        torch.cuda.synchronize(dev)
        g_c.launch()
        stream.synchronize()
        per_call[c] = elapsed(ev_c) / K   # ms per launch of the call
        release(g_c, ev_c)
    if ex.read_error() != 0:
        raise RuntimeError("device error flag set during the timed regions")

    # ---- the accepted-path K/V commit (a row beyond the step: measured alone) ----
    # Its destinations get room for N more tokens per sequence (the workloads'
    # caches are sized to their prefixes): a contiguous buffer, or for paged
    # caches a small pool holding just the pages the commit writes, reached
    # through a block table whose other entries point at page 0. The bytes
    # moved are those of a commit into the real cache.
    commit_sets = []
    for i in range(R):
        inp, bf = sets[i], bufs[i]
        L = inp["prefix_len"].cpu()
        if w.paged:
            span = (w.N + 15) // 16 + 1
            mp = (int(L.max().item()) + w.N + 15) // 16
            table = torch.zeros((w.batch, mp), dtype=torch.int32)
            for b_ in range(w.batch):
                p0 = int(L[b_].item()) // 16
                for k in range(span):
                    if p0 + k < mp:
                        table[b_, p0 + k] = b_ * span + k
            kd = torch.zeros((w.batch * span, 16, w.hkv, w.D), dtype=torch.bfloat16, device=dev)
            table = table.to(dev)
        else:
            table = None
            kd = torch.zeros((w.batch, int(L.max().item()) + w.N, w.hkv, w.D),
                             dtype=torch.bfloat16, device=dev)
        commit_sets.append(dict(k=kd, v=torch.zeros_like(kd), table=table,
                                new_len=torch.empty_like(inp["prefix_len"])))

    def commit_fn(i):
        inp, bf, cs = sets[i % R], bufs[i % R], commit_sets[i % R]
        return lambda: jtree.jt_tree_commit_kv(
            inp["k_tree"], inp["v_tree"], cs["k"], cs["v"], inp["prefix_len"], bf.acc["acc_len"],
            bf.acc["acc_nodes"], new_prefix_len=cs["new_len"], block_table=cs["table"], exec=ex)

    # Entropy scan and hybrid-scored expansion (separate outputs, so the
    # step's own buffers are untouched).
    ent = [torch.empty((w.batch, w.N), dtype=torch.float32, device=dev) for _ in range(R)]
    scored = [{k: torch.empty_like(t) for k, t in bf.tree.items()} for bf in bufs]

    def entropy_fn(i):
        inp, bf = sets[i % R], bufs[i % R]
        return lambda: jtree.jt_topw(inp["draft"], w.W, bf.tok, bf.logp, exec=ex,
                                     entropy=ent[i % R])

    def scored_fn(i):
        bf = bufs[i % R]
        return lambda: jtree.jt_tree_expand(bf.tok, bf.logp, w.B, out=scored[i % R], exec=ex,
                                            entropy=ent[i % R], mode=jtree.JT_SCORE_HYBRID,
                                            alpha=0.5)

    sampled_out = [{k: torch.empty_like(t) for k, t in bf.acc.items()} for bf in bufs]

    def sampled_fn(i):
        inp, bf = sets[i % R], bufs[i % R]
        return lambda: jtree.jt_tree_accept(inp["target"], bf.tree["parent"], bf.tree["token"],
                                            bf.tree["n_nodes"], w.N, out=sampled_out[i % R],
                                            exec=ex, temperature=1.0, seed=1234 + i)

    # Draft LM head fused with top-W: the draft's hidden states for this
    # step's rows through a synthetic LM-head matrix of the target's shape
    # (d 4096, the workload's vocabulary; random weights: timing only).
    d_model = 4096
    gl = torch.Generator(device=dev).manual_seed(4242)
    w_lm = (torch.randn((w.V, d_model), generator=gl, device=dev) * 0.02).to(torch.bfloat16)
    hid = [(torch.randn((w.batch * w.N, d_model), generator=gl, device=dev)).to(torch.bfloat16)
           for _ in range(R)]
    lm_tok = [torch.empty((w.batch * w.N, w.W), dtype=torch.int32, device=dev) for _ in range(R)]
    lm_logp = [torch.empty((w.batch * w.N, w.W), dtype=torch.float32, device=dev)
               for _ in range(R)]

    def lmhead_fn(i):
        return lambda: jtree.jt_lmhead_topw(hid[i % R], w_lm, w.W, tok=lm_tok[i % R],
                                            logp=lm_logp[i % R], exec=ex)

    next_ms = {}
    with torch.cuda.stream(stream):
        for i in range(R):
            for fn in (commit_fn, entropy_fn, scored_fn, sampled_fn, lmhead_fn):
                fn(i)()
    stream.synchronize()
    if ex.read_error() != 0:
        raise RuntimeError("device error flag set by a next-row call")
    for name, fn in (("jt_tree_commit_kv", commit_fn), ("jt_topw_entropy", entropy_fn),
                     ("jt_tree_expand_scored", scored_fn), ("jt_tree_accept_sampled", sampled_fn),
                     ("jt_lmhead_topw", lmhead_fn)):
        g_c, ev_c = capture_fn(fn)
        torch.cuda.synchronize(dev)
        g_c.launch()
        stream.synchronize()
        next_ms[name] = elapsed(ev_c) / K
        release(g_c, ev_c)
    commit_ms = next_ms["jt_tree_commit_kv"]
    acc_tokens_sets = [int(bf.acc["acc_len"].sum().item()) for bf in bufs]
    commit_bytes = statistics.mean(acc_tokens_sets) * 2 * 2 * 2 * w.hkv * w.D  # K,V; read+write

    my_nodes = sum(nodes[i % R] for i in range(K))
    value = job_throughput(my_nodes, total_ms / 1000.0, dev)   # all ranks' nodes / slowest rank
    total_ms = max_over_ranks(total_ms, dev)

    # Roofline of the dominant call.
    peaks = load_peaks()
    works = [algorithmic_work(w, m["prefix_len"], m["n_nodes"], m["depth_sum"], pr)
             for m, pr in zip(metas, acc_rows)]
    avg_work = {c: {"bytes": statistics.mean(wk[c]["bytes"] for wk in works),
                    "flops": None if works[0][c]["flops"] is None
                    else statistics.mean(wk[c]["flops"] for wk in works)} for c in CALLS}
    dom = max(CALLS, key=lambda c: per_call[c])
    # Per-call durations come from each call timed alone: burst peaks apply.
    attn_tensor = avg_work["jt_tree_attn"]["flops"] / (
        peaks["bf16_tflops"] * 1e12) > avg_work["jt_tree_attn"]["bytes"] / (
        peaks["hbm_gbs"] * 1e9)
    if dom == "jt_tree_attn" and attn_tensor:
        achieved = avg_work[dom]["flops"] / (per_call[dom] / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        achieved = avg_work[dom]["bytes"] / (per_call[dom] / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = committed_traffic(dom, w.name)
    roof["peak_source"] = peaks["source"] + (" burst" if roof["bound"] == "tensor" else "")
    roof["algorithmic_per_launch"] = avg_work[dom]["flops"] if roof["bound"] == "tensor" \
        else avg_work[dom]["bytes"]

    calls_out = {}
    for c in CALLS:
        d = {"us": per_call[c] * 1e3, "share": per_call[c] / sum(per_call.values()),
             "alg_bytes": avg_work[c]["bytes"],
             "hbm_frac": avg_work[c]["bytes"] / (per_call[c] / 1e3) / 1e9 / peaks["hbm_gbs"]}
        if avg_work[c]["flops"]:
            d["alg_flops"] = avg_work[c]["flops"]
            d["tensor_frac"] = avg_work[c]["flops"] / (per_call[c] / 1e3) / (
                peaks["bf16_tflops"] * 1e12)
        calls_out[c] = d

    topw_b = avg_work["jt_topw"]["bytes"] + w.batch * w.N * 4
    lm_rows = w.batch * w.N
    lm_bytes = w.V * d_model * 2 + lm_rows * d_model * 2 + lm_rows * w.W * 8
    lm_flops = 2.0 * lm_rows * d_model * w.V
    lm_s = next_ms["jt_lmhead_topw"] / 1e3
    lm_row = {"us": lm_s * 1e6, "alg_bytes": lm_bytes, "alg_flops": lm_flops,
              "hbm_frac": lm_bytes / lm_s / 1e9 / peaks["hbm_gbs"],
              "tensor_frac": lm_flops / lm_s / (peaks["bf16_tflops"] * 1e12),
              "note": ("draft hidden [batch*N][4096] x synthetic LM head [vocab][4096] bf16, "
                       "top-W per row without writing logits; not in the step")}
    next_rows = {
        "jt_tree_commit_kv": {
            "us": commit_ms * 1e3, "alg_bytes": commit_bytes,
            "hbm_frac": commit_bytes / (commit_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "note": "accepted-path K/V commit, K launches alone; not in the step"},
        "jt_topw_entropy": {
            "us": next_ms["jt_topw_entropy"] * 1e3, "alg_bytes": topw_b,
            "hbm_frac": topw_b / next_ms["jt_topw_entropy"] * 1e3 / 1e9 / peaks["hbm_gbs"],
            "note": "top-W + log-softmax + per-depth entropy in one pass; not in the step"},
        "jt_tree_expand_scored": {
            "us": next_ms["jt_tree_expand_scored"] * 1e3,
            "note": "hybrid score (alpha 0.5) expansion; not in the step"},
        "jt_lmhead_topw": lm_row,
        "jt_tree_accept_sampled": {
            "us": next_ms["jt_tree_accept_sampled"] * 1e3,
            "note": ("temperature-1 acceptance (one Gumbel-max draw per visited node, "
                     "counter-based noise for every logit it scans); not in the step")},
    }

    # ---- end to end through the public API with host buffers ---------------
    e2e_steps = args.e2e_steps or max(3, min(K, 200))
    host = {k: (None if t is None else t.cpu().pin_memory()) for k, t in sets[0].items()}
    devb = {k: (None if t is None else torch.empty_like(t)) for k, t in sets[0].items()}
    res_keys = ["acc_len", "acc_tokens", "bonus"]
    buf = bufs[0]
    res_host = {k: torch.empty(buf.acc[k].shape, dtype=buf.acc[k].dtype).pin_memory()
                for k in res_keys}
    n_host = torch.empty((w.batch,), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in res_host.values()) + n_host.numel() * 4
    with torch.cuda.stream(stream):
        def e2e_step():
            for k, t in host.items():
                if t is not None:
                    devb[k].copy_(t, non_blocking=True)
            run_step(w, devb, buf, ex)
            for k in res_keys:
                res_host[k].copy_(buf.acc[k], non_blocking=True)
            n_host.copy_(buf.tree["n_nodes"], non_blocking=True)
            stream.synchronize()  # the caller reads the accepted tokens every step
        for _ in range(3):
            e2e_step()
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_s = time.perf_counter() - t0
    e2e_value = job_throughput(e2e_steps * nodes[0], e2e_s, dev)
    e2e = {"value": e2e_value, "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = oracle_leg(w, sets[0])
        cpu = {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if rank == 0:
        wdesc["l2"] = (f"{R} rotating input sets of {nbytes / 1e6:.1f} MB "
                       f"({R * nbytes / 1e6:.0f} MB > 129 MB L2)" if R > 1 else
                       f"inputs of {nbytes / 1e6:.0f} MB per step exceed the 129 MB L2")
        wdesc["graph"] = ("K steps captured in one CUDA graph, launched once; per-call times from "
                          "one graph per call of K launches of that call alone (same input sets)")
        wdesc["nodes_per_step"] = statistics.mean(nodes)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32",
                "data": "synthetic (seeded, no dataset or weights)", "config": wdesc,
                "impl": "libjtree", "roofline": roof, "calls": calls_out,
                "next_rows": next_rows,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches * world,
                "clocks": sampler.summary()}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
