#!/usr/bin/env python3
"""Benchmark: tree nodes verified per second for one decode step's hot path.

A step is the whole path through libjtree's C ABI on inputs resident in HBM:
top-W per depth -> best-first expansion -> tree mask -> tree attention ->
greedy acceptance. The headline workload (default) is the largest one that
fits one GPU: batch 64, prefixes U[2048, 16384] in 16-token pages, a
128-node tree (N=16, W=4) per sequence, 32 query / 4 KV heads of 128,
vocabulary 151936 (MoE-target attention shape). The other four workloads
(tiny, Qwen3-8B chain, high budget, mid-batch) are measured in the same run
and reported under "per_config".

Timing: W eager warm-up steps, then EXACTLY K steps captured into one CUDA
graph and launched once, bracketed by a barrier and a device synchronise on
both sides, timed by CUDA events recorded on the launching stream at the two
ends. Each call's average duration comes from a further timed region per
call: one graph of K launches of that call alone on the same input sets
(events at its two ends); those feed the roofline figures. Steps rotate
through enough independent input sets that the inputs exceed the 129 MB L2
(or one set alone exceeds it). SM clocks and throttle reasons are sampled
through NVML during the timed regions.

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path shards by sequence with no exchange: weak scaling); value = nodes of all
ranks / the slowest rank's time.

The CPU oracle (the plain C++ reference, untuned) is timed on whole steps:
every row of a sequence's step (its top-W rows, expansion, mask, every
(node, head) attention row, acceptance walk), with the rows of a step spread
over the host's cores (each thread runs the unchanged single-threaded oracle
on its share). --impl reference times only that oracle, one sequence's whole
step per timed step.

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
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree nodes verified/sec per step (attn+top-W+accept); % of GB300 HBM/tensor roofline"
UNIT = "nodes/s"
DEFAULT_WORKLOAD = "moe-paged"
L2_BYTES = 129e6
CALLS = ["jt_topw", "jt_tree_expand", "jt_tree_mask", "jt_tree_attn", "jt_tree_accept"]
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
# CPU oracle: whole steps on the host cores.
# --------------------------------------------------------------------------
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleInputs:
    """Host copies of one input set for the oracle (bf16 tensors as bit
    patterns). Draft and target rows are copied per sequence, untimed."""

    def __init__(self, w, inp):
        import numpy as np
        import torch

        def bits(t):
            return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)

        self.w = w
        self.q, self.kt, self.vt = bits(inp["q"]), bits(inp["k_tree"]), bits(inp["v_tree"])
        self.kc, self.vc = bits(inp["k_cache"]), bits(inp["v_cache"])
        self.prefix = inp["prefix_len"].cpu().numpy()
        self.bt = None if inp["block_table"] is None else inp["block_table"].cpu().numpy()
        self._draft, self._target = inp["draft"], inp["target"]

    def rows_of(self, b):
        """(draft [1][N][V], target [1][B+1][V]) of sequence b, float32 on the host."""
        return self._draft[b:b + 1].cpu().numpy(), self._target[b:b + 1].cpu().numpy()


def oracle_sequence_step(oi, b, rows, pool, threads):
    """The oracle's whole step for sequence b: its N top-W rows, the
    expansion, the mask, every (node, head) attention row and the acceptance
    walk. With threads > 1 the top-W rows and the attention rows are spread
    over the pool (each task is the unchanged single-threaded oracle on its
    rows). Returns (nodes, seconds)."""
    import numpy as np

    import oracle
    w = oi.w
    draft, target = rows
    paged = oi.bt is not None
    sl = slice(b, b + 1)
    t0 = time.perf_counter()
    if threads > 1:
        parts = list(pool.map(lambda d: oracle.topw(draft[:, d:d + 1], w.W), range(w.N)))
        tok = np.concatenate([p[0] for p in parts], axis=1)
        logp = np.concatenate([p[1] for p in parts], axis=1)
    else:
        tok, logp = oracle.topw(draft, w.W)
    tree = oracle.tree_expand(tok, logp, w.B)
    mask = oracle.tree_mask(tree["parent"], tree["n_nodes"])
    n = int(tree["n_nodes"][0])
    rws = np.array([(0, v, h) for v in range(n) for h in range(w.hq)], np.int32).reshape(-1, 3)

    def attn(r):
        return oracle.tree_attn(oi.q[sl], oi.kt[sl], oi.vt[sl], oi.kc if paged else oi.kc[sl],
                                oi.vc if paged else oi.vc[sl], oi.prefix[sl], tree["n_nodes"],
                                mask, hq=w.hq, hkv=w.hkv, block_table=oi.bt[sl] if paged else None,
                                rows=r)

    if threads > 1 and len(rws) > 1:
        list(pool.map(attn, np.array_split(rws, min(len(rws), 4 * threads))))
    elif len(rws):
        attn(rws)
    oracle.tree_accept(target, tree["parent"], tree["token"], tree["n_nodes"], w.N)
    return n, time.perf_counter() - t0


def oracle_timing(w, inp, seqs, threads, budget_s=None, warmup=0):
    """Times the oracle's whole step for the sequences `seqs`, in order, on
    `threads` host threads; stops once budget_s seconds of oracle time are
    spent (at least one sequence). Returns dict(nodes, seconds, seqs)."""
    import concurrent.futures as cf

    import oracle
    oracle.build()
    oi = OracleInputs(w, inp)
    nodes, secs, done = 0, 0.0, []
    with cf.ThreadPoolExecutor(max_workers=threads) as pool:
        for i in range(warmup):
            b = seqs[i % len(seqs)]
            oracle_sequence_step(oi, b, oi.rows_of(b), pool, threads)
        for b in seqs:
            n, dt = oracle_sequence_step(oi, b, oi.rows_of(b), pool, threads)
            nodes += n
            secs += dt
            done.append(b)
            if budget_s is not None and secs >= budget_s:
                break
    return {"nodes": nodes, "seconds": secs, "seqs": done}


def describe_oracle(w, r, threads, whole):
    what = ("the whole step (every sequence)" if whole else
            f"{len(r['seqs'])} of the {w.batch} sequences, each sequence's whole step")
    return (f"oracle on {what} of {w.name}: top-W of its {w.N} rows (V={w.V}), expansion, mask, "
            f"attention of every (node, head) row over its prefix and tree keys, acceptance walk; "
            f"{r['nodes']} nodes in {r['seconds']:.2f} s on {threads} host thread(s)")


# --------------------------------------------------------------------------
# GPU measurement of one workload.
# --------------------------------------------------------------------------
def call_fns(w, jtree, inp, bf, ex):
    return {
        "jt_topw": lambda: jtree.jt_topw(inp["draft"], w.W, bf.tok, bf.logp, exec=ex),
        "jt_tree_expand": lambda: jtree.jt_tree_expand(bf.tok, bf.logp, w.B, out=bf.tree, exec=ex),
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


class Timer:
    """CUDA graphs of K launches with events at their two ends."""

    def __init__(self, rt, stream):
        self.rt, self.stream = rt, stream
        self.sptr = ctypes.c_void_p(stream.cuda_stream)

    def capture(self, body):
        import torch
        events = [ctypes.c_void_p(), ctypes.c_void_p()]
        for ev in events:
            _ok(self.rt.cudaEventCreateWithFlags(ctypes.byref(ev), 0), "cudaEventCreateWithFlags")
        g = Graph(self.rt, self.stream)
        with torch.cuda.stream(self.stream):
            with g:
                _ok(self.rt.cudaEventRecordWithFlags(events[0], self.sptr, 1),
                    "cudaEventRecordWithFlags")
                body()
                _ok(self.rt.cudaEventRecordWithFlags(events[1], self.sptr, 1),
                    "cudaEventRecordWithFlags")
        g.upload()
        return g, events

    def elapsed(self, events):
        ms = ctypes.c_float(0)
        _ok(self.rt.cudaEventElapsedTime(ctypes.byref(ms), events[0], events[1]),
            "cudaEventElapsedTime")
        return ms.value

    def release(self, g, events):
        g.close()
        for ev in events:
            self.rt.cudaEventDestroy(ev)

    def run(self, body, dev, sampler=None, dist=None):
        """Captures body (K launches), then times one launch of the graph."""
        import torch
        g, ev = self.capture(body)
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        if sampler is not None:
            with sampler:
                g.launch()
                self.stream.synchronize()
        else:
            g.launch()
            self.stream.synchronize()
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
        ms = self.elapsed(ev)
        nodes = g.kernel_nodes()
        self.release(g, ev)
        return ms, nodes


def measure(w, K, Wm, dev, stream, timer, ex, seed0=0, dist=None, local=0):
    """K whole steps (the headline timed region) and K launches of each call
    alone, on rotating input sets; returns the raw measurements."""
    import torch
    from tree_causal_verification_gb300.step import StepBuffers, run_step
    first, meta0 = make_set(w, seed0, dev)
    nbytes = set_bytes(first)
    R = max(1, min(16, math.ceil(2.0 * L2_BYTES / nbytes)))
    sets, metas = [first], [meta0]
    for s in range(1, R):
        i, m = make_set(w, seed0 + s, dev)
        sets.append(i)
        metas.append(m)
    bufs = [StepBuffers(w, dev) for _ in range(R)]   # each set keeps its own tree / mask
    with torch.cuda.stream(stream):
        for i in range(max(Wm, R)):
            run_step(w, sets[i % R], bufs[i % R], ex)
    stream.synchronize()
    if ex.read_error() != 0:
        raise RuntimeError(f"device error flag set during warm-up ({w.name})")
    acc_rows = [int(b_.acc["acc_len"].sum().item()) + w.batch for b_ in bufs]  # rows on the paths

    def steps():
        for i in range(K):
            fns = call_fns(w, jtree_mod(), sets[i % R], bufs[i % R], ex)
            for c in CALLS:
                fns[c]()

    bus = ctypes.create_string_buffer(64)
    timer.rt.cudaDeviceGetPCIBusId(bus, 64, local)
    sampler = ClockSampler(bus.value.decode())
    total_ms, launches = timer.run(steps, dev, sampler=sampler, dist=dist)
    per_call = {}
    for c in CALLS:
        def one(c=c):
            for i in range(K):
                call_fns(w, jtree_mod(), sets[i % R], bufs[i % R], ex)[c]()
        per_call[c] = timer.run(one, dev)[0] / K     # ms per launch of the call
    if ex.read_error() != 0:
        raise RuntimeError(f"device error flag set during the timed regions ({w.name})")
    return {"w": w, "total_ms": total_ms, "per_call": per_call, "launches": launches,
            "nodes": [sum(m["n_nodes"]) for m in metas], "metas": metas, "acc_rows": acc_rows,
            "R": R, "nbytes": nbytes, "sets": sets, "bufs": bufs, "clocks": sampler.summary()}


def jtree_mod():
    from tree_causal_verification_gb300 import jtree
    return jtree


def summarise(m, peaks, K):
    """Per-call times and roofline fractions of one workload's measurement."""
    w = m["w"]
    works = [algorithmic_work(w, mt["prefix_len"], mt["n_nodes"], mt["depth_sum"], pr)
             for mt, pr in zip(m["metas"], m["acc_rows"])]
    avg = {c: {"bytes": statistics.mean(wk[c]["bytes"] for wk in works),
               "flops": None if works[0][c]["flops"] is None
               else statistics.mean(wk[c]["flops"] for wk in works)} for c in CALLS}
    pc = m["per_call"]
    calls = {}
    for c in CALLS:
        d = {"us": pc[c] * 1e3, "share": pc[c] / sum(pc.values()), "alg_bytes": avg[c]["bytes"],
             "hbm_frac": avg[c]["bytes"] / (pc[c] / 1e3) / 1e9 / peaks["hbm_gbs"]}
        if avg[c]["flops"]:
            d["alg_flops"] = avg[c]["flops"]
            d["tensor_frac"] = avg[c]["flops"] / (pc[c] / 1e3) / (peaks["bf16_tflops"] * 1e12)
        calls[c] = d
    dom = max(CALLS, key=lambda c: pc[c])
    # Per-call durations come from each call timed alone: burst peaks apply.
    tensor = avg[dom]["flops"] is not None and avg[dom]["flops"] / (peaks["bf16_tflops"] * 1e12) \
        > avg[dom]["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if tensor:
        roof = {"kernel": dom, "bound": "tensor",
                "achieved": avg[dom]["flops"] / (pc[dom] / 1e3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": avg[dom]["bytes"] / (pc[dom] / 1e3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # A recorded figure is per launch of the named workload at its own size.
    from tree_causal_verification_gb300 import synth
    roof["traffic"] = committed_traffic(dom, w.name) if synth.WORKLOADS.get(w.name) == w else None
    roof["peak_source"] = peaks["source"] + (" burst" if tensor else " copy")
    roof["algorithmic_per_launch"] = avg[dom]["flops"] if tensor else avg[dom]["bytes"]
    nodes_per_step = statistics.mean(m["nodes"])
    my_nodes = sum(m["nodes"][i % m["R"]] for i in range(K))
    return {"roofline": roof, "calls": calls, "nodes_per_step": nodes_per_step,
            "my_nodes": my_nodes, "ms_per_step": m["total_ms"] / K}


def l2_note(m):
    R, nbytes = m["R"], m["nbytes"]
    return (f"{R} rotating input sets of {nbytes / 1e6:.1f} MB ({R * nbytes / 1e6:.0f} MB > "
            f"129 MB L2)" if R > 1 else f"inputs of {nbytes / 1e6:.0f} MB per step exceed the "
            f"129 MB L2")


def workload_desc(w):
    return {"workload": w.name, "batch": w.batch, "prefix": [w.prefix_lo, w.prefix_hi],
            "B": w.B, "N": w.N, "W": w.W, "hq": w.hq, "hkv": w.hkv, "head_dim": w.D,
            "vocab": w.V, "paged": w.paged}


def next_rows_of(w, m, K, dev, timer, ex, peaks):
    """Rows beyond the step, each call timed alone (K launches in a graph)."""
    import torch
    jtree = jtree_mod()
    sets, bufs, R = m["sets"], m["bufs"], m["R"]
    # The accepted-path K/V commit. Its destinations get room for N more
    # tokens per sequence (the workloads' caches are sized to their
    # prefixes): a contiguous buffer, or for paged caches a small pool holding
    # just the pages the commit writes, reached through a block table whose
    # other entries point at page 0. The bytes moved are those of a commit
    # into the real cache.
    commit_sets = []
    for i in range(R):
        inp = sets[i]
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

    fns = (("jt_tree_commit_kv", commit_fn), ("jt_topw_entropy", entropy_fn),
           ("jt_tree_expand_scored", scored_fn), ("jt_tree_accept_sampled", sampled_fn),
           ("jt_lmhead_topw", lmhead_fn))
    with torch.cuda.stream(timer.stream):
        for i in range(R):
            for _, fn in fns:
                fn(i)()
    timer.stream.synchronize()
    if ex.read_error() != 0:
        raise RuntimeError("device error flag set by a next-row call")
    next_ms = {}
    for name, fn in fns:
        def body(fn=fn):
            for i in range(K):
                fn(i)()
        next_ms[name] = timer.run(body, dev)[0] / K
    commit_ms = next_ms["jt_tree_commit_kv"]
    acc_tokens_sets = [int(bf.acc["acc_len"].sum().item()) for bf in bufs]
    commit_bytes = statistics.mean(acc_tokens_sets) * 2 * 2 * 2 * w.hkv * w.D  # K,V; read+write
    topw_b = w.batch * w.N * (4 * w.V + 8 * w.W) + w.batch * w.N * 4
    lm_rows = w.batch * w.N
    lm_bytes = w.V * d_model * 2 + lm_rows * d_model * 2 + lm_rows * w.W * 8
    lm_flops = 2.0 * lm_rows * d_model * w.V
    lm_s = next_ms["jt_lmhead_topw"] / 1e3
    return {
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
        "jt_lmhead_topw": {
            "us": lm_s * 1e6, "alg_bytes": lm_bytes, "alg_flops": lm_flops,
            "hbm_frac": lm_bytes / lm_s / 1e9 / peaks["hbm_gbs"],
            "tensor_frac": lm_flops / lm_s / (peaks["bf16_tflops"] * 1e12),
            "note": ("draft hidden [batch*N][4096] x synthetic LM head [vocab][4096] bf16, "
                     "top-W per row without writing logits; not in the step")},
        "jt_tree_accept_sampled": {
            "us": next_ms["jt_tree_accept_sampled"] * 1e3,
            "note": ("temperature-1 acceptance (one Gumbel-max draw per visited node, "
                     "counter-based noise for every logit it scans); not in the step")},
    }


def end_to_end(w, m, K, dev, stream, ex, e2e_steps, dist=None):
    """The same metric through the public API with host buffers: every step
    copies its inputs from pinned host memory, runs the five calls and reads
    the accepted tokens back (synchronising, as a caller would)."""
    import torch
    from tree_causal_verification_gb300.step import run_step
    src = m["sets"][0]
    host = {}
    for k, t in src.items():
        if t is None:
            host[k] = None
        else:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host[k] = h
    devb = {k: (None if t is None else torch.empty_like(t)) for k, t in src.items()}
    res_keys = ["acc_len", "acc_tokens", "bonus"]
    buf = m["bufs"][0]
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
    del devb, host
    from tree_causal_verification_gb300.dist import job_throughput
    return {"value": job_throughput(e2e_steps * m["nodes"][0], e2e_s, dev), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}


# --------------------------------------------------------------------------
# The reference arm: the CPU oracle alone.
# --------------------------------------------------------------------------
def reference_arm(args, w, rank):
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"   # input generation only
    inp, meta = make_oracle_set(w, 0, dev)
    threads = host_cores()
    seqs = [i % w.batch for i in range(args.steps)]
    r = oracle_timing(w, inp, seqs, threads, warmup=args.warmup)
    value = r["nodes"] / r["seconds"]
    sample = describe_oracle(w, r, threads, whole=False) + \
        f"; {args.warmup} untimed warm-up sequence step(s)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * r["seconds"] / len(r["seqs"]), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_desc(w), step="one sequence's whole step per timed step"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def make_oracle_set(w, seed, dev):
    """The benchmark's inputs for the oracle alone: drawn like make_set (on the
    GPU when there is one, so the bytes are the GPU arm's), with the target
    rows drawn for the oracle's own tree."""
    import torch

    import oracle
    from tree_causal_verification_gb300 import synth
    draft_ext = synth.draft_logits(w, seed, dev)
    kv = synth.kv_inputs(w, seed, dev)
    oracle.build()
    tok, logp = oracle.topw(draft_ext[:, : w.N].cpu().numpy(), w.W)
    tree = oracle.tree_expand(tok, logp, w.B)
    target = synth.target_logits(w, draft_ext, torch.from_numpy(tree["depth"]),
                                 torch.from_numpy(tree["n_nodes"]), seed)
    inp = dict(kv)
    inp["draft"] = draft_ext[:, : w.N].contiguous()
    inp["target"] = target
    return inp, {"n_nodes": tree["n_nodes"].tolist()}


# --------------------------------------------------------------------------
# Main.
# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="jtree", choices=["jtree", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the headline workload")
    ap.add_argument("--no-next-rows", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the headline workload's batch (smaller profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    import torch
    from tree_causal_verification_gb300 import jtree, synth
    from tree_causal_verification_gb300.dist import job_throughput, max_over_ranks, rank_world

    rank, world, local = rank_world()
    w = synth.WORKLOADS[args.workload]
    if args.batch is not None:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch)
    if args.impl == "reference":
        reference_arm(args, w, rank)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    rt = _cudart()
    stream = torch.cuda.Stream(dev)
    timer = Timer(rt, stream)
    ex = jtree.Exec(dev)
    K, Wm = args.steps, args.warmup
    peaks = load_peaks()

    # ---- headline workload (each rank an independent replica) ----
    m = measure(w, K, Wm, dev, stream, timer, ex, seed0=1000 * rank, dist=dist, local=local)
    sm = summarise(m, peaks, K)
    value = job_throughput(sm["my_nodes"], m["total_ms"] / 1000.0, dev)
    total_ms = max_over_ranks(m["total_ms"], dev)
    next_rows = None if args.no_next_rows else next_rows_of(w, m, K, dev, timer, ex, peaks)
    e2e = end_to_end(w, m, K, dev, stream, ex, args.e2e_steps or max(3, min(K, 50)), dist)
    cpu_inp = m["sets"][0]
    launches, clocks = m["launches"], m["clocks"]
    wdesc = workload_desc(w)
    wdesc["l2"] = l2_note(m)
    wdesc["nodes_per_step"] = sm["nodes_per_step"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_cores()
        r = oracle_timing(w, cpu_inp, list(range(w.batch)), threads, budget_s=15.0)
        cpu = {"value": r["nodes"] / r["seconds"], "unit": UNIT, "cores": threads,
               "kind": "oracle", "sample": describe_oracle(w, r, threads, whole=w.batch == 1)}
    del m, cpu_inp
    torch.cuda.empty_cache()

    # ---- the other workloads, same run (single-GPU runs only) ----
    per_config = {}
    if world == 1 and not args.no_per_config:
        for name in synth.WORKLOAD_ORDER:
            if name == w.name:
                continue
            wo = synth.WORKLOADS[name]
            mo = measure(wo, K, Wm, dev, stream, timer, ex, local=local)
            so = summarise(mo, peaks, K)
            entry = {"value": so["my_nodes"] / (mo["total_ms"] / 1000.0), "unit": UNIT,
                     "ms_per_step": so["ms_per_step"], "nodes_per_step": so["nodes_per_step"],
                     "config": dict(workload_desc(wo), l2=l2_note(mo)),
                     "roofline": so["roofline"], "calls": so["calls"], "clocks": mo["clocks"],
                     "gpu_launches": mo["launches"]}
            if rank == 0 and not args.no_cpu_baseline:
                # The oracle on the whole step: all host cores, and one core
                # where a whole step takes at most a few seconds.
                threads = host_cores()
                seqs = list(range(wo.batch))
                r = oracle_timing(wo, mo["sets"][0], seqs, threads)
                entry["cpu_baseline"] = {
                    "value": r["nodes"] / r["seconds"], "unit": UNIT, "cores": threads,
                    "kind": "oracle", "sample": describe_oracle(wo, r, threads, whole=True)}
                if wo.batch == 1:
                    r1 = oracle_timing(wo, mo["sets"][0], seqs, 1)
                    entry["cpu_baseline_1core"] = {
                        "value": r1["nodes"] / r1["seconds"], "unit": UNIT, "cores": 1,
                        "kind": "oracle", "sample": describe_oracle(wo, r1, 1, whole=True)}
            per_config[name] = entry
            del mo
            torch.cuda.empty_cache()

    if rank == 0:
        wdesc["graph"] = ("K steps captured in one CUDA graph, launched once; per-call times from "
                          "one graph per call of K launches of that call alone (same input sets)")
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
                "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32",
                "data": "synthetic (seeded, no dataset or weights)", "config": wdesc,
                "impl": "libjtree", "roofline": sm["roofline"], "calls": sm["calls"],
                "next_rows": next_rows, "per_config": per_config,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * world,
                "clocks": clocks}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
