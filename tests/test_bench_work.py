"""The algorithmic work bench.py divides by to report roofline fractions,
checked against sums done by hand for the batch-1 chain workload (one
sequence, prefix 2048, a 16-node chain, 32 query / 8 KV heads of 128,
vocabulary 151936, width 1)."""
import importlib.util
import json
import os

from tree_causal_verification_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def test_chain_workload_shape():
    w = synth.WORKLOADS["qwen3-8b-chain"]
    assert (w.batch, w.prefix_lo, w.prefix_hi, w.B, w.N, w.W) == (1, 2048, 2048, 16, 16, 1)
    assert (w.hq, w.hkv, w.D, w.V) == (32, 8, 128, 151936)


def test_chain_algorithmic_work():
    w = synth.WORKLOADS["qwen3-8b-chain"]
    # A chain of 16 nodes: depths 1..16, 136 ancestor-or-self pairs in all;
    # one accepted row read (acc_len 0 + the root row).
    work = bench.algorithmic_work(w, [2048], [16], 136, 1)
    # Prefix K and V: 2048 keys x 8 heads x 128 x 2 bytes x 2 = 8,388,608;
    # tree K and V 65,536; q in and out 262,144.
    assert work["jt_tree_attn"]["bytes"] == 8_716_288
    # 4 flops per (query row, visible key, head dim): 32 heads x 128 x
    # (16 x 2048 + 136) x 4.
    assert work["jt_tree_attn"]["flops"] == 539_099_136
    # 16 rows of 151936 fp32 logits read, 16 (token, logp) pairs written.
    assert work["jt_topw"]["bytes"] == 9_724_032
    # One row of target logits plus the tree (parent and token, 8 bytes a node).
    assert work["jt_tree_accept"]["bytes"] == 151936 * 4 + 16 * 8
    assert work["jt_tree_mask"]["bytes"] == 16 * 4 + 16 * 1 * 4


def test_peaks_are_the_measured_ones():
    peaks = bench.load_peaks()
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        assert peaks["source"] == "measured"
        assert peaks["hbm_gbs"] == d["hbm_gbs"] and peaks["bf16_tflops"] == d["bf16_tflops"]
    else:
        assert peaks["source"] == "fallback"


def test_committed_traffic_follows_the_source():
    """A recorded DRAM traffic figure is reported only for the source it was taken on."""
    t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for call, per_workload in t.items():
        for workload, rec in per_workload.items():
            got = bench.committed_traffic(call, workload)
            if rec["sha1"] == bench.source_sha(call):
                assert got == rec["bytes_per_launch"]
            else:
                assert got is None
