"""The DRAM traffic a bench line reports comes from the capture of its own
variant of the path (workload, recompute, fp32, tile shape) and only while the
kernel sources are the ones it was taken on."""
import argparse
import json
import os

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _args(**kw):
    a = dict(rows=0, vocab=0, chunk_rows=0, vocab_slab=0, ce_logits=False, low_memory=False, fp32=False,
             tile128=False)
    a.update(kw)
    return argparse.Namespace(**a)


def _recorded():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_keys_name_the_variant():
    w = workloads.WORKLOADS["dsv3"]
    assert bench._traffic_key(_args(), w) == "dsv3"
    assert bench._traffic_key(_args(low_memory=True), w) == "dsv3-lowmem"
    assert bench._traffic_key(_args(fp32=True), w) == "dsv3-fp32"
    assert bench._traffic_key(_args(tile128=True), w) == "dsv3-tile128"
    assert bench._traffic_key(_args(ce_logits=True), workloads.WORKLOADS["llama"]) == "llama-ce_logits"
    for over in (dict(rows=2048), dict(vocab=32768), dict(chunk_rows=4096), dict(vocab_slab=8192)):
        assert bench._traffic_key(_args(**over), w) is None, over


def test_each_variant_reports_its_own_capture():
    rec = _recorded()
    w = workloads.WORKLOADS["dsv3"]
    if rec["dsv3"]["grad_W_gemm"]["source_sha256"] != bench.kernel_source_hash():
        return              # kernels changed since the capture: nothing is reported (next test)
    bf16 = bench.recorded_traffic(bench._traffic_key(_args(), w), "grad_W_gemm")
    tf32 = bench.recorded_traffic(bench._traffic_key(_args(fp32=True), w), "grad_W_gemm")
    assert bf16 == rec["dsv3"]["grad_W_gemm"]["bytes_per_launch"]
    assert tf32 == rec["dsv3-fp32"]["grad_W_gemm"]["bytes_per_launch"] and tf32 != bf16
    assert bench.recorded_traffic(bench._traffic_key(_args(tile128=True), w), "grad_W_gemm") is None
    assert bench.recorded_traffic(None, "grad_W_gemm") is None


def test_other_chunk_sizes_report_no_traffic():
    """A capture holds launches of one chunk size; a line whose call chunks
    differently (the frozen head's default of 9728 rows, say) gets none."""
    rec = _recorded()
    if rec["dsv3"]["fwd_gemm_stats"]["source_sha256"] != bench.kernel_source_hash():
        return
    assert bench.recorded_traffic("dsv3", "fwd_gemm_stats", 8192) is not None
    assert bench.recorded_traffic("dsv3", "fwd_gemm_stats", 9728) is None
    for key, kernels in rec.items():
        if not key.startswith("_"):
            assert all(e["chunk_rows"] % 128 == 0 for e in kernels.values()), key
    # the frozen head's forward + grad_h line runs 9728-row chunks by default
    assert rec["frozen_grad_h"]["grad_h_gemm"]["chunk_rows"] == 9728


def test_changed_kernels_report_no_traffic(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 64)
    assert bench.recorded_traffic("dsv3", "fwd_gemm_stats") is None


def test_recorded_entries_are_whole():
    for key, kernels in _recorded().items():
        if key.startswith("_"):
            continue
        for name, e in kernels.items():
            assert abs(e["bytes_per_launch"] - (e["dram_read"] + e["dram_write"])) < 1.0, (key, name)
            assert len(e["source_sha256"]) == 64 and "--clock-control none" in e["command"], (key, name)
            assert "bench.py" in e["command"], (key, name)
