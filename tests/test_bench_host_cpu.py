"""Host-side logic of the bench that decides whether a number stands: the
clock record taken during the timed region, and the committed ncu traffic
that is reported only for the kernel sources it was taken on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_clock_summary_median_max_and_reasons():
    lines = [
        "0, 2070, 2070, 1100.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1395.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070",          # a non-numeric sample is skipped
        "0, 2070",                 # a partial last line is skipped
    ]
    r = bench.Clocks.summarize(lines)
    assert r["samples"] == 3 and r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_slowdown_and_empty_record():
    lines = ["0, 1500, 2070, 900, 0x40, Not Active, Active, Not Active, Not Active"]
    r = bench.Clocks.summarize(lines)
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1500.0
    assert bench.Clocks.summarize([]) is None


def test_traffic_reported_only_for_the_sources_it_was_taken_on(monkeypatch):
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    key = "decode_fused_kernel/llama8b_decode"
    files = ["decode.cu", "dkv_internal.cuh"]
    # sources with the hash the record was taken on: the record is reported
    monkeypatch.setattr(bench, "kernel_source_hash", lambda fs: rec[key]["src_sha256_16"])
    assert bench.ncu_traffic(key, files)["host_link_bytes"] == rec[key]["host_link_bytes"]
    # any change to the sources (a different hash) withdraws it
    monkeypatch.setattr(bench, "kernel_source_hash", lambda fs: "0" * 16)
    assert bench.ncu_traffic(key, files) is None
    assert bench.ncu_traffic("no_such_kernel/none", files) is None


def test_oracle_prefill_sample_counts_its_work():
    """The CPU-baseline sample of the prefill: a positive time, the thread
    count it ran on, and FLOPs = the whole projection plus the attention of
    the sampled rows (first and last token included), each row over all heads."""
    from zero_copy_offloaded_gb300 import workloads as wl
    w = wl.Workload("t", "prefill", B=1, H=64, Hq=4, Hkv=2, D=16, P=40, T=12, seed=3)
    dt, cores, flops, sample = bench.oracle_prefill_sample(w, nrows=5)
    assert dt > 0 and cores >= 1
    attn = flops - w.proj_flops()
    per_key = 4 * w.Hq * w.D
    assert attn % per_key == 0
    keys = attn // per_key  # sum over the sampled rows t of P + t + 1
    # five distinct rows among 0..T-1, the first and last included
    lo = (w.P + 1) + (w.P + w.T) + sum(w.P + 1 + t for t in range(1, 4))
    hi = (w.P + 1) + (w.P + w.T) + sum(w.P + 1 + t for t in range(w.T - 4, w.T - 1))
    assert lo <= keys <= hi
    assert "5 seeded query rows" in sample
