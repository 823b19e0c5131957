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
