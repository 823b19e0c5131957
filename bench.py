#!/usr/bin/env python
"""Benchmark of the zero-copy host-resident KV-cache attention path on GB300.

Default line: Llama-3-8B-shaped single-layer fused decode (B=8, 32/8 heads,
head_dim 128, bf16, 32768 cached tokens per sequence in pinned, mapped host
memory).  One step = one dkv_decode call (projection of the new token, append
to the host cache, split-KV attention over the host-resident cache, combine).
Lengths are reset between steps so every step appends at the same position.

Reported alongside (same run, same process):
  * the host-link read/write rate of a plain zero-copy streaming kernel (the
    roofline denominator for the decode), the HBM read rate, cudaMemcpy H2D;
  * two internal baselines on the same cache: naive untiled zero-copy
    attention and copy-to-HBM-then-attend;
  * the Llama-3-8B-shaped chunked prefill (T=4096 over a 28672-token prefix):
    TFLOP/s against the min-of-rooflines bound;
  * the fp64 CPU oracle timed on this host (a bounded sample).

--impl reference times the CPU oracle (the only reference available for this
method) on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from zero_copy_offloaded_gb300 import workloads as wl  # noqa: E402

L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dkv", choices=["dkv", "reference"])
    ap.add_argument("--workload", default="llama8b_decode")
    ap.add_argument("--prefill-workload", default="llama8b_prefill")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the headline decode (no baselines, prefill, oracle timing)")
    ap.add_argument("--prefill-only", action="store_true")
    ap.add_argument("--profile-prefill", action="store_true",
                    help="profiling aid: two warm-up prefill calls, then one fused prefill and "
                         "one naive untiled prefill of --prefill-workload, untimed")
    ap.add_argument("--sweep", action="store_true",
                    help="one JSON line per workload: every decode workload with its naive and "
                         "copy-to-HBM baselines, then every prefill workload")
    return ap.parse_args()


def bench_fp8_decode(w, dkv, torch, dev, stream, flush, link_rd, steps):
    """The decode workload on an 8-bit E4M3 cache (the same values, converted
    with torch's float8 type as input construction): half the host bytes."""
    tdt = torch.bfloat16
    cache = dkv.KVCache(w.B, w.Hkv, w.D, w.S_max, w.dtype, kv_format="e4m3")
    for b in range(w.B):
        for h in range(w.Hkv):
            kk, vv = wl.cache_slice(w, b, h)
            for host, bits in ((cache.k_host, kk), (cache.v_host, vv)):
                f = torch.from_numpy(wl.bits_to_f32(bits, w.dtype)).to(torch.float8_e4m3fn)
                host[b, h, :w.P] = f.view(torch.uint8).numpy()
    dense = wl.make_dense(w)
    x, wq, wk, wv = (torch.from_numpy(dense[k].view(np.int16)).view(tdt).to(dev)
                     for k in ("x", "wq", "wk", "wv"))
    x = x.reshape(w.B, 1, w.H)
    out = torch.empty((w.B, 1, w.Hq, w.D), dtype=tdt, device=dev)
    lens = np.full(w.B, w.P, np.int32)
    dkv.dkv_cache_kernel_timing(cache.h, True)

    def step():
        cache.set_lengths(lens)
        cache.decode(x, wq, wk, wv, w.Hq, out, stream)
    for _ in range(3):
        step()
    ms, kern = [], []
    for _ in range(max(steps, 5)):
        ms.append(_time_once(torch, stream, flush, step))
        kern.append(dkv.dkv_cache_last_kernel_ms(cache.h))
    cache.free()
    step_ms, kern_ms = statistics.median(ms), statistics.median(kern)
    hb = w.host_read_bytes() // 2  # one byte per element
    gbs = hb / (kern_ms * 1e-3) / 1e9
    return {"workload": w.name, "kv_format": "e4m3", "host_read_bytes": hb, "step_ms": step_ms,
            "tok_s": w.B / (step_ms * 1e-3), "fused_kernel_ms": kern_ms,
            "host_link_gbs": gbs, "frac_of_link": gbs / link_rd}


def bench_paged_decode(w, page_tokens, dkv, torch, dev, stream, flush, link_rd, steps):
    """The decode workload on a paged cache: pages of `page_tokens` rows, each
    sequence's pages drawn by a seeded permutation of the pool (no two
    consecutive logical pages adjacent), the same inputs as the dense run."""
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    npg = -(-w.S_max // page_tokens)
    table = np.random.default_rng(w.seed).permutation(w.B * npg).reshape(w.B, npg)
    table = table.astype(np.int32)
    cache = dkv.PagedKVCache(w.B, w.Hkv, w.D, page_tokens, w.B * npg, npg, w.dtype)
    cache.set_page_table(table)
    full = w.P // page_tokens  # whole pages of prefix; the rest of the last page below
    for b in range(w.B):
        for h in range(w.Hkv):
            kk, vv = wl.cache_slice(w, b, h)
            for pool, rows in ((cache.k_host, kk), (cache.v_host, vv)):
                pool[table[b, :full], h] = rows[:full * page_tokens].reshape(full, page_tokens, w.D)
                tail = w.P - full * page_tokens
                if tail:
                    pool[table[b, full], h, :tail] = rows[full * page_tokens:]
    dense = wl.make_dense(w)
    x, wq, wk, wv = (torch.from_numpy(dense[k].view(np.int16)).view(tdt).to(dev)
                     for k in ("x", "wq", "wk", "wv"))
    x = x.reshape(w.B, 1, w.H)
    out = torch.empty((w.B, 1, w.Hq, w.D), dtype=tdt, device=dev)
    lens = np.full(w.B, w.P, np.int32)
    dkv.dkv_cache_kernel_timing(cache.h, True)

    def step():
        cache.set_lengths(lens)
        cache.decode(x, wq, wk, wv, w.Hq, out, stream)
    for _ in range(3):
        step()
    ms, kern = [], []
    for _ in range(max(steps, 5)):
        ms.append(_time_once(torch, stream, flush, step))
        kern.append(dkv.dkv_cache_last_kernel_ms(cache.h))
    cache.free()
    step_ms, kern_ms = statistics.median(ms), statistics.median(kern)
    gbs = w.host_read_bytes() / (kern_ms * 1e-3) / 1e9
    return {"workload": w.name, "page_tokens": page_tokens, "pages": int(w.B * npg),
            "step_ms": step_ms, "tok_s": w.B / (step_ms * 1e-3), "fused_kernel_ms": kern_ms,
            "host_link_gbs": gbs, "frac_of_link": gbs / link_rd}


def bench_multilayer(dkv, torch, dev, stream, flush, link_rd, steps, layers=32, B=1, P=4096):
    """A whole decode step of a `layers`-layer model with Llama-3-8B attention
    shapes (32/8 heads, D = 128, H = 4096), per-layer caches of B x P tokens
    in one layered pinned allocation, distinct seeded weights per layer:
    per-layer launches against one captured graph per step.  The caches grow
    by one row per step (capacity for every step is allocated)."""
    H, Hq, Hkv, D = 4096, 32, 8, 128
    w = wl.Workload("layer", "decode", B=B, H=H, Hq=Hq, Hkv=Hkv, D=D, P=P)
    total = 2 * (steps + 8) + 2
    cache = dkv.LayeredKVCache(layers, B, Hkv, D, P + total, "bf16")
    for l in range(layers):
        wl_l = w.with_(seed=1000 + l)
        for b in range(B):
            for h in range(Hkv):
                kk, vv = wl.cache_slice(wl_l, b, h)
                cache.k_host[l, b, h, :P] = kk
                cache.v_host[l, b, h, :P] = vv
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    sd = 1.0 / np.sqrt(H)

    def rnd(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * scale).to(torch.bfloat16)
    xs = [rnd(B, 1, H) for _ in range(layers)]
    wqs = [rnd(H, Hq * D, scale=sd) for _ in range(layers)]
    wks = [rnd(H, Hkv * D, scale=sd) for _ in range(layers)]
    wvs = [rnd(H, Hkv * D, scale=sd) for _ in range(layers)]
    outs = [torch.empty((B, 1, Hq, D), dtype=torch.bfloat16, device=dev) for _ in range(layers)]
    cache.set_lengths(np.full(B, P, np.int32))

    def per_layer():
        for l in range(layers):
            cache.decode_layer(l, xs[l], wqs[l], wks[l], wvs[l], Hq, outs[l], stream)
    cache.capture_step(xs, wqs, wks, wvs, Hq, outs)

    def graph():
        cache.launch_step(stream)
    res = {}
    for name, fn in (("per_layer_launches", per_layer), ("graph", graph)):
        for _ in range(3):
            fn()
        res[name] = statistics.median(_time_once(torch, stream, flush, fn)
                                      for _ in range(max(steps, 5)))
    cache.sync(stream)
    cache.free()
    hb = layers * w.host_read_bytes()
    best = min(res.values())
    return {"layers": layers, "B": B, "P": P, "per_layer_host_bytes": w.host_read_bytes(),
            "step_ms_per_layer_launches": res["per_layer_launches"],
            "step_ms_graph": res["graph"], "tok_s_graph": B / (res["graph"] * 1e-3),
            "host_link_gbs_graph": hb / (res["graph"] * 1e-3) / 1e9,
            "frac_of_link_graph": hb / (res["graph"] * 1e-3) / 1e9 / link_rd,
            "best_ms": best}


def _timed_steps(torch, stream, flush, fn, steps, warmup, min_s=0.3, max_steps=2000):
    """`warmup` untimed calls, then at least `steps` timed ones (CUDA events
    on the launching stream, L2 flushed outside the events), continued until
    `min_s` of wall time has passed so that the clock sampler sees the region."""
    for _ in range(max(warmup, 3)):
        flush.zero_()
        fn()
    ms = []
    t0 = time.perf_counter()
    while len(ms) < steps or (time.perf_counter() - t0 < min_s and len(ms) < max_steps):
        ms.append(_time_once(torch, stream, flush, fn))
    return ms


def bench_decode_config(w, dkv, torch, dev, stream, flush, link_rd, steps, warmup, clock_index,
                        baselines=True):
    """One decode workload on its own cache: median step time, the fused
    kernel's time and host-link rate against the link probe, the SM clock
    sampled during the timed steps, and (baselines) the naive untiled
    zero-copy attention, copy-to-HBM-then-attend and separate-kernel times on
    the same cache."""
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    cache = dkv.KVCache(w.B, w.Hkv, w.D, w.S_max, w.dtype)
    wl.fill_cache(w, cache.k_host, cache.v_host)
    dense = wl.make_dense(w)
    x, wq, wk, wv = (torch.from_numpy(dense[k].view(np.int16)).view(tdt).to(dev)
                     for k in ("x", "wq", "wk", "wv"))
    x = x.reshape(w.B, 1, w.H)
    out = torch.empty((w.B, 1, w.Hq, w.D), dtype=tdt, device=dev)
    lens = np.full(w.B, w.P, np.int32)
    dkv.dkv_cache_reserve(cache.h, w.Hq, 1)
    dkv.dkv_cache_kernel_timing(cache.h, True)
    kern = []

    def step():
        cache.set_lengths(lens)
        cache.decode(x, wq, wk, wv, w.Hq, out, stream)
        kern.append(dkv.dkv_cache_last_kernel_ms(cache.h))
    clocks = Clocks(clock_index)
    clocks.start()
    ms = _timed_steps(torch, stream, flush, step, steps, warmup)
    clk = clocks.stop()
    kern_ms = statistics.median(kern[max(warmup, 3):])
    step_ms = statistics.median(ms)
    hb = w.host_read_bytes()
    res = {"B": w.B, "P": w.P, "D": w.D, "Hq": w.Hq, "Hkv": w.Hkv, "dtype": w.dtype,
           "spike_frac": w.spike_frac, "steps_timed": len(ms), "step_ms": step_ms,
           "tok_s": w.B / (step_ms * 1e-3), "fused_kernel_ms": kern_ms,
           "host_link_gbs": hb / (kern_ms * 1e-3) / 1e9,
           "frac_of_link": hb / (kern_ms * 1e-3) / 1e9 / link_rd, "clocks": clk}
    # what launch and completion alone add to an event-timed kernel of the
    # decode's shape (an empty cooperative kernel, one 320-thread CTA with
    # 200 KB of shared memory per SM), and the fraction of the link that
    # a kernel of zero compute time would reach at this cache size
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    floor = statistics.median(_timed_steps(
        torch, stream, flush, lambda: dkv.dkv_probe_launch(sms, 320, 200 * 1024, stream), 50, 5,
        min_s=0.0))
    link_ms = hb / (link_rd * 1e9) * 1e3
    res["launch_floor_ms"] = floor
    res["frac_of_link_ceiling"] = link_ms / (link_ms + floor)
    if baselines:
        q = torch.randn((w.B, w.Hq, w.D), device=dev).to(tdt)
        o2 = torch.empty_like(q)
        cache.set_lengths(lens)
        res["naive_zero_copy_ms"] = min(
            _time_once(torch, stream, flush,
                       lambda: dkv.dkv_attend_naive(cache.h, q, w.Hq, o2, stream))
            for _ in range(3))
        cbytes = w.B * w.Hkv * w.S_max * w.D * 2
        ks = torch.empty(cbytes, dtype=torch.uint8, device=dev)
        vs = torch.empty(cbytes, dtype=torch.uint8, device=dev)

        def staged():
            cache.set_lengths(lens)
            dkv.dkv_decode_staged(cache.h, x, wq, wk, wv, w.H, w.Hq, out, ks, vs, stream)
        res["copy_to_hbm_then_attend_ms"] = min(_time_once(torch, stream, flush, staged)
                                                for _ in range(3))
        del ks, vs

        def unfused():
            cache.set_lengths(lens)
            dkv.dkv_decode_unfused(cache.h, x, wq, wk, wv, w.H, w.Hq, out, stream)
        res["separate_kernels_ms"] = min(_time_once(torch, stream, flush, unfused)
                                         for _ in range(3))
    cache.free()
    return res


def bench_configs(args, dkv, torch, dev, stream, flush, pk, link_rd, link_wr, hbm_rd,
                  clock_index):
    """Every other workload of the benchmark's configuration list, compactly:
    the tiny decode, the long-context sweep (batch 1 and 4 at 16K, 64K and 128K
    cached tokens, 1 % of keys x8) and the fp16 head_dim-64 MHA decode and
    prefill, each with its baselines and its own clock record."""
    res = {}
    for name in ("tiny_decode", "longctx_b1_s16k", "longctx_b1_s64k", "longctx_b1_s128k",
                 "longctx_b4_s16k", "longctx_b4_s64k", "longctx_b4_s128k", "mha_fp16_decode"):
        res[name] = bench_decode_config(wl.WORKLOADS[name], dkv, torch, dev, stream, flush,
                                        link_rd, args.steps, args.warmup, clock_index)
    a2 = argparse.Namespace(**vars(args))
    a2.prefill_workload = "mha_fp16_prefill"
    res["mha_fp16_prefill"] = bench_prefill(a2, dkv, torch, dev, stream, flush, pk, link_rd,
                                            link_wr, hbm_rd, clock_index=clock_index)
    # the Llama-3-8B-shaped chunked prefill on an 8-bit E4M3 cache
    a3 = argparse.Namespace(**vars(args))
    a3.prefill_workload = "llama8b_prefill"
    res["llama8b_prefill_e4m3"] = bench_prefill(a3, dkv, torch, dev, stream, flush, pk, link_rd,
                                                link_wr, hbm_rd, clock_index=clock_index,
                                                kv_format="e4m3")
    return res


def sweep(args, dkv, torch, dev, stream, flush, pk):
    """All workloads, one JSON line each (secondary measurements, not the headline)."""
    # link denominators over a 1 GiB mapped buffer
    probe = dkv.KVCache(1, 8, 128, 262144, "bf16")
    kd, _ = dkv.dkv_cache_device_ptrs(probe.h)
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    nbytes = 8 * 262144 * 128 * 2
    best = min(_time_once(torch, stream, flush,
                          lambda: dkv.dkv_probe_read(kd, nbytes, sink, stream)) for _ in range(3))
    link_rd = nbytes / (best * 1e-3) / 1e9
    probe.free()
    pinned = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    best = min(_time_once(torch, stream, flush,
                          lambda: dkv.dkv_probe_write(pinned.data_ptr(), pinned.numel(), stream))
               for _ in range(3))
    link_wr = pinned.numel() / (best * 1e-3) / 1e9
    hbm = pk.get("hbm_gbs") or 6800.0
    print(json.dumps({"sweep": "link", "zero_copy_read_gbs": link_rd,
                      "zero_copy_write_gbs": link_wr}), flush=True)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clock_index = vis.split(",")[0] if vis else "0"
    for name, w in wl.WORKLOADS.items():
        if w.phase != "decode":
            continue
        res = bench_decode_config(w, dkv, torch, dev, stream, flush, link_rd, args.steps,
                                  args.warmup, clock_index)
        print(json.dumps({"sweep": name, "phase": "decode", **res}), flush=True)
    for name in ("llama8b_decode", "longctx_b1_s128k"):
        res = bench_fp8_decode(wl.WORKLOADS[name], dkv, torch, dev, stream, flush, link_rd,
                               args.steps)
        print(json.dumps({"sweep": name + "_e4m3", "phase": "decode", **res}), flush=True)
    res = bench_multilayer(dkv, torch, dev, stream, flush, link_rd, args.steps)
    print(json.dumps({"sweep": "multilayer_decode_step", "phase": "decode", **res}), flush=True)
    for name in ("llama8b_decode", "longctx_b1_s128k"):
        res = bench_paged_decode(wl.WORKLOADS[name], 16, dkv, torch, dev, stream, flush, link_rd,
                                 args.steps)
        print(json.dumps({"sweep": name + "_paged16", "phase": "decode", **res}), flush=True)
    for name, w in wl.WORKLOADS.items():
        if w.phase != "prefill":
            continue
        a2 = argparse.Namespace(**vars(args))
        a2.prefill_workload = name
        res = bench_prefill(a2, dkv, torch, dev, stream, flush, pk, link_rd, link_wr, hbm)
        print(json.dumps({"sweep": name, "phase": "prefill", **res}), flush=True)


def kernel_source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "zero_copy_offloaded_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(key, files):
    """Per-launch traffic from a committed ncu capture, if it was taken on the
    kernel sources as they are now (else None)."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))[key]
    except (OSError, ValueError, KeyError):
        return None
    return rec if rec.get("src_sha256_16") == kernel_source_hash(files) else None


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:  # no nvidia-smi on this machine
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        lines = open(self.f.name).read().strip().splitlines()
        os.unlink(self.f.name)
        return self.summarize(lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock, max clock and the throttle reasons seen active in
        `nvidia-smi --format=csv,noheader,nounits` lines of the query Q."""
        rows = [r.split(",") for r in lines if r.strip()]
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:  # a partial line (the sampler stopped mid-write)
                continue
            try:
                clk, top = float(r[1]), float(r[2])
            except ValueError:  # a non-numeric sample
                continue
            sm.append(clk)
            mx = max(mx, top)
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# ---------------------------------------------------------------- oracle
def oracle_decode_sample(w: wl.Workload, seqs: int = 1, threads: int = 0):
    """Time the fp64 oracle on `seqs` sequences of the decode workload, on
    `threads` host threads (0: every core in the affinity mask)."""
    import oracle
    oracle.set_threads(threads or host_cores())
    d = wl.make_dense(w.with_(B=seqs))
    k = np.zeros((seqs, w.Hkv, w.S_max, w.D), np.uint16)
    v = np.zeros_like(k)
    wl.fill_cache(w.with_(B=seqs), k, v)
    oracle.lib()
    t0 = time.perf_counter()
    oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    dt = time.perf_counter() - t0
    return dt, oracle.max_threads()


def oracle_prefill_sample(w: wl.Workload, nrows: int = 512, threads: int = 0):
    """Time the fp64 oracle on the prefill workload with a seeded subset of
    query rows (the first and last token of sequence 0 among them): the whole
    projection (every new K/V row is a key of some sampled row), then attention
    of the sampled rows over all heads.  Returns (seconds, threads, algorithmic
    FLOPs of that work, sample description)."""
    import oracle
    oracle.set_threads(threads or host_cores())
    d = wl.make_dense(w)
    k = np.zeros((w.B, w.Hkv, w.S_max, w.D), np.uint16)
    v = np.zeros_like(k)
    wl.fill_cache(w, k, v)
    rng = np.random.default_rng(0)
    extra = max(0, min(nrows, w.T) - 2)
    ts = sorted({0, w.T - 1} | set(int(t) for t in rng.choice(w.T, extra, replace=False)))
    rows = [(0, t) for t in ts]
    oracle.lib()
    t0 = time.perf_counter()
    oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype, rows=rows)
    dt = time.perf_counter() - t0
    flops = w.proj_flops() + sum(4 * w.Hq * w.D * (w.P + t + 1) for _, t in rows)
    sample = (f"{w.name}: the whole projection ({w.B * w.T} tokens) and {len(rows)} seeded "
              f"query rows of sequence 0 (all {w.Hq} heads)")
    return dt, oracle.max_threads(), flops, sample


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    seqs = 1
    times = []
    for i in range(args.warmup + args.steps):
        dt, cores = oracle_decode_sample(w, seqs)
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = seqs * len(times) / tot
    line = {
        "impl": "reference", "metric": "fused KV-proj+attn decode tok/s", "value": value,
        "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "P": w.P, "H": w.H, "Hq": w.Hq, "Hkv": w.Hkv,
                   "D": w.D, "kv_dtype": w.dtype},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": f"{seqs} of {w.B} sequences per step (all heads, P={w.P})"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import zero_copy_offloaded_gb300 as dkv

    from zero_copy_offloaded_gb300 import ranks as rk

    rks = rk.Ranks.from_env()
    world, rank, local = rks.world, rks.rank, rks.local
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    def barrier():
        rk.barrier(dist)
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return rk.max_over_ranks(v, dist, dev)

    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if args.sweep:
        return sweep(args, dkv, torch, dev, stream, flush, pk)
    if args.profile_prefill:
        w = wl.WORKLOADS[args.prefill_workload]
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        cache = dkv.KVCache(w.B, w.Hkv, w.D, w.S_max, w.dtype)
        wl.fill_cache(w, cache.k_host, cache.v_host)
        dense = wl.make_dense(w)
        x, wq, wk, wv = (torch.from_numpy(dense[k].view(np.int16)).view(tdt).to(dev)
                         for k in ("x", "wq", "wk", "wv"))
        out = torch.empty((w.B, w.T, w.Hq, w.D), dtype=tdt, device=dev)
        lens = np.full(w.B, w.P, np.int32)
        for i in range(3):
            cache.set_lengths(lens)
            cache.prefill(x, wq, wk, wv, w.Hq, out, stream)
        cache.set_lengths(lens)
        dkv.dkv_prefill_naive(cache.h, x, w.T, wq, wk, wv, w.H, w.Hq, out, stream)
        cache.sync(stream)
        cache.free()
        return
    if args.prefill_only:
        # prefill alone (profiling aid): link/HBM rates from the probes, then the prefill
        probe_cache = dkv.KVCache(1, 8, 128, 65536, "bf16")
        kd, _ = dkv.dkv_cache_device_ptrs(probe_cache.h)
        sink = torch.zeros(4, dtype=torch.int32, device=dev)
        nbytes = 8 * 65536 * 128 * 2
        best = min(_time_once(torch, stream, flush,
                              lambda: dkv.dkv_probe_read(kd, nbytes, sink, stream)) for _ in range(3))
        link_rd = nbytes / (best * 1e-3) / 1e9
        probe_cache.free()
        res = bench_prefill(args, dkv, torch, dev, stream, flush, pk, link_rd, link_rd * 0.9,
                            pk.get("hbm_gbs") or 6800.0)
        if rank == 0:
            print(json.dumps({"prefill": res, "link_read_gbs": link_rd}), flush=True)
        return
    w = wl.WORKLOADS[args.workload]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16

    def dev_tensor(bits):
        return torch.from_numpy(bits.view(np.int16)).view(tdt).to(dev)

    # ------------------------------------------------ decode workload setup
    cache = dkv.KVCache(w.B, w.Hkv, w.D, w.S_max, w.dtype)
    wl.fill_cache(w, cache.k_host, cache.v_host)
    dense = wl.make_dense(w)
    x, wq, wk, wv = (dev_tensor(dense[k]) for k in ("x", "wq", "wk", "wv"))
    x = x.reshape(w.B, 1, w.H)
    out = torch.empty((w.B, 1, w.Hq, w.D), dtype=tdt, device=dev)
    lens = np.full(w.B, w.P, np.int32)
    dkv.dkv_cache_reserve(cache.h, w.Hq, 1)
    dkv.dkv_cache_kernel_timing(cache.h, True)

    def step():
        cache.set_lengths(lens)
        cache.decode(x, wq, wk, wv, w.Hq, out, stream)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    cache.sync(stream)

    # ------------------------------------------------ timed decode
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    clocks = Clocks(vis.split(",")[local] if vis else str(local))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    kern_ms = []
    launches = 0
    barrier()
    clocks.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # L2 flush outside the timed events
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        launches += dkv.dkv_last_launch_count()
        kern_ms.append(dkv.dkv_cache_last_kernel_ms(cache.h))
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    cache.sync(stream)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    tot_s = max_over_ranks(sum(step_ms) / 1e3)
    value = rk.job_rate(w.B * args.steps, world, tot_s)
    fused_ms = statistics.mean(kern_ms)

    # ------------------------------------------------ link / HBM probes
    kd, vd = dkv.dkv_cache_device_ptrs(cache.h)
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    cache_bytes = w.B * w.Hkv * w.S_max * w.D * 2  # one of K / V

    def time_kernel(fn, reps=5):
        best = 1e30
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    link_rd_ms = time_kernel(lambda: dkv.dkv_probe_read(kd, cache_bytes, sink, stream))
    link_rd = cache_bytes / (link_rd_ms * 1e-3) / 1e9
    pinned = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    link_wr_ms = time_kernel(lambda: dkv.dkv_probe_write(pinned.data_ptr(), pinned.numel(), stream))
    link_wr = pinned.numel() / (link_wr_ms * 1e-3) / 1e9
    hbm_buf = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    hbm_ms = time_kernel(lambda: dkv.dkv_probe_read(hbm_buf, hbm_buf.numel(), sink, stream))
    hbm_rd = hbm_buf.numel() / (hbm_ms * 1e-3) / 1e9
    del hbm_buf
    dst = torch.empty(pinned.numel(), dtype=torch.uint8, device=dev)
    h2d_ms = time_kernel(lambda: dst.copy_(pinned, non_blocking=True))
    h2d = pinned.numel() / (h2d_ms * 1e-3) / 1e9
    del dst

    host_bytes = w.host_read_bytes()
    achieved = host_bytes / (fused_ms * 1e-3) / 1e9
    tr = ncu_traffic(f"decode_fused_kernel/{w.name}", ["decode.cu", "dkv_internal.cuh"])
    roofline = {"bound": "host_link", "achieved": achieved, "peak": link_rd, "unit": "GB/s",
                "frac": achieved / link_rd,
                # host-link bytes (sysmem sectors x 32 B) of one launch from ncu; HBM bytes beside
                "traffic": tr["host_link_bytes"] if tr else None,
                "traffic_dram": tr["dram_bytes"] if tr else None,
                "peak_source": "zero-copy streaming read probe over the same cache, same run",
                "kernel": "decode_fused_kernel", "kernel_ms": fused_ms,
                "algorithmic_bytes_per_launch": host_bytes}

    # ------------------------------------------------ e2e through the C ABI with host buffers
    x_host = torch.from_numpy(dense["x"].view(np.int16)).view(tdt).reshape(w.B, 1, w.H).pin_memory()
    out_host = torch.empty(out.shape, dtype=tdt, pin_memory=True)
    x_dev = torch.empty_like(x)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        cache.set_lengths(lens)
        cache.decode(x_dev, wq, wk, wv, w.Hq, out, stream)
        out_host.copy_(out, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_val = rk.job_rate(w.B * len(e2e_ms), world, max_over_ranks(sum(e2e_ms) / 1e3))

    extras = {}
    if not args.no_extras:
        # naive untiled zero-copy attention and copy-to-HBM-then-attend, same cache
        q = torch.randn((w.B, w.Hq, w.D), device=dev).to(tdt)
        o2 = torch.empty_like(q)
        cache.set_lengths(lens)
        naive_ms = time_kernel(lambda: dkv.dkv_attend_naive(cache.h, q, w.Hq, o2, stream), reps=3)
        ks = torch.empty(cache_bytes, dtype=torch.uint8, device=dev)
        vs = torch.empty(cache_bytes, dtype=torch.uint8, device=dev)

        def staged():
            cache.set_lengths(lens)
            dkv.dkv_decode_staged(cache.h, x, wq, wk, wv, w.H, w.Hq, out, ks, vs, stream)
        staged_ms = time_kernel(staged, reps=3)
        del ks, vs

        def unfused():
            cache.set_lengths(lens)
            dkv.dkv_decode_unfused(cache.h, x, wq, wk, wv, w.H, w.Hq, out, stream)
        unfused_ms = time_kernel(unfused, reps=3)
        extras["baselines"] = {
            "fused_zero_copy_step_ms": statistics.mean(step_ms),
            "naive_zero_copy_attention_ms": naive_ms,
            "copy_to_hbm_then_attend_ms": staged_ms,
            "separate_kernels_ms": unfused_ms,
            "hbm_staging_bytes": 2 * cache_bytes,
        }
        clock_index = vis.split(",")[local] if vis else str(local)
        extras["prefill"] = bench_prefill(args, dkv, torch, dev, stream, flush, pk, link_rd,
                                          link_wr, hbm_rd, clock_index=clock_index)
    cache.free()
    if not args.no_extras:
        # the same decode on a paged cache (16-token pages, shuffled page table)
        extras["paged_decode"] = bench_paged_decode(w, 16, dkv, torch, dev, stream, flush,
                                                    link_rd, args.steps)
        # the same decode on an 8-bit E4M3 cache (half the host bytes)
        extras["fp8_decode"] = bench_fp8_decode(w, dkv, torch, dev, stream, flush, link_rd,
                                                args.steps)
        # a 32-layer step of small per-layer caches: launches per layer vs one graph
        extras["multilayer_decode_step"] = bench_multilayer(dkv, torch, dev, stream, flush,
                                                            link_rd, args.steps)
        # every other configuration, compactly, each with its baselines and clocks
        extras["configs"] = bench_configs(args, dkv, torch, dev, stream, flush, pk, link_rd,
                                          link_wr, hbm_rd, clock_index)

    cpu = None
    if rank == 0 and not args.no_extras:
        dt, cores = oracle_decode_sample(w, 1)
        cpu = {"value": 1.0 / dt, "unit": "tok/s", "cores": cores, "kind": "oracle",
               "sample": f"1 of {w.B} sequences (all {w.Hq} heads, P={w.P}), one step"}
        # beside it, the same oracle on the tiny decode workload on every core and on one
        tw = wl.WORKLOADS["tiny_decode"]
        t_all, _ = min(oracle_decode_sample(tw) for _ in range(3))
        t_one, _ = min(oracle_decode_sample(tw, threads=1) for _ in range(3))
        cpu["tiny_decode"] = {"tok_s_all_cores": 1.0 / t_all, "tok_s_one_core": 1.0 / t_one}
        # and on the prefill workload, a bounded sample in the prefill's unit
        pdt, pcores, pflops, psample = oracle_prefill_sample(wl.WORKLOADS[args.prefill_workload])
        cpu["prefill"] = {"value": pflops / pdt / 1e12, "unit": "TFLOP/s", "cores": pcores,
                          "kind": "oracle", "seconds": pdt, "sample": psample}

    if rank == 0:
        line = {
            "metric": "fused KV-proj+attn decode tok/s", "value": value, "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "P": w.P, "H": w.H, "Hq": w.Hq,
                       "Hkv": w.Hkv, "D": w.D, "kv_cache": "pinned mapped host memory",
                       "l2": "flushed between steps (256 MiB write outside the timed events)",
                       "parallelism": f"replicas{world}"},
            "host_link_gbs": host_bytes / (statistics.mean(step_ms) * 1e-3) / 1e9,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "tok/s",
                    "h2d_bytes_per_step": int(x_host.numel() * 2),
                    "d2h_bytes_per_step": int(out_host.numel() * 2)},
            "gpu_launches": launches,
            "clocks": clk,
            "link": {"zero_copy_read_gbs": link_rd, "zero_copy_write_gbs": link_wr,
                     "memcpy_h2d_gbs": h2d, "hbm_read_gbs": hbm_rd,
                     "hbm_measured_peak_gbs": pk.get("hbm_gbs")},
            "wall_s_timed": wall,
            **extras,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _time_once(torch, stream, flush, fn):
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b)


def prefill_partial_rows(w, chunk=256):
    """Rows of per-chunk partials the fused prefill writes (and the combine
    reads): for every sequence, KV-stationary chunk and query head, the new
    tokens that see the chunk (causal: token t sees keys 0..P+t)."""
    rows = 0
    for _ in range(w.B):
        for k0 in range(0, w.P + w.T, chunk):
            rows += w.T - max(0, k0 - w.P)
    return rows * w.Hq


def bench_prefill(args, dkv, torch, dev, stream, flush, pk, link_rd, link_wr, hbm_rd,
                  clock_index=None, naive_max_ms=400.0, kv_format="native"):
    """One prefill workload: the whole call (Q projection + fused kernel +
    combine) timed over `steps` calls after `warmup` (median; lengths reset
    before each so every call appends at the same position), the fused
    kernel's own time, the SM clock during the timed calls, TFLOP/s against
    the min-of-rooflines bound, and two baselines on the same inputs:
    copy-to-HBM-then-prefill and the naive untiled zero-copy prefill (every
    (Q tile, chunk) pair fetching its chunk across the link; timed only if one
    call stays under `naive_max_ms`).  kv_format "e4m3": the same workload on an
    8-bit E4M3 cache (the values converted with torch's float8 type as input
    construction), half the host bytes; the baselines are 16-bit only."""
    w = wl.WORKLOADS[args.prefill_workload]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    fp8 = kv_format == "e4m3"
    cache = dkv.KVCache(w.B, w.Hkv, w.D, w.S_max, w.dtype, kv_format=kv_format)
    if fp8:
        for b in range(w.B):
            for h in range(w.Hkv):
                kk, vv = wl.cache_slice(w, b, h)
                for host, bits in ((cache.k_host, kk), (cache.v_host, vv)):
                    f = torch.from_numpy(wl.bits_to_f32(bits, w.dtype)).to(torch.float8_e4m3fn)
                    host[b, h, :w.P] = f.view(torch.uint8).numpy()
    else:
        wl.fill_cache(w, cache.k_host, cache.v_host)
    dense = wl.make_dense(w)
    x, wq, wk, wv = (torch.from_numpy(dense[k].view(np.int16)).view(tdt).to(dev)
                     for k in ("x", "wq", "wk", "wv"))
    out = torch.empty((w.B, w.T, w.Hq, w.D), dtype=tdt, device=dev)
    lens = np.full(w.B, w.P, np.int32)
    dkv.dkv_cache_reserve(cache.h, w.Hq, w.T)

    def call():
        cache.set_lengths(lens)
        cache.prefill(x, wq, wk, wv, w.Hq, out, stream)
    # whole calls without the library's per-kernel events, which would sit
    # between the launches and keep them from overlapping
    dkv.dkv_cache_kernel_timing(cache.h, False)
    clocks = Clocks(clock_index) if clock_index is not None else None
    if clocks:
        clocks.start()
    times = _timed_steps(torch, stream, flush, call, max(args.steps, 10), args.warmup)
    clk = clocks.stop() if clocks else None
    cache.sync(stream)
    # then the fused kernel's own time, from calls with those events on
    dkv.dkv_cache_kernel_timing(cache.h, True)
    kern = []
    for _ in range(max(args.steps, 10)):
        _time_once(torch, stream, flush, call)
        kern.append(dkv.dkv_cache_last_kernel_ms(cache.h))
    dkv.dkv_cache_kernel_timing(cache.h, False)
    cache.sync(stream)

    def naive():
        cache.set_lengths(lens)
        dkv.dkv_prefill_naive(cache.h, x, w.T, wq, wk, wv, w.H, w.Hq, out, stream)
    naive_ms = staged_ms = None
    nstage = w.B * w.Hkv * w.S_max * w.D
    if not fp8:
        naive_ms = _time_once(torch, stream, flush, naive)   # first call: also the size check
        if naive_ms <= naive_max_ms:
            naive_ms = min([naive_ms] + [_time_once(torch, stream, flush, naive)
                                         for _ in range(2)])
        cache.sync(stream)
        # baseline: copy the cached prefix to HBM, then the same fused prefill from there
        k_stage = torch.empty(nstage, dtype=tdt, device=dev)
        v_stage = torch.empty(nstage, dtype=tdt, device=dev)

        def staged():
            cache.set_lengths(lens)
            dkv.dkv_prefill_staged(cache.h, x, w.T, wq, wk, wv, w.H, w.Hq, out, k_stage,
                                   v_stage, stream)
        staged_ms = statistics.median(_timed_steps(torch, stream, flush, staged, 5, 2, min_s=0))
        cache.sync(stream)
        del k_stage, v_stage
    info = dkv.dkv_cache_info(cache.h)
    cache.free()
    ms = statistics.median(times)
    files = ["prefill_tc.cu", "dkv_internal.cuh", "tc_common.cuh"]
    tr = None if fp8 else ncu_traffic(f"prefill_tc_kernel/{w.name}", files)
    tr_source = "ncu capture of this workload" if tr else None
    if tr is None and not fp8 and w.name == "llama8b_prefill":
        # captures stay small: the quarter-size case, scaled by the partial rows
        # (the fused kernel's writes and the combine's reads are the chunks'
        # partials; its reads are the Q tiles that each chunk takes again)
        q = ncu_traffic("prefill_tc_kernel/llama8b_prefill_quarter", files)
        if q:
            f = prefill_partial_rows(w) / prefill_partial_rows(
                wl.WORKLOADS["llama8b_prefill_quarter"])
            tr = {k: int(v * f) for k, v in q.items() if k.endswith("bytes")}
            tr_source = f"quarter-size capture scaled by the partial rows ({f:.2f}x)"
    flops = w.flops()
    tflops_peak = pk.get("bf16_tflops") or 1900.0
    hb_rd = w.host_read_bytes() // (2 if fp8 else 1)
    hb_wr = w.host_write_bytes() // (2 if fp8 else 1)
    t_link_rd = hb_rd / (link_rd * 1e9)
    t_link_wr = hb_wr / (link_wr * 1e9)
    t_hbm = w.hbm_min_bytes() / (hbm_rd * 1e9)
    t_flop = flops / (tflops_peak * 1e12)
    t_roof = max(t_link_rd, t_link_wr, t_hbm, t_flop)
    dram = (tr["dram_bytes"] + tr["combine_dram_read_bytes"] + tr["combine_dram_write_bytes"]
            if tr else None)
    return {"workload": w.name, "kv_format": kv_format, "host_read_bytes": hb_rd,
            "host_write_bytes": hb_wr, "ms": ms, "calls_timed": len(times),
            "fused_kernel_ms": statistics.median(kern),
            "tflops": flops / (ms * 1e-3) / 1e12, "flops": flops,
            "roofline_ms": t_roof * 1e3,
            "roofline_terms_ms": {"link_read": t_link_rd * 1e3, "link_write": t_link_wr * 1e3,
                                  "hbm": t_hbm * 1e3, "tensor": t_flop * 1e3},
            "frac_of_roofline": t_roof / (ms * 1e-3),
            "clocks": clk,
            "copy_to_hbm_then_prefill_ms": staged_ms,
            "naive_zero_copy_ms": naive_ms if naive_ms and naive_ms <= naive_max_ms else None,
            "naive_zero_copy_first_call_ms": naive_ms,
            # DRAM bytes of one fused launch and of the combine, from a committed ncu
            # capture of the current sources (None once they change), and the whole
            # call's DRAM bytes over the algorithmic HBM minimum
            "traffic_dram": tr["dram_bytes"] if tr else None,
            "traffic_dram_combine": (tr["combine_dram_read_bytes"] + tr["combine_dram_write_bytes"]
                                     if tr else None),
            "hbm_min_bytes": w.hbm_min_bytes(),
            "traffic_dram_over_hbm_min": dram / w.hbm_min_bytes() if dram else None,
            "traffic_source": tr_source,
            "partial_rows": prefill_partial_rows(w),
            "hbm_staging_bytes": None if fp8 else 2 * nstage * 2,
            "tensor_peak_tflops": tflops_peak,
            "device_workspace_bytes": info["device_workspace_bytes"]}


if __name__ == "__main__":
    main()
