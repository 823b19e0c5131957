"""Prefill parity: Q projection + fused KV-stationary prefill + combine
(through the C ABI) against the fp64 oracle on the same seeded inputs.

Bars: appended K/V rows within 1 ulp of the oracle's fp32-sequential
projection rounded to the dtype (the fused projection runs on the tensor
cores, whose summation order differs), or within the fp32 summation error
bound where the sum nearly cancels; attention output max-abs <= 1e-2 and
sum|err|/sum|ref| <= 2e-3 versus fp64; prefix rows and rows past the append
untouched."""
import numpy as np
import pytest

import zero_copy_offloaded_gb300 as dkv
from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import (Case, torch_dtype, assert_close, assert_close_beyond_rounding, assert_projection_close,
                      out_f64)

pytestmark = pytest.mark.gpu


def check_prefill(case: Case, out, ref, label="", rows=None, beyond_rounding=False):
    w = case.w
    T = out.shape[1]
    got = out_f64(out, w.dtype).reshape(w.B, T, w.Hq, w.D)
    if beyond_rounding:
        res = assert_close_beyond_rounding(got, ref["out"], w.dtype, label)
    elif rows is None:
        res = assert_close(got, ref["out"], label)
    else:
        g = np.stack([got[b, t] for (b, t) in rows])
        r = np.stack([ref["out"][(b, t)] for (b, t) in rows])
        res = assert_close(g, r, label)
    check_appends(case, T, label)
    return res


def check_appends(case: Case, T, label=""):
    """Appended rows against the oracle's projection (1 ulp or the fp32
    bound), prefix rows unchanged, rows past the append untouched."""
    w = case.w
    kh, vh = case.k_logical(), case.v_logical()
    x = case.dense["x"]
    for b in range(w.B):
        p = int(case.lens[b])
        for name, host, wmat in (("k", kh, case.dense["wk"]), ("v", vh, case.dense["wv"])):
            got = host[b, :, p:p + T].transpose(1, 0, 2).reshape(T, w.Hkv * w.D)
            assert_projection_close(got, x[b], wmat, w.dtype, f"{label} {name} append b={b}")
        assert np.array_equal(kh[b, :, :p], case.k0[b, :, :p])
        assert np.array_equal(vh[b, :, :p], case.v0[b, :, :p])
        assert np.all(kh[b, :, p + T:] == case.canary) and np.all(vh[b, :, p + T:] == case.canary)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 2), (64, 4, 4), (128, 8, 1), (64, 16, 2)])
@pytest.mark.parametrize("P,T", [(0, 1), (0, 37), (5, 300), (300, 17), (600, 129)])
def test_prefill_shapes(dtype, D, Hq, Hkv, P, T):
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=Hq, Hkv=Hkv, D=D, P=P, T=T, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=P + T)
    case = Case(w, s_max=P + T + 3)
    try:
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(), f"{dtype} D{D} G{Hq // Hkv} P{P} T{T}")
    finally:
        case.free()


def _late_max_fraction(ref, K, w, nchunks):
    """Fraction of (query row, prefix chunk) pairs whose scores past the
    chunk's first 64 keys exceed the max of those 64 by more than 2^15 in
    weight (computed from the oracle's q, in fp64).  Each such pair makes the
    fused kernel rescale the weights it has already written (it does so once a
    64-key piece's weights sum to more than 2^14), so this is a lower bound on
    how often the rescale runs."""
    q = wl.bits_to_f32(ref["q"], w.dtype).astype(np.float64)  # [B,T,Hq,D]
    G = w.Hq // w.Hkv
    hits = total = 0
    for b in range(w.B):
        for h in range(w.Hq):
            s = q[b, :, h] @ K[b, h // G, :nchunks * 256].T / np.sqrt(w.D) * np.log2(np.e)
            for c in range(nchunks):  # chunks wholly in the prefix: every query sees them
                m0 = s[:, c * 256:c * 256 + 64].max(axis=1)
                m1 = s[:, c * 256 + 64:c * 256 + 256].max(axis=1)
                hits += int(np.sum(m1 > m0 + 15))
                total += m0.size
    return hits / total


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_prefill_spiky_keys(dtype):
    """5 % of the cached key rows scaled by 8 (the long-context recipe, denser):
    attention concentrates on few keys, and the outputs on single value rows."""
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=700, T=90, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", spike_frac=0.05,
                    seed=11)
    case = Case(w, s_max=w.P + w.T + 3)
    try:
        out = case.run_prefill()
        ref = case.oracle()
        # attention concentrates on single value rows, so outputs reach |o| >= 4
        # where bf16's own rounding exceeds the flat max-abs bar
        check_prefill(case, out, ref, f"spiky {dtype}", beyond_rounding=True)
    finally:
        case.free()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_prefill_late_key_spikes(dtype):
    """The key at offset 200 of every 256-key chunk scaled by 40.

    The fused kernel forms a row's weights against the max of the chunk's
    first 64 scores and, when a later 64-key piece's weights sum to more than
    2^14, rescales the weights it has written and continues against that
    piece's max.  Here that happens for a known share of the rows (bounded
    below from the oracle's q), and the outputs are compared with the oracle
    as everywhere else."""
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=768, T=64, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=23)
    case = Case(w, s_max=w.P + w.T + 3)
    try:
        kf = wl.bits_to_f32(case.k0, dtype)
        rows = np.arange(200, w.P, 256)
        kf[:, :, rows] *= np.float32(40.0)
        case.k0[:, :, rows] = wl.to_bits(kf[:, :, rows], dtype)
        case.cache.k_host[...] = case.k0
        out = case.run_prefill()
        ref = case.oracle()
        K = wl.bits_to_f32(case.k0, dtype).astype(np.float64)
        frac = _late_max_fraction(ref, K, w, w.P // 256)
        assert frac > 0.1, f"the rescale is taken by only {frac:.3f} of the rows"
        check_prefill(case, out, ref, f"late spikes {dtype}", beyond_rounding=True)
    finally:
        case.free()


def test_prefill_max_batch():
    """64 sequences (the largest batch), ragged prefixes including 0, T crossing a chunk."""
    w = wl.Workload("t", "prefill", B=64, H=64, Hq=4, Hkv=2, D=64, P=300, T=20, seed=65)
    lens = [(13 * b) % 301 for b in range(64)]
    case = Case(w, lens=lens, s_max=330)
    try:
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(), "prefill B=64")
        assert list(case.cache.lengths()) == [n + 20 for n in lens]
    finally:
        case.free()


def test_prefill_ragged_lengths():
    w = wl.Workload("t", "prefill", B=3, H=64, Hq=8, Hkv=2, D=128, P=520, T=40, seed=4)
    case = Case(w, lens=[0, 520, 257], s_max=600)
    try:
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(), "ragged")
        assert list(case.cache.lengths()) == [40, 560, 297]
    finally:
        case.free()


def test_prefill_then_decode_matches_oracle():
    w = wl.Workload("t", "prefill", B=1, H=128, Hq=8, Hkv=2, D=64, P=100, T=64, seed=8)
    case = Case(w, s_max=200)
    try:
        out = case.run_prefill()
        ref = case.oracle()
        check_prefill(case, out, ref, "prefill")
        from .helpers import to_dev
        x2 = wl.make_dense(w.with_(T=1, seed=99))["x"]
        out2 = case.run_decode(to_dev(x2, w.dtype))
        ref2 = case.oracle(x_bits=x2, k=ref["k_cache_after"], v=ref["v_cache_after"],
                           lens=case.lens + w.T)
        got = out_f64(out2, w.dtype).reshape(w.B, w.Hq, w.D)
        assert_close(got, ref2["out"].reshape(w.B, w.Hq, w.D), "decode after prefill")
    finally:
        case.free()


def test_prefill_staged_baseline():
    """The copy-to-HBM baseline: the cached prefix is copied into HBM buffers
    and the same fused prefill reads it from there.  Against the oracle as
    every prefill, and bit-identical to the zero-copy prefill of the same
    inputs (the same kernel over the same values); refusals for a missing
    staging buffer and a paged cache."""
    import torch
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=300, T=70, seed=37)
    case = Case(w, lens=[300, 45], s_max=380)
    try:
        n = w.B * w.Hkv * case.s_max * w.D
        k_stage = torch.zeros(n, dtype=torch_dtype(w.dtype), device="cuda")
        v_stage = torch.zeros_like(k_stage)
        out_s = case.out_tensor(w.T)
        dkv.dkv_prefill_staged(case.cache.h, case.x, w.T, case.wq, case.wk, case.wv, w.H, w.Hq,
                               out_s, k_stage, v_stage, None)
        case.cache.sync()
        ref = case.oracle()
        check_prefill(case, out_s, ref, "staged prefill")
        # the zero-copy prefill on the same caches (reset) gives the same bits
        case.cache.k_host[...] = case.k0
        case.cache.v_host[...] = case.v0
        case.cache.set_lengths(case.lens.astype(np.int32))
        out_z = case.run_prefill()
        assert torch.equal(out_s.view(torch.int16), out_z.view(torch.int16))
        case.cache.set_lengths(case.lens.astype(np.int32))  # room for T more rows
        with pytest.raises(dkv.DkvError) as ei:
            dkv.dkv_prefill_staged(case.cache.h, case.x, w.T, case.wq, case.wk, case.wv, w.H,
                                   w.Hq, out_s, None, v_stage, None)
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
    finally:
        case.free()
    pw = wl.Workload("t", "prefill", B=1, H=128, Hq=8, Hkv=2, D=64, P=20, T=8, seed=3)
    pc = Case(pw, s_max=32, page_tokens=16)
    try:
        st = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(dkv.DkvError) as ei:
            dkv.dkv_prefill_staged(pc.cache.h, pc.x, pw.T, pc.wq, pc.wk, pc.wv, pw.H, pw.Hq,
                                   pc.out_tensor(pw.T), st, st, None)
        assert ei.value.name == "DKV_ERR_UNSUPPORTED"
    finally:
        pc.free()


def _edge_and_random_rows(w, n_per_seq, seed):
    """Query rows (b, t) for a sampled full-size check: for every sequence the
    first and last token, the first and last token of every 256-key chunk that
    holds new tokens (where the fused projection, the append and the causal
    diagonal meet), then seeded random tokens up to n_per_seq rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        ts = {0, w.T - 1}
        for k0 in range(w.P // 256 * 256, w.P + w.T, 256):   # chunks with new keys
            ts.add(max(0, k0 - w.P))
            ts.add(min(w.T - 1, k0 + 255 - w.P))
        while len(ts) < n_per_seq:
            ts.add(int(rng.integers(0, w.T)))
        rows += [(b, t) for t in sorted(ts)]
    return rows


@pytest.mark.slow
def test_prefill_mha_fp16_full_size():
    """fp16 MHA prefill workload at full size (B=2, T=2048 over P=6144): 512
    query rows per sequence against the oracle, every appended row checked."""
    w = wl.WORKLOADS["mha_fp16_prefill"]
    case = Case(w)
    try:
        out = case.run_prefill()
        rows = _edge_and_random_rows(w, 512, seed=0)
        assert len(rows) == 2 * 512
        check_prefill(case, out, case.oracle(rows=rows), "mha_fp16_prefill", rows=rows)
    finally:
        case.free()


@pytest.mark.slow
def test_prefill_llama8b_full_size_sampled_rows():
    """Llama-3-8B-shaped chunked prefill at full size (T=4096 over P=28672),
    in the launch configuration the benchmark times: every appended row is
    checked, attention on 512 seeded query rows including the first and last
    token of each of the 16 chunks that hold new tokens."""
    w = wl.WORKLOADS["llama8b_prefill"]
    case = Case(w)
    try:
        out = case.run_prefill()
        rows = _edge_and_random_rows(w, 512, seed=0)
        assert len(rows) == 512
        for i in range(16):
            assert (0, 256 * i) in rows and (0, 256 * i + 255) in rows
        check_prefill(case, out, case.oracle(rows=rows), "llama8b_prefill", rows=rows)
    finally:
        case.free()


@pytest.mark.parametrize("dtype,D,page_tokens", [("bf16", 64, 0), ("fp16", 128, 0),
                                                 ("bf16", 128, 16)])
def test_prefill_long_units_split_last_wave(dtype, D, page_tokens):
    """64 Q tiles per chunk (T = 2048, G = 4) with ragged prefixes: the units
    holding new tokens fit in one wave and run first, and the prefix units
    (fewer than one wave here) all run as two CTAs each, one per half of the
    chunk's Q tiles; dense and paged caches.  Every output row and appended
    row against the oracle."""
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=D, P=1024, T=2048, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=77 + page_tokens)
    case = Case(w, lens=[1024, 300], s_max=1024 + 2048 + 3, page_tokens=page_tokens)
    try:
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(),
                      f"long units, split last wave {dtype} D={D} pages={page_tokens}")
    finally:
        case.free()


def test_prefill_bf16_value_chunk_scale():
    """bf16 V beyond fp16's range.  The fused kernel runs P.V in fp16, so a
    stationary V chunk whose max |V| reaches 2^15 is converted times 2^-k
    (k > 0) and the combine multiplies that chunk's partial by 2^k.  Here
    chunk 0 holds V x 2^20, chunk 1 plain V (k = 0), chunk 2 mixes rows
    x 2^20 with rows x 2^-10 (the small ones land near fp16's subnormals after
    the scaling), chunk 3 holds V x 2^15 (the threshold), and the new tokens'
    rows are projected.  Attention is linear in V, so the max-abs bar applies
    to the error in units of the row's own value scale: |err| minus the
    output's own rounding <= 1e-2 * max(1, sum_j w_j |v_j|), with the weights
    w_j and the absolute-value attention taken from the oracle; the mean
    relative bar is unchanged."""
    import oracle
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=1100, T=90, dtype="bf16",
                    seed=41)
    case = Case(w, s_max=w.P + w.T + 3)
    try:
        vf = wl.bits_to_f32(case.v0, "bf16").astype(np.float64)
        scale = np.ones(case.s_max)
        scale[0:256] = 2.0 ** 20
        scale[512:768:2] = 2.0 ** 20
        scale[513:768:2] = 2.0 ** -10
        scale[768:1024] = 2.0 ** 15
        vf[:, :, :w.P] *= scale[None, None, :w.P, None]
        case.v0[:, :, :w.P] = oracle.round_bits(vf[:, :, :w.P], "bf16")
        case.cache.v_host[...] = case.v0
        out = case.run_prefill()
        ref = case.oracle()
        got = out_f64(out, "bf16").reshape(w.B, w.T, w.Hq, w.D)
        # sum_j w_j |v_j| per output element, from the oracle's attention of |V|
        G = w.Hq // w.Hkv
        ref_abs = np.zeros_like(ref["out"])
        for b in range(w.B):
            p = int(case.lens[b])
            for kvh in range(w.Hkv):
                kf = oracle.decode_bits(ref["k_cache_after"][b, kvh, :p + w.T], "bf16")
                va = np.abs(oracle.decode_bits(ref["v_cache_after"][b, kvh, :p + w.T], "bf16"))
                q = oracle.decode_bits(ref["q"][b, :, kvh * G:(kvh + 1) * G], "bf16")
                pos = np.repeat(p + np.arange(w.T), G)
                ref_abs[b, :, kvh * G:(kvh + 1) * G] = oracle.attend(
                    kf, va, q.reshape(-1, w.D), pos).reshape(w.T, G, w.D)
        rounded = oracle.decode_bits(oracle.round_bits(ref["out"], "bf16"), "bf16")
        excess = np.abs(got - ref["out"]) - np.abs(rounded - ref["out"])
        assert np.all(excess <= 1e-2 * np.maximum(1.0, ref_abs)), float(
            np.max(excess / np.maximum(1.0, ref_abs)))
        mr = np.abs(got - ref["out"]).sum() / np.abs(ref["out"]).sum()
        assert mr <= 2e-3, mr
        assert ref_abs.max() > 2.0 ** 17  # the scaled chunks carry real weight
        check_appends(case, w.T, "V chunk scale")
    finally:
        case.free()


@pytest.mark.parametrize("dtype,D,Hq,Hkv,P,T", [("bf16", 128, 8, 2, 600, 129),
                                               ("fp16", 64, 8, 8, 300, 70)])
def test_prefill_naive_baseline(dtype, D, Hq, Hkv, P, T):
    """The naive untiled baseline (one CTA per Q tile and chunk, every pair
    fetching its chunk from the host): against the oracle, and bit-identical
    to the fused prefill on the same inputs (the same per-chunk work); the
    appended rows are written once."""
    import torch
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=Hq, Hkv=Hkv, D=D, P=P, T=T, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=P + T + 1)
    case = Case(w, lens=[P, P // 3], s_max=P + T + 5)
    try:
        out_n = case.out_tensor(T)
        dkv.dkv_prefill_naive(case.cache.h, case.x, T, case.wq, case.wk, case.wv, w.H, w.Hq,
                              out_n, None)
        case.cache.sync()
        ref = case.oracle()
        check_prefill(case, out_n, ref, f"naive prefill {dtype}")
        assert list(case.cache.lengths()) == [P + T, P // 3 + T]
        case.cache.k_host[...] = case.k0
        case.cache.v_host[...] = case.v0
        case.cache.set_lengths(case.lens.astype(np.int32))
        out_f = case.run_prefill()
        assert torch.equal(out_n.view(torch.int16), out_f.view(torch.int16))
    finally:
        case.free()
