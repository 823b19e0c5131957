"""8-bit E4M3 K/V caches: the fused decode and prefill read half the bytes
across the host link.  Against the fp64 oracle on the same E4M3 cache: appended K/V rows
bit-exact (the same fp32 in-order chain as the oracle, rounded once to E4M3 to
nearest, ties to even, saturating), outputs max-abs <= 1e-2 and mean-rel <= 2e-3
(the attention over the decoded E4M3 values; the quantisation of the cache is
the format's, not an error of the kernel), prefix rows and canaries untouched.
With few keys an output is close to a single value row and can reach |o| >= 4,
where bf16's own rounding of the output exceeds 1e-2: the max-abs bar is applied
to the error beyond that rounding."""
import numpy as np
import pytest

import zero_copy_offloaded_gb300 as dkv
from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, to_dev
from .test_decode_gpu import check_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 32, 8), (64, 8, 8), (128, 8, 1), (64, 16, 2)])
@pytest.mark.parametrize("P", [0, 1, 127, 300, 1000])
def test_fp8_decode_shapes(D, Hq, Hkv, P):
    w = wl.Workload("t", "decode", B=2, H=256, Hq=Hq, Hkv=Hkv, D=D, P=P, seed=P + D + Hq)
    case = Case(w, s_max=P + 5, kv_format="e4m3")
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"e4m3 D{D} G{Hq // Hkv} P{P}",
                     beyond_rounding=True)
    finally:
        case.free()


def test_fp8_decode_ragged_paged_and_unfused():
    w = wl.Workload("t", "decode", B=3, H=128, Hq=8, Hkv=2, D=128, P=700, seed=12)
    for page_tokens in (0, 16):
        case = Case(w, lens=[700, 15, 256], s_max=720, page_tokens=page_tokens,
                    kv_format="e4m3")
        try:
            out = case.run_decode()
            check_decode(case, out, case.oracle(), f"e4m3 paged={page_tokens}",
                         beyond_rounding=True)
            assert case.spare_pages_untouched()
        finally:
            case.free()
    case = Case(w, lens=[700, 15, 256], s_max=720, kv_format="e4m3")
    try:
        out = case.out_tensor(1)
        dkv.dkv_decode_unfused(case.cache.h, case.x.reshape(w.B, 1, w.H), case.wq, case.wk,
                               case.wv, w.H, w.Hq, out, None)
        case.cache.sync()
        check_decode(case, out, case.oracle(), "e4m3 unfused", beyond_rounding=True)
    finally:
        case.free()


def test_fp8_decode_spiky_keys_and_saturation():
    """Key rows ×8 (up to ~40 in E4M3) in the cache, and inputs scaled so that
    some fresh K/V sums pass 448: the appended rows saturate exactly as the
    oracle's rounding does."""
    w = wl.Workload("t", "decode", B=2, H=256, Hq=8, Hkv=2, D=128, P=500, spike_frac=0.05,
                    seed=19)
    case = Case(w, s_max=520, kv_format="e4m3")
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "e4m3 spiky", beyond_rounding=True)
        big = case.dense["x"].copy()
        xf = wl.bits_to_f32(big, w.dtype) * np.float32(300.0)
        xb = wl.to_bits(xf, w.dtype)
        ref = case.oracle(x_bits=xb, k=case.k_logical().copy(), v=case.v_logical().copy(),
                          lens=case.lens + 1)
        assert np.any(ref["k_new"] == 0x7E) or np.any(ref["k_new"] == 0xFE)  # saturated
        out2 = case.run_decode(to_dev(xb, w.dtype))
        kh, vh = case.k_logical(), case.v_logical()
        for b in range(w.B):
            p = int(case.lens[b]) + 1
            assert np.array_equal(kh[b, :, p], ref["k_new"][b, 0])
            assert np.array_equal(vh[b, :, p], ref["v_new"][b, 0])
        assert out2 is not None
    finally:
        case.free()


def test_fp8_refusals():
    c = dkv.KVCache(1, 2, 64, 64, "bf16", kv_format="e4m3")
    try:
        import torch
        x = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
        wq = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
        wk = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((1, 4, 4, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(dkv.DkvError) as ei:   # the baselines stay 16-bit only
            dkv.dkv_prefill_naive(c.h, x, 4, wq, wk, wk, 64, 4, out, None)
        assert ei.value.name == "DKV_ERR_UNSUPPORTED"
        c.set_lengths([3])
        with pytest.raises(dkv.DkvError) as ei:
            dkv.dkv_attend_naive(c.h, out[:, 0], 4, out[:, 1], None)
        assert ei.value.name == "DKV_ERR_UNSUPPORTED"
        info = dkv.dkv_cache_info(c.h)
        assert info["kv_format"] == 1 and info["host_pinned_bytes"] == 2 * 1 * 2 * 64 * 64
    finally:
        c.free()
    with pytest.raises(dkv.DkvError) as ei:
        dkv.KVCache(1, 2, 64, 64, "fp16", kv_format="e4m3")
    assert ei.value.name == "DKV_ERR_UNSUPPORTED"


def e4m3_ulp_distance(a, b):
    """Distance in representable steps between two arrays of E4M3 codes."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x80, -(x & 0x7F), x)
    return np.abs(ordered(a) - ordered(b))


def check_prefill_e4m3(case, out, ref, label, rows=None):
    """The fused prefill's projection sums on the tensor cores in another
    order than the oracle's fp32 chain and then rounds once to E4M3.  So each
    appended code is the oracle's, or one step away where the exact sum lies
    within the fp32 summation error bound (H * 2^-24 * sum|x_j w_j|) of the
    midpoint between the two codes.  One E4M3 step is an eighth of the value,
    so such a code moves outputs by far more than the attention's own error:
    the outputs are compared with the oracle's attention over the cache as
    written (the oracle's q, the written K/V rows decoded).  Prefix rows and
    canaries untouched.  Returns (max-abs beyond rounding, mean-rel, share of
    appended codes equal to the oracle's)."""
    import oracle
    from .helpers import assert_close_beyond_rounding, out_f64
    w = case.w
    T = out.shape[1]
    G = w.Hq // w.Hkv
    kh, vh = case.k_logical(), case.v_logical()
    xr = case.dense["x"]
    exact_n = tot = 0
    for b in range(w.B):
        p = int(case.lens[b])
        for host, new, wm in ((kh, ref["k_new"], case.dense["wk"]),
                              (vh, ref["v_new"], case.dense["wv"])):
            g = host[b, :, p:p + T].transpose(1, 0, 2).reshape(T, -1)   # [T, Hkv*D]
            r = new[b].reshape(T, -1)
            d = e4m3_ulp_distance(g, r)
            assert d.max() <= 1, f"{label}: appended code {d.max()} steps from the oracle's"
            if (d == 1).any():
                _, ex = oracle.project(xr[b], wm, w.dtype, exact=True)
                bound = w.H * 2.0 ** -24 * (np.abs(oracle.decode_bits(xr[b], w.dtype))
                                            @ np.abs(oracle.decode_bits(wm, w.dtype)))
                mid = (oracle.decode_e4m3(g) + oracle.decode_e4m3(r)) / 2
                off = d == 1
                assert np.all(np.abs(ex[off] - mid[off]) <= bound[off]), (
                    f"{label}: a code one step from the oracle's is not at a rounding tie")
            exact_n += int((d == 0).sum())
            tot += d.size
        assert np.array_equal(kh[b, :, :p], case.k0[b, :, :p])
        assert np.array_equal(vh[b, :, :p], case.v0[b, :, :p])
        assert np.all(kh[b, :, p + T:] == case.canary) and np.all(vh[b, :, p + T:] == case.canary)
    # the oracle's attention over the cache as written (all rows, or the
    # sampled (b, t) rows)
    want = [(b, t) for b in range(w.B) for t in range(T)] if rows is None else list(rows)
    by_b = {}
    for b, t in want:
        by_b.setdefault(b, []).append(t)
    got_all = out_f64(out, w.dtype).reshape(w.B, T, w.Hq, w.D)
    att, got = [], []
    for b, ts in by_b.items():
        p = int(case.lens[b])
        ts = np.asarray(ts)
        a = np.zeros((len(ts), w.Hq, w.D))
        for kvh in range(w.Hkv):
            kf = oracle.decode_e4m3(kh[b, kvh, :p + T])
            vf = oracle.decode_e4m3(vh[b, kvh, :p + T])
            q = oracle.decode_bits(ref["q"][b][np.ix_(ts, range(kvh * G, (kvh + 1) * G))],
                                   w.dtype)
            pos = np.repeat(p + ts, G)
            a[:, kvh * G:(kvh + 1) * G] = oracle.attend(
                kf, vf, q.reshape(-1, w.D), pos).reshape(len(ts), G, w.D)
        att.append(a)
        got.append(got_all[b, ts])
    mx, mr = assert_close_beyond_rounding(np.concatenate(got), np.concatenate(att), w.dtype,
                                          label)
    return mx, mr, exact_n / tot


@pytest.mark.parametrize("D,Hq,Hkv,P,T", [(128, 8, 2, 600, 129), (64, 8, 8, 300, 70),
                                         (128, 32, 8, 1000, 300), (64, 16, 2, 0, 37)])
def test_fp8_prefill_shapes(D, Hq, Hkv, P, T):
    """The KV-stationary prefill on an E4M3 cache: host rows converted in the
    stationary tile (K to bf16, V to fp16), new rows rounded once to E4M3."""
    w = wl.Workload("t", "prefill", B=2, H=256, Hq=Hq, Hkv=Hkv, D=D, P=P, T=T,
                    seed=P + T + D)
    case = Case(w, lens=[P, P // 2], s_max=P + T + 3, kv_format="e4m3")
    try:
        out = case.run_prefill()
        check_prefill_e4m3(case, out, case.oracle(), f"e4m3 prefill D{D} G{Hq // Hkv} P{P} T{T}")
        assert list(case.cache.lengths()) == [P + T, P // 2 + T]
    finally:
        case.free()


def test_fp8_prefill_paged_spiky_then_decode():
    """Paged E4M3 cache (16-token pages, shuffled), 5 % of the key rows x8, a
    prefill and then a decode on the grown cache, both against the oracle."""
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=520, T=90,
                    spike_frac=0.05, seed=29)
    case = Case(w, lens=[520, 257], s_max=640, page_tokens=16, kv_format="e4m3")
    try:
        out = case.run_prefill()
        ref = case.oracle()
        check_prefill_e4m3(case, out, ref, "e4m3 paged prefill")
        assert case.spare_pages_untouched()
        # the decode's oracle starts from the cache as the prefill wrote it
        k_written, v_written = case.k_logical().copy(), case.v_logical().copy()
        x2 = wl.make_dense(w.with_(T=1, seed=5))["x"]
        out2 = case.run_decode(to_dev(x2, w.dtype))
        ref2 = case.oracle(x_bits=x2, k=k_written, v=v_written, lens=case.lens + w.T)
        from .helpers import assert_close_beyond_rounding, out_f64
        assert_close_beyond_rounding(out_f64(out2, w.dtype).reshape(w.B, w.Hq, w.D),
                                     ref2["out"].reshape(w.B, w.Hq, w.D), w.dtype,
                                     "decode after e4m3 prefill")
    finally:
        case.free()


@pytest.mark.slow
def test_fp8_prefill_llama8b_full_size_sampled_rows():
    """The Llama-3-8B-shaped chunked prefill (T=4096 over P=28672) on an E4M3
    cache, as the benchmark runs it: every appended code checked, attention
    on 512 seeded query rows including the first and last token of every
    chunk that holds new tokens."""
    from .test_prefill_gpu import _edge_and_random_rows
    w = wl.WORKLOADS["llama8b_prefill"]
    case = Case(w, kv_format="e4m3")
    try:
        out = case.run_prefill()
        rows = _edge_and_random_rows(w, 512, seed=1)
        ref = case.oracle(rows=rows[:1])  # q, k_new and v_new of every token
        _, _, exact = check_prefill_e4m3(case, out, ref, "e4m3 llama8b_prefill", rows=rows)
        assert exact > 0.99
    finally:
        case.free()
