"""Decode parity: the fused zero-copy decode (through the C ABI) against the
fp64 oracle on the same seeded inputs.

Bars: appended K/V rows bit-exact (the kernel's projection is the same fp32
FMA chain over H in order as the oracle's); attention output max-abs <= 1e-2
and sum|err|/sum|ref| <= 2e-3 versus fp64; prefix rows untouched; rows past
the append untouched (canary)."""
import numpy as np
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, assert_close, assert_close_beyond_rounding, out_f64, errors

pytestmark = pytest.mark.gpu


def check_decode(case: Case, out, ref, label="", beyond_rounding=False):
    w = case.w
    got = out_f64(out, w.dtype).reshape(w.B, w.Hq, w.D)
    if beyond_rounding:
        mx, mr = assert_close_beyond_rounding(got, ref["out"].reshape(w.B, w.Hq, w.D), w.dtype,
                                              label)
    else:
        mx, mr = assert_close(got, ref["out"].reshape(w.B, w.Hq, w.D), label)
    kh, vh = case.k_logical(), case.v_logical()
    for b in range(w.B):
        p = int(case.lens[b])
        assert np.array_equal(kh[b, :, p], ref["k_new"][b, 0]), f"{label} k append b={b}"
        assert np.array_equal(vh[b, :, p], ref["v_new"][b, 0]), f"{label} v append b={b}"
        assert np.array_equal(kh[b, :, :p], case.k0[b, :, :p]), f"{label} k prefix b={b}"
        assert np.array_equal(vh[b, :, :p], case.v0[b, :, :p]), f"{label} v prefix b={b}"
        assert np.all(kh[b, :, p + 1:] == case.canary) and np.all(vh[b, :, p + 1:] == case.canary)
    return mx, mr


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D,Hq,Hkv", [(64, 8, 2), (128, 8, 8), (128, 16, 8), (64, 16, 2),
                                      (128, 32, 4)])
@pytest.mark.parametrize("P", [0, 1, 63, 64, 300, 1000])
def test_decode_shapes(dtype, D, Hq, Hkv, P):
    w = wl.Workload("t", "decode", B=2, H=256, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=P + D)
    case = Case(w, s_max=P + 5)
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"{dtype} D{D} G{Hq // Hkv} P{P}")
    finally:
        case.free()


def test_decode_ragged_lengths():
    w = wl.Workload("t", "decode", B=5, H=128, Hq=8, Hkv=2, D=128, P=700, seed=3)
    case = Case(w, lens=[0, 1, 129, 700, 333], s_max=800)
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "ragged")
        assert list(case.cache.lengths()) == [1, 2, 130, 701, 334]
    finally:
        case.free()


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_decode_forced_splits(splits):
    w = wl.Workload("t", "decode", B=2, H=256, Hq=8, Hkv=2, D=128, P=2000, seed=5)
    case = Case(w, tuning=dict(splits=splits))
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"splits={splits}")
    finally:
        case.free()


@pytest.mark.parametrize("tile_n,stages", [(32, 2), (64, 3), (128, 2)])
def test_decode_tiles_and_stages(tile_n, stages):
    w = wl.Workload("t", "decode", B=3, H=128, Hq=4, Hkv=1, D=128, P=999, seed=9)
    case = Case(w, tuning=dict(tile_n=tile_n, stages=stages))
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"N={tile_n} m={stages}")
    finally:
        case.free()


def test_decode_two_steps():
    w = wl.Workload("t", "decode", B=2, H=256, Hq=8, Hkv=2, D=64, P=500, seed=2)
    case = Case(w, s_max=510)
    try:
        out1 = case.run_decode()
        ref1 = case.oracle()
        check_decode(case, out1, ref1, "step1")
        x2 = wl.make_dense(w.with_(seed=77))["x"]
        from .helpers import to_dev
        out2 = case.run_decode(to_dev(x2, w.dtype))
        ref2 = case.oracle(x_bits=x2, k=ref1["k_cache_after"], v=ref1["v_cache_after"],
                           lens=case.lens + 1)
        got = out_f64(out2, w.dtype).reshape(w.B, w.Hq, w.D)
        assert_close(got, ref2["out"].reshape(w.B, w.Hq, w.D), "step2")
        assert np.array_equal(case.cache.k_host[:, :, : 502], ref2["k_cache_after"][:, :, :502])
        assert np.array_equal(case.cache.v_host[:, :, : 502], ref2["v_cache_after"][:, :, :502])
    finally:
        case.free()


@pytest.mark.parametrize("page_tokens", [0, 16])
@pytest.mark.parametrize("dtype,D,Hq,Hkv", [("bf16", 128, 32, 8), ("fp16", 64, 8, 8)])
def test_decode_unfused_baseline(dtype, D, Hq, Hkv, page_tokens):
    """The separate-kernel baseline (a projection launch that appends, then an
    attention launch that reads every row, the new one included, from the
    host cache) meets the same bars: bit-exact appends, outputs within the
    tolerances."""
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("t", "decode", B=3, H=256, Hq=Hq, Hkv=Hkv, D=D, P=333, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=17)
    case = Case(w, lens=[333, 0, 64], s_max=340, page_tokens=page_tokens)
    try:
        out = case.out_tensor(1)
        dkv.dkv_decode_unfused(case.cache.h, case.x.reshape(w.B, 1, w.H), case.wq, case.wk,
                               case.wv, w.H, w.Hq, out, None)
        case.cache.sync()
        check_decode(case, out, case.oracle(), f"unfused {dtype} pages={page_tokens}")
        assert list(case.cache.lengths()) == [334, 1, 65]
        assert dkv.dkv_last_launch_count() == 3
    finally:
        case.free()


def test_decode_tiny_workload_full_size():
    case = Case(wl.WORKLOADS["tiny_decode"])
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "tiny_decode")
    finally:
        case.free()


def test_decode_capacity_error_leaves_cache_unchanged():
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("t", "decode", B=1, H=64, Hq=2, Hkv=1, D=64, P=10, seed=1)
    case = Case(w, s_max=10)
    try:
        with pytest.raises(dkv.DkvError) as ei:
            case.run_decode()
        assert ei.value.name == "DKV_ERR_CAPACITY"
        assert list(case.cache.lengths()) == [10]
        assert np.array_equal(case.cache.k_host, case.k0)
    finally:
        case.free()


@pytest.mark.slow
def test_decode_llama8b_full_size():
    """Llama-3-8B-shaped decode at its full size (B=8, P=32768)."""
    case = Case(wl.WORKLOADS["llama8b_decode"])
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "llama8b_decode")
    finally:
        case.free()


@pytest.mark.slow
def test_decode_longctx_spiked():
    """Long-context decode with 1% of keys scaled x8 (peaked softmax), B=4, S=16K."""
    case = Case(wl.WORKLOADS["longctx_b4_s16k"])
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "longctx_b4_s16k")
    finally:
        case.free()


@pytest.mark.parametrize("B,H,D", [(31, 208, 128), (33, 128, 128), (40, 64, 128), (3, 208, 64)])
def test_decode_projection_batch_edges(B, H, D):
    """The projection's batch mapping at its edges: two weight blocks per pass
    up to 32 sequences (31: up to eight chains a thread), one block per pass
    beyond (33, 40), and a hidden size whose last 128-row chunk is partial
    (208 = 128 + 80); appends bit-exact, outputs within the bars."""
    w = wl.Workload("t", "decode", B=B, H=H, Hq=8, Hkv=2, D=D, P=70, seed=B + H)
    lens = [(11 * b + 3) % 71 for b in range(B)]
    case = Case(w, lens=lens, s_max=80)
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"B={B} H={H} D={D}")
        assert list(case.cache.lengths()) == [n + 1 for n in lens]
    finally:
        case.free()


def test_decode_max_batch():
    """The largest batch a call takes (64 sequences), ragged lengths including 0."""
    w = wl.Workload("t", "decode", B=64, H=128, Hq=8, Hkv=2, D=64, P=200, seed=64)
    lens = [(7 * b) % 201 for b in range(64)]
    case = Case(w, lens=lens, s_max=210)
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "B=64")
        assert list(case.cache.lengths()) == [n + 1 for n in lens]
    finally:
        case.free()


@pytest.mark.slow
def test_decode_longctx_128k_full():
    """One sequence at 131072 cached keys (1 % of keys x8), every query head
    against the full oracle."""
    case = Case(wl.WORKLOADS["longctx_b1_s128k"])
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "longctx_b1_s128k")
    finally:
        case.free()


@pytest.mark.slow
def test_decode_mha_fp16_full_size():
    case = Case(wl.WORKLOADS["mha_fp16_decode"])
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), "mha_fp16_decode")
    finally:
        case.free()
