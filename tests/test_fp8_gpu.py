"""8-bit E4M3 K/V caches: the fused decode reads half the bytes across the host
link.  Against the fp64 oracle on the same E4M3 cache: appended K/V rows
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
        with pytest.raises(dkv.DkvError) as ei:
            c.prefill(x, wq, wk, wk, 4, out)
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
