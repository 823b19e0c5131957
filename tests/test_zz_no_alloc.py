"""dkv_decode_noalloc: the decode entry point for callers that may not
allocate GPU memory (allocator callbacks, plug-ins whose host runtime owns
all device memory, fixed-budget services).  Its scratch is a fixed
__device__ array shared by every call and keeping the last call's contents,
so two calls in a row with different inputs, lengths and split counts must
both match the fp64 oracle, appended rows included.

This file is collected last on purpose; it must pass both alone in a fresh
process and after the rest of the suite."""
import numpy as np
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, assert_close, out_f64, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(case, x, lens, out):
    import zero_copy_offloaded_gb300 as dkv
    w = case.w
    kd, vd = dkv.dkv_cache_device_ptrs(case.cache.h)
    dkv.dkv_decode_noalloc(x.reshape(w.B, 1, w.H), case.wq, case.wk, case.wv, kd, vd,
                           np.asarray(lens, np.int32), w.B, w.H, w.Hq, w.Hkv, w.D, case.s_max,
                           w.dtype, out)


@pytest.mark.parametrize("dtype,D,Hq,Hkv,P", [("bf16", 128, 16, 4, 3000), ("fp16", 64, 8, 8, 700)])
def test_noalloc_two_calls_against_oracle(dtype, D, Hq, Hkv, P):
    """Call 1 at the full prefix, call 2 with other hidden states and shorter,
    ragged lengths (fewer key-range splits, so a partial the first call left
    in the scratch must not be reused).  Each output is compared with the
    oracle, and the whole host cache with the oracle's cache after the
    append (bit-exact: the decode projection is the oracle's fp32 chain)."""
    import torch
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("noalloc", "decode", B=3, H=256, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=21)
    case = Case(w)
    try:
        lens1 = np.full(w.B, P, np.int64)
        x2_bits = wl.make_dense(w.with_(seed=77))["x"]
        lens2 = np.array([P // 4, P // 2 + 5, 17], np.int64)
        calls = [(case.x, case.dense["x"], lens1), (to_dev(x2_bits, dtype), x2_bits, lens2)]
        k_state, v_state = case.k0, case.v0
        for i, (x_dev, x_bits, lens) in enumerate(calls):
            out = case.out_tensor(1)
            out.fill_(float("nan"))
            _noalloc(case, x_dev, lens, out)
            dkv.dkv_decode_noalloc_status()
            torch.cuda.synchronize()
            ref = case.oracle(x_bits=x_bits, k=k_state, v=v_state, lens=lens)
            got = out_f64(out, w.dtype).reshape(w.B, w.Hq, w.D)
            assert_close(got, ref["out"].reshape(w.B, w.Hq, w.D), f"no-alloc call {i}")
            assert np.array_equal(case.cache.k_host, ref["k_cache_after"]), f"call {i} K cache"
            assert np.array_equal(case.cache.v_host, ref["v_cache_after"]), f"call {i} V cache"
            k_state, v_state = ref["k_cache_after"], ref["v_cache_after"]
    finally:
        case.free()


def test_noalloc_timeout_gives_nan_and_status_then_recovers():
    """A withheld producer signal makes the bounded wait give up: the call's
    outputs are NaN (never a merge of stale scratch), the status query
    reports DKV_ERR_TIMEOUT and clears it, and the next call is correct."""
    import torch
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("noalloc_to", "decode", B=2, H=128, Hq=8, Hkv=2, D=128, P=900, seed=5)
    case = Case(w)
    try:
        lens = np.full(w.B, w.P, np.int64)
        good = case.out_tensor(1)
        _noalloc(case, case.x, lens, good)   # leaves valid partials in the scratch
        dkv.dkv_decode_noalloc_status()
        dkv.dkv_decode_noalloc_debug_withhold(True)
        try:
            out = case.out_tensor(1)
            out.zero_()
            _noalloc(case, case.x, lens, out)
            with pytest.raises(dkv.DkvError) as ei:
                dkv.dkv_decode_noalloc_status()
            assert ei.value.name == "DKV_ERR_TIMEOUT"
            assert torch.isnan(out.float()).all()
        finally:
            dkv.dkv_decode_noalloc_debug_withhold(False)
        dkv.dkv_decode_noalloc_status()  # cleared by the read
        assert np.array_equal(case.cache.k_host[:, :, :w.P], case.k0[:, :, :w.P])
        out = case.out_tensor(1)
        _noalloc(case, case.x, lens, out)
        dkv.dkv_decode_noalloc_status()
        ref = case.oracle()
        assert_close(out_f64(out, w.dtype).reshape(w.B, w.Hq, w.D),
                     ref["out"].reshape(w.B, w.Hq, w.D), "after recovery")
    finally:
        case.free()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """64 sequences of 256 query heads at head_dim 128 need more than the 8 MiB
    static scratch even with one split: DKV_ERR_CAPACITY before any launch."""
    import torch
    import zero_copy_offloaded_gb300 as dkv
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_decode_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, [8] * 64, 64, 256, 256,
                               32, 128, 64, "bf16", dummy)
    assert ei.value.name == "DKV_ERR_CAPACITY"


def test_noalloc_rejects_bad_arguments():
    import zero_copy_offloaded_gb300 as dkv
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_decode_noalloc(None, None, None, None, None, None, [0], 1, 64, 2, 1, 64, 8,
                               "bf16", None, 0)
    assert ei.value.name == "DKV_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        dkv.dkv_decode_noalloc(None, None, None, None, None, None, [0], 2, 64, 2, 1, 64, 8,
                               "bf16", None, 0)
