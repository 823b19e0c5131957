"""dkv_decode_noalloc: the decode entry point for callers that may not
allocate GPU memory (allocator callbacks, plug-ins whose host runtime owns
all device memory, fixed-budget services).  Its scratch is a fixed
__device__ array shared by every call, so two calls in a row must both match
the regular dkv_decode, which allocates its own workspace.

This file is collected last on purpose; it must pass both alone in a fresh
process and after the rest of the suite."""
import numpy as np
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, assert_close, out_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D,Hq,Hkv,P", [("bf16", 128, 16, 4, 3000), ("fp16", 64, 8, 8, 700)])
def test_noalloc_matches_decode_on_two_calls(dtype, D, Hq, Hkv, P):
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("noalloc", "decode", B=3, H=256, Hq=Hq, Hkv=Hkv, D=D, P=P, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=21)
    case = Case(w)
    try:
        ref = case.run_decode()                      # regular entry point, own workspace
        ref_f = out_f64(ref, w.dtype)
        k_after = case.cache.k_host.copy()
        v_after = case.cache.v_host.copy()
        kd, vd = dkv.dkv_cache_device_ptrs(case.cache.h)
        lens = np.full(w.B, P, np.int32)
        for call in range(2):
            out = case.out_tensor(1)
            out.fill_(float("nan"))
            dkv.dkv_decode_noalloc(case.x.reshape(w.B, 1, w.H), case.wq, case.wk, case.wv, kd, vd,
                                   lens, w.B, w.H, w.Hq, w.Hkv, w.D, case.s_max, w.dtype, out)
            import torch
            torch.cuda.synchronize()
            got = out_f64(out, w.dtype)
            assert_close(got, ref_f, f"no-alloc call {call}")
            # the append lands on the same rows with the same values
            assert np.array_equal(case.cache.k_host, k_after)
            assert np.array_equal(case.cache.v_host, v_after)
    finally:
        case.free()


def test_noalloc_rejects_bad_arguments():
    import zero_copy_offloaded_gb300 as dkv
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_decode_noalloc(None, None, None, None, None, None, [0], 1, 64, 2, 1, 64, 8,
                               "bf16", None, 0)
    assert ei.value.name == "DKV_ERR_INVALID_ARG"
