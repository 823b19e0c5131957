"""Failure detection without faulting the GPU: a bounded device-side wait
that nothing completes gives up after about a second, the kernel returns,
the host reads DKV_ERR_TIMEOUT from the status word, and the next call on
the same context is correct."""
import numpy as np
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, assert_close, out_f64

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_then_recovers():
    import zero_copy_offloaded_gb300 as dkv
    w = wl.Workload("t", "decode", B=2, H=128, Hq=8, Hkv=2, D=128, P=700, seed=31)
    case = Case(w)
    try:
        dkv.dkv_cache_debug_withhold(case.cache.h, True)
        out = case.out_tensor(1)
        case.cache.decode(case.x.reshape(w.B, 1, w.H), case.wq, case.wk, case.wv, w.Hq, out)
        with pytest.raises(dkv.DkvError) as ei:
            case.cache.sync()
        assert ei.value.name == "DKV_ERR_TIMEOUT"
        # the combine saw the error: NaN outputs, not a merge of unwritten partials
        import torch
        assert torch.isnan(out.float()).all()
        # the status word was cleared by the read; the prefix is intact
        assert np.array_equal(case.cache.k_host[:, :, : w.P], case.k0[:, :, : w.P])
        dkv.dkv_cache_debug_withhold(case.cache.h, False)
        case.cache.set_lengths(case.lens.astype(np.int32))
        out = case.run_decode()
        ref = case.oracle()
        assert_close(out_f64(out, w.dtype).reshape(w.B, w.Hq, w.D),
                     ref["out"].reshape(w.B, w.Hq, w.D), "after recovery")
        case.cache.sync()  # no stale timeout left behind
    finally:
        case.free()


@pytest.mark.parametrize("D", [128, 64])
def test_withheld_prefill_rows_time_out_then_recover(D):
    """The prefill withholds the arrival of its chunks' host rows: the bounded
    waits give up, DKV_ERR_TIMEOUT is reported, the outputs are NaN (the
    combine sees the status), the prefix is intact, and the next prefill on
    the same context is correct.  D = 64 stages the new-token projection four
    deep, D = 128 two deep; both must drain their in-flight loads and give up."""
    import torch
    import zero_copy_offloaded_gb300 as dkv
    from .test_prefill_gpu import check_prefill
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=D, P=600, T=70, seed=37)
    case = Case(w, s_max=w.P + w.T + 3)
    try:
        dkv.dkv_cache_debug_withhold(case.cache.h, True)
        out = case.out_tensor(w.T)
        out.zero_()
        case.cache.prefill(case.x, case.wq, case.wk, case.wv, w.Hq, out)
        with pytest.raises(dkv.DkvError) as ei:
            case.cache.sync()
        assert ei.value.name == "DKV_ERR_TIMEOUT"
        assert torch.isnan(out.float()).all()
        assert np.array_equal(case.cache.k_host[:, :, : w.P], case.k0[:, :, : w.P])
        dkv.dkv_cache_debug_withhold(case.cache.h, False)
        case.cache.k_host[...] = case.k0
        case.cache.v_host[...] = case.v0
        case.cache.set_lengths(case.lens.astype(np.int32))
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(), "prefill after recovery")
    finally:
        case.free()
