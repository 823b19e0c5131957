"""Handle lifetime through the C ABI: a freed cache handle is refused by every
call (a second free included) with INVALID_ARG, never touched."""
import numpy as np
import pytest

import zero_copy_offloaded_gb300 as dkv

pytestmark = pytest.mark.gpu


def test_freed_handle_is_refused():
    import torch
    c = dkv.KVCache(1, 2, 64, 32, "bf16")
    h = c.h
    c.set_lengths([4])
    dkv.dkv_free(h)
    c.h = None  # the wrapper must not free it again
    c.k_host = c.v_host = None
    for call in (lambda: dkv.dkv_free(h),
                 lambda: dkv.dkv_cache_info(h),
                 lambda: dkv.dkv_cache_set_lengths(h, np.array([1], np.int32))):
        with pytest.raises(dkv.DkvError) as ei:
            call()
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
    x = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    wk = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 1, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_decode(h, x, wq, wk, wk, 64, 4, out)
    assert ei.value.name == "DKV_ERR_INVALID_ARG"


def test_launch_probe_runs_and_times_an_empty_kernel():
    """The launch-floor probe launches cooperatively in the decode's shape (one
    320-thread CTA with 200 KB of shared memory per SM) and in a small shape;
    its event-timed cost is positive and well under a millisecond."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = torch.cuda.current_stream()
    for grid, smem in ((sms, 200 * 1024), (4, 0)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dkv.dkv_probe_launch(grid, 320, smem, s)  # warm (function attributes)
        a.record(s)
        dkv.dkv_probe_launch(grid, 320, smem, s)
        b.record(s)
        b.synchronize()
        assert 0.0 < a.elapsed_time(b) < 1.0
