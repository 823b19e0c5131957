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
