"""Tensor-core projection (dkv_project, the Q projection of prefill) against
the oracle's fp32-sequential projection rounded to the dtype.

The tensor cores sum in a different order, so an element may differ from the
oracle's by one ulp of the dtype.  Where the sum nearly cancels, two fp32
summation orders can differ by more ulps of the (tiny) result; there the bar
is the fp32 summation error bound (see helpers.assert_projection_close)."""
import numpy as np
import pytest

from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import assert_projection_close, to_bits, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


def run_project(M, K, N, dtype, seed=0, rows=None):
    import torch
    import zero_copy_offloaded_gb300 as dkv
    rng = np.random.default_rng(seed)
    x = wl.to_bits(rng.standard_normal((M, K)).astype(np.float32), dtype)
    w = wl.to_bits((rng.standard_normal((K, N)) / np.sqrt(K)).astype(np.float32), dtype)
    y = torch.full((M, N), float("nan"), dtype=torch_dtype(dtype), device="cuda")
    dkv.dkv_project(to_dev(x, dtype), to_dev(w, dtype), y, M, K, N, dtype)
    torch.cuda.synchronize()
    sel = np.arange(M) if rows is None else np.asarray(rows)
    return to_bits(y)[sel], x[sel], w


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (200, 512, 384), (1, 4096, 64), (300, 136, 256),
                                   (130, 104, 192)])
def test_project_within_one_ulp_or_error_bound(dtype, M, K, N):
    got, x, w = run_project(M, K, N, dtype, seed=M + K + N)
    exact_frac, ulp1_frac, _ = assert_projection_close(got, x, w, dtype)
    assert exact_frac > 0.9 and ulp1_frac > 0.999


def test_project_llama8b_q_projection_sampled_rows():
    """x [4096, 4096] . Wq [4096, 4096]: the Q projection of the chunked prefill."""
    rows = [0, 1, 127, 128, 2047, 4095] + list(np.random.default_rng(1).integers(0, 4096, 26))
    got, x, w = run_project(4096, 4096, 4096, "bf16", seed=3, rows=rows)
    exact_frac, ulp1_frac, _ = assert_projection_close(got, x, w, "bf16")
    assert exact_frac > 0.9 and ulp1_frac > 0.999
