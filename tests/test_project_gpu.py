"""Tensor-core projection (dkv_project, the Q projection of prefill) against
the oracle's fp32-sequential projection rounded to the dtype.

The tensor cores sum in a different order, so an element may differ from the
oracle's by one ulp of the dtype.  Where the sum nearly cancels, two fp32
summation orders can differ by more ulps of the (tiny) result; there the bar
is the fp32 summation error bound: |gpu - exact| <= K * 2^-24 * sum|x_j w_j|
plus half an ulp of the result (exact = the oracle's fp64 sum)."""
import numpy as np
import pytest

import oracle
from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import to_bits, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between two arrays of 16-bit float bits."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def run_project(M, K, N, dtype, seed=0, rows=None):
    import torch
    import zero_copy_offloaded_gb300 as dkv
    rng = np.random.default_rng(seed)
    x = wl.to_bits(rng.standard_normal((M, K)).astype(np.float32), dtype)
    w = wl.to_bits((rng.standard_normal((K, N)) / np.sqrt(K)).astype(np.float32), dtype)
    y = torch.full((M, N), float("nan"), dtype=torch_dtype(dtype), device="cuda")
    dkv.dkv_project(to_dev(x, dtype), to_dev(w, dtype), y, M, K, N, dtype)
    torch.cuda.synchronize()
    got = to_bits(y)
    sel = np.arange(M) if rows is None else np.asarray(rows)
    ref, exact = oracle.project(x[sel], w, dtype, exact=True)
    xf, wf = oracle.decode_bits(x[sel], dtype), oracle.decode_bits(w, dtype)
    bound = K * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf))
    return got[sel], ref, exact, bound


def check(got, ref, exact, bound, dtype):
    d = ulp_distance(got, ref)
    g = oracle.decode_bits(got, dtype)
    half_ulp = np.abs(g) * (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) + 1e-30
    ok = (d <= 1) | (np.abs(g - exact) <= bound + half_ulp)
    assert ok.all(), f"{(~ok).sum()} elements outside 1 ulp and the fp32 error bound"
    return float(np.mean(d == 0)), float(np.mean(d <= 1))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M,K,N", [(128, 64, 128), (200, 512, 384), (1, 4096, 64), (300, 136, 256)])
def test_project_within_one_ulp_or_error_bound(dtype, M, K, N):
    exact_frac, ulp1_frac = check(*run_project(M, K, N, dtype, seed=M + K + N), dtype)
    assert exact_frac > 0.9 and ulp1_frac > 0.999


def test_project_llama8b_q_projection_sampled_rows():
    """x [4096, 4096] . Wq [4096, 4096]: the Q projection of the chunked prefill."""
    rows = [0, 1, 127, 128, 2047, 4095] + list(np.random.default_rng(1).integers(0, 4096, 26))
    exact_frac, ulp1_frac = check(*run_project(4096, 4096, 4096, "bf16", seed=3, rows=rows), "bf16")
    assert exact_frac > 0.9 and ulp1_frac > 0.999
