"""Paged caches: the K and V pools hold pages of page_tokens rows of one KV
head, and a per-sequence page table maps logical pages to pool pages.  The
same fused decode and prefill (through the C ABI) run on them and are compared
with the fp64 oracle on the logical cache (the pages gathered back in order).

Bars as for dense caches: decode appends bit-exact, prefill appends within
1 ulp or the fp32 summation bound, outputs max-abs <= 1e-2 and mean-rel <= 2e-3;
prefix rows, rows past the append (canary) and pool pages outside every table
(canary) untouched."""
import numpy as np
import pytest

import zero_copy_offloaded_gb300 as dkv
from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import Case, assert_close, out_f64, to_dev
from .test_decode_gpu import check_decode
from .test_prefill_gpu import check_prefill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [("bf16", 128, 8, 2), ("fp16", 64, 4, 4),
                                            ("bf16", 64, 16, 2)])
@pytest.mark.parametrize("page_tokens", [16, 64])
def test_paged_decode(dtype, D, Hq, Hkv, page_tokens):
    w = wl.Workload("t", "decode", B=3, H=128, Hq=Hq, Hkv=Hkv, D=D, P=700, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=21)
    case = Case(w, lens=[700, 15, 256], s_max=720, page_tokens=page_tokens, table_seed=page_tokens)
    try:
        out = case.run_decode()
        check_decode(case, out, case.oracle(), f"paged{page_tokens} {dtype} D{D}")
        assert case.spare_pages_untouched()
        assert list(case.cache.lengths()) == [701, 16, 257]
    finally:
        case.free()


def test_paged_decode_steps_cross_a_page_boundary():
    """Appends at rows 14, 15, 16, 17 of 16-token pages: the third step opens
    the sequence's next page."""
    w = wl.Workload("t", "decode", B=2, H=128, Hq=8, Hkv=2, D=128, P=14, seed=5)
    case = Case(w, s_max=40, page_tokens=16, table_seed=9)
    try:
        lens = case.lens.copy()
        k, v = case.k0, case.v0
        for step in range(4):
            xb = wl.make_dense(w.with_(T=1, seed=100 + step))["x"]
            out = case.run_decode(to_dev(xb, w.dtype))
            ref = case.oracle(x_bits=xb, k=k, v=v, lens=lens)
            got = out_f64(out, w.dtype).reshape(w.B, w.Hq, w.D)
            assert_close(got, ref["out"].reshape(w.B, w.Hq, w.D), f"step {step}")
            kl, vl = case.k_logical(), case.v_logical()
            for b in range(w.B):
                assert np.array_equal(kl[b, :, lens[b]], ref["k_new"][b, 0])
                assert np.array_equal(vl[b, :, lens[b]], ref["v_new"][b, 0])
            k, v = ref["k_cache_after"], ref["v_cache_after"]
            lens = lens + 1
        assert case.spare_pages_untouched()
    finally:
        case.free()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("P,T", [(0, 37), (300, 129), (517, 90)])
def test_paged_prefill(dtype, P, T):
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=P, T=T, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=P + T)
    case = Case(w, s_max=P + T + 3, page_tokens=16, table_seed=P)
    try:
        out = case.run_prefill()
        check_prefill(case, out, case.oracle(), f"paged {dtype} P{P} T{T}")
        assert case.spare_pages_untouched()
    finally:
        case.free()


def test_paged_prefill_then_decode():
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=64, P=40, T=50, seed=13)
    case = Case(w, lens=[40, 7], s_max=120, page_tokens=16, table_seed=3)
    try:
        out = case.run_prefill()
        ref = case.oracle()
        check_prefill(case, out, ref, "paged prefill")
        x2 = wl.make_dense(w.with_(T=1, seed=77))["x"]
        out2 = case.run_decode(to_dev(x2, w.dtype))
        ref2 = case.oracle(x_bits=x2, k=ref["k_cache_after"], v=ref["v_cache_after"],
                           lens=case.lens + w.T)
        got = out_f64(out2, w.dtype).reshape(w.B, w.Hq, w.D)
        assert_close(got, ref2["out"].reshape(w.B, w.Hq, w.D), "decode after paged prefill")
        assert case.spare_pages_untouched()
    finally:
        case.free()


def test_paged_missing_page_is_a_capacity_error():
    """A row the call would read or append that sits on no page is refused
    before any launch, and the lengths stay as they were."""
    w = wl.Workload("t", "decode", B=2, H=64, Hq=4, Hkv=2, D=64, P=32, seed=2)
    case = Case(w, s_max=64, page_tokens=16)
    try:
        table = case.table.copy()
        table[1, 2] = -1  # row 32 (the append of sequence 1) has no page
        case.cache.set_page_table(table)
        with pytest.raises(dkv.DkvError) as ei:
            case.run_decode()
        assert ei.value.name == "DKV_ERR_CAPACITY"
        assert list(case.cache.lengths()) == [32, 32]
        with pytest.raises(dkv.DkvError) as ei:
            case.cache.set_page_table(np.full_like(table, case.cache.num_pages))
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
    finally:
        case.free()


def test_paged_cache_rejects_dense_only_baselines():
    import torch
    c = dkv.PagedKVCache(1, 2, 64, 16, 4, 4)
    try:
        c.set_page_table(np.array([[0, 1, 2, 3]], np.int32))
        c.set_lengths([5])
        q = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(q)
        with pytest.raises(dkv.DkvError) as ei:
            dkv.dkv_attend_naive(c.h, q, 4, out, None)
        assert ei.value.name == "DKV_ERR_UNSUPPORTED"
        info = dkv.dkv_cache_info(c.h)
        assert (info["page_tokens"], info["num_pages"], info["max_pages_per_seq"]) == (16, 4, 4)
        assert info["max_tokens"] == 64
        assert info["host_pinned_bytes"] == 2 * 4 * 2 * 16 * 64 * 2
    finally:
        c.free()
