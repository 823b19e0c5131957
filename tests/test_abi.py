"""The C-ABI library builds, loads and exports every symbol include/dkv.h
declares; argument errors return before any GPU work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import zero_copy_offloaded_gb300 as dkv
from zero_copy_offloaded_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dkv.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return dkv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dkv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["dkv_cache_alloc", "dkv_free", "dkv_decode", "dkv_prefill",
                 "dkv_cache_host_ptrs", "dkv_cache_set_lengths", "dkv_sync_status"]:
        assert must in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", dkv.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (dkv_[a-z0-9_]+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(L, n)


def test_exports_are_plain_c():
    out = subprocess.run(["nm", "-D", "--defined-only", dkv.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    # every exported dkv symbol is unmangled
    assert not re.search(r"\bT _Z\S*dkv_(cache|decode|prefill|free)", out)


def test_status_strings(L):
    assert dkv.dkv_status_str(0) == "ok"
    assert "capacity" in dkv.dkv_status_str(3)
    assert "timed out" in dkv.dkv_status_str(7)


def test_invalid_arguments_fail_before_gpu_work(L):
    h = ctypes.c_void_p()
    assert L.dkv_cache_alloc(None, 1, 1, 128, 16, 0) == 1
    assert L.dkv_cache_alloc(ctypes.byref(h), 0, 1, 128, 16, 0) == 1
    assert L.dkv_cache_alloc(ctypes.byref(h), 1, 1, 128, 0, 0) == 1
    assert L.dkv_cache_alloc(ctypes.byref(h), 1, 1, 128, 16, 7) == 1
    assert L.dkv_cache_alloc(ctypes.byref(h), 65, 1, 128, 16, 0) == 1
    assert L.dkv_cache_alloc(ctypes.byref(h), 1, 1, 96, 16, 0) == 2  # unsupported head_dim
    assert h.value is None
    assert L.dkv_free(None) == 1
    assert L.dkv_decode(None, None, None, None, None, 64, 8, None, None) == 1
    assert L.dkv_prefill(None, None, 4, None, None, None, 64, 8, None, None) == 1
    assert L.dkv_sync_status(None, None) == 1
    assert L.dkv_probe_read(None, 16, None, None) == 1
    assert L.dkv_probe_write(None, 0, None) == 1
    assert L.dkv_probe_launch(0, 320, 0, None) == 1       # empty grid
    assert L.dkv_probe_launch(1, 100, 0, None) == 1       # threads not a warp multiple
    assert L.dkv_probe_launch(1, 320, 300000, None) == 1  # more shared memory than a CTA has
    assert "invalid" in dkv.dkv_last_error()
    # paged caches: page size a power of two, positive pool and table sizes
    assert L.dkv_cache_alloc_paged(ctypes.byref(h), 1, 1, 128, 12, 4, 4, 0) == 1
    assert L.dkv_cache_alloc_paged(ctypes.byref(h), 1, 1, 128, 16, 0, 4, 0) == 1
    assert L.dkv_cache_alloc_paged(ctypes.byref(h), 1, 1, 128, 16, 4, 0, 0) == 1
    assert L.dkv_cache_alloc_paged(ctypes.byref(h), 1, 1, 96, 16, 4, 4, 0) == 2
    assert h.value is None
    assert L.dkv_cache_set_page_table(None, None) == 1
    # layered caches and captured steps
    assert L.dkv_cache_alloc_layered(ctypes.byref(h), 0, 1, 1, 128, 16, 0) == 1
    assert L.dkv_cache_alloc_layered(ctypes.byref(h), 2, 0, 1, 128, 16, 0) == 1
    assert h.value is None
    assert L.dkv_decode_layer(None, 0, None, None, None, None, 64, 8, None, None) == 1
    assert L.dkv_prefill_layer(None, 0, None, 4, None, None, None, 64, 8, None, None) == 1
    assert L.dkv_step_graph_capture(None, 64, 8, None, None, None, None, None) == 1
    assert L.dkv_step_graph_launch(None, None) == 1


def test_binding_raises_typed_errors(L):
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_cache_alloc(1, 1, 96, 16)
    assert ei.value.name == "DKV_ERR_UNSUPPORTED"


def test_fault_injection_on_host_alloc(L, monkeypatch):
    monkeypatch.setenv("DKV_FAULT_INJECT", "host_alloc")
    with pytest.raises(dkv.DkvError) as ei:
        dkv.dkv_cache_alloc(1, 1, 128, 16)
    assert ei.value.name == "DKV_ERR_ALLOC"
    assert "injected" in str(ei.value)
