"""Zero-copy host-resident KV-cache attention for GB300 (DirectKV's hot path).

A thin ctypes binding over ``libdkv.so`` whose C ABI is ``include/dkv.h``.
Every function here only marshals arguments (tensor -> device pointer,
stream -> cudaStream_t) and calls the library of the same name; every step
of the computation runs in the library's CUDA kernels.  There is no CPU or
PyTorch fallback: if the library is missing or a call fails, a
``DkvError`` is raised.

PyTorch is used only as plumbing for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "DkvError", "BF16", "FP16", "lib", "lib_path", "KVCache",
    "dkv_cache_alloc", "dkv_free", "dkv_cache_host_ptrs", "dkv_cache_device_ptrs",
    "dkv_cache_set_lengths", "dkv_cache_get_lengths", "dkv_cache_info", "dkv_cache_reserve",
    "dkv_cache_set_tuning", "dkv_decode", "dkv_prefill", "dkv_sync_status", "dkv_status_str",
    "dkv_last_error", "dkv_probe_read", "dkv_probe_write", "dkv_probe_launch", "dkv_attend_naive",
    "dkv_decode_staged", "dkv_prefill_staged", "dkv_prefill_naive", "dkv_decode_unfused", "dkv_last_launch_count", "dkv_cache_kernel_timing",
    "dkv_cache_last_kernel_ms", "dkv_cache_alloc_paged", "dkv_cache_set_page_table",
    "PagedKVCache", "LayeredKVCache", "dkv_cache_alloc_layered", "dkv_decode_layer",
    "dkv_prefill_layer", "dkv_step_graph_capture", "dkv_step_graph_launch",
    "dkv_cache_alloc_ex", "KV_FORMATS", "dkv_decode_noalloc", "dkv_decode_noalloc_status",
    "dkv_decode_noalloc_debug_withhold", "dkv_pci_numa_node", "dkv_numa_probe",
]

BF16 = 0
FP16 = 1
_DTYPE = {"bf16": BF16, "fp16": FP16, BF16: BF16, FP16: FP16}
STATUS = {0: "DKV_OK", 1: "DKV_ERR_INVALID_ARG", 2: "DKV_ERR_UNSUPPORTED", 3: "DKV_ERR_CAPACITY",
          4: "DKV_ERR_NO_MAPPED_MEMORY", 5: "DKV_ERR_ALLOC", 6: "DKV_ERR_CUDA",
          7: "DKV_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))


def lib_path() -> str:
    return os.path.join(_HERE, "_build", "libdkv.so")


class DkvError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {detail}")


class _CacheInfo(ctypes.Structure):
    _fields_ = [("host_pinned_bytes", ctypes.c_size_t),
                ("device_workspace_bytes", ctypes.c_size_t),
                ("device_staging_bytes", ctypes.c_size_t),
                ("batch", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("dtype", ctypes.c_int), ("page_tokens", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
                ("layers", ctypes.c_int), ("kv_format", ctypes.c_int),
                ("numa_node_wanted", ctypes.c_int), ("numa_node", ctypes.c_int)]


class _CacheDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("dtype", ctypes.c_int), ("kv_format", ctypes.c_int), ("layers", ctypes.c_int),
                ("page_tokens", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("max_pages_per_seq", ctypes.c_int)]


KV_FORMATS = {"native": 0, "e4m3": 1}


_lib = None


def lib(build_if_missing: bool = False):
    """The loaded libdkv (built in-tree by ``zero_copy_offloaded_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError(f"{path} is missing: run zero_copy_offloaded_gb300/build.py "
                              "(the CUDA library is required; there is no fallback)")
        from . import build as _b
        _b.build()
    L = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "dkv_cache_alloc": [ctypes.POINTER(P), I, I, I, I, I],
        "dkv_cache_alloc_paged": [ctypes.POINTER(P), I, I, I, I, I, I, I],
        "dkv_cache_set_page_table": [P, P],
        "dkv_cache_alloc_layered": [ctypes.POINTER(P), I, I, I, I, I, I],
        "dkv_cache_alloc_ex": [ctypes.POINTER(P), ctypes.POINTER(_CacheDesc)],
        "dkv_decode_layer": [P, I, P, P, P, P, I, I, P, P],
        "dkv_prefill_layer": [P, I, P, I, P, P, P, I, I, P, P],
        "dkv_step_graph_capture": [P, I, I, P, P, P, P, P],
        "dkv_step_graph_launch": [P, P],
        "dkv_free": [P],
        "dkv_cache_host_ptrs": [P, ctypes.POINTER(P), ctypes.POINTER(P)],
        "dkv_cache_device_ptrs": [P, ctypes.POINTER(P), ctypes.POINTER(P)],
        "dkv_cache_set_lengths": [P, P],
        "dkv_cache_get_lengths": [P, P],
        "dkv_cache_info": [P, ctypes.POINTER(_CacheInfo)],
        "dkv_cache_reserve": [P, I, I],
        "dkv_cache_set_tuning": [P, I, I, I],
        "dkv_decode": [P, P, P, P, P, I, I, P, P],
        "dkv_prefill": [P, P, I, P, P, P, I, I, P, P],
        "dkv_sync_status": [P, P],
        "dkv_probe_read": [P, Z, P, P],
        "dkv_probe_write": [P, Z, P],
        "dkv_probe_launch": [I, I, I, P],
        "dkv_attend_naive": [P, P, I, P, P],
        "dkv_decode_staged": [P, P, P, P, P, I, I, P, P, P, P],
        "dkv_prefill_staged": [P, P, I, P, P, P, I, I, P, P, P, P],
        "dkv_prefill_naive": [P, P, I, P, P, P, I, I, P, P],
        "dkv_decode_unfused": [P, P, P, P, P, I, I, P, P],
        "dkv_cache_kernel_timing": [P, I],
        "dkv_cache_last_kernel_ms": [P, ctypes.POINTER(ctypes.c_float)],
        "dkv_decode_noalloc": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P],
        "dkv_decode_noalloc_status": [P],
        "dkv_decode_noalloc_debug_withhold": [I],
        "dkv_project": [P, P, P, I, I, I, I, P],
        "dkv_cache_debug_withhold": [P, I],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.dkv_status_str.argtypes = [ctypes.c_int]
    L.dkv_status_str.restype = ctypes.c_char_p
    L.dkv_last_error.argtypes = []
    L.dkv_last_error.restype = ctypes.c_char_p
    L.dkv_last_launch_count.argtypes = []
    L.dkv_last_launch_count.restype = ctypes.c_int
    L.dkv_pci_numa_node.argtypes = [ctypes.c_char_p, ctypes.c_char_p]
    L.dkv_pci_numa_node.restype = ctypes.c_int
    L.dkv_numa_probe.argtypes = [ctypes.c_int]
    L.dkv_numa_probe.restype = ctypes.c_int
    _lib = L
    return L


def _check(st: int, where: str):
    if st != 0:
        raise DkvError(st, where, lib().dkv_last_error().decode())


def _ptr(t) -> int | None:
    """Device pointer of a CUDA tensor (or an int / None passed through)."""
    if t is None or isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return t.data_ptr()
    raise TypeError(f"cannot take a device pointer of {type(t)}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def dkv_status_str(st: int) -> str:
    return lib().dkv_status_str(st).decode()


def dkv_last_error() -> str:
    return lib().dkv_last_error().decode()


def dkv_last_launch_count() -> int:
    return lib().dkv_last_launch_count()


def dkv_cache_alloc(batch, n_kv_heads, head_dim, max_tokens, dtype="bf16") -> int:
    h = ctypes.c_void_p()
    _check(lib().dkv_cache_alloc(ctypes.byref(h), batch, n_kv_heads, head_dim, max_tokens,
                                 _DTYPE[dtype]), "dkv_cache_alloc")
    return h.value


def dkv_cache_alloc_paged(batch, n_kv_heads, head_dim, page_tokens, num_pages,
                          max_pages_per_seq, dtype="bf16") -> int:
    h = ctypes.c_void_p()
    _check(lib().dkv_cache_alloc_paged(ctypes.byref(h), batch, n_kv_heads, head_dim, page_tokens,
                                       num_pages, max_pages_per_seq, _DTYPE[dtype]),
           "dkv_cache_alloc_paged")
    return h.value


def dkv_cache_set_page_table(h, table):
    """table: int32 [batch, max_pages_per_seq] of pool page indices (-1: none)."""
    t = np.ascontiguousarray(table, dtype=np.int32)
    _check(lib().dkv_cache_set_page_table(h, t.ctypes.data), "dkv_cache_set_page_table")


def dkv_cache_alloc_ex(batch, n_kv_heads, head_dim, max_tokens=0, dtype="bf16",
                       kv_format="native", layers=1, page_tokens=0, num_pages=0,
                       max_pages_per_seq=0) -> int:
    d = _CacheDesc(batch, n_kv_heads, head_dim, max_tokens, _DTYPE[dtype], KV_FORMATS[kv_format],
                   layers, page_tokens, num_pages, max_pages_per_seq)
    h = ctypes.c_void_p()
    _check(lib().dkv_cache_alloc_ex(ctypes.byref(h), ctypes.byref(d)), "dkv_cache_alloc_ex")
    return h.value


def dkv_cache_alloc_layered(layers, batch, n_kv_heads, head_dim, max_tokens, dtype="bf16") -> int:
    h = ctypes.c_void_p()
    _check(lib().dkv_cache_alloc_layered(ctypes.byref(h), layers, batch, n_kv_heads, head_dim,
                                         max_tokens, _DTYPE[dtype]), "dkv_cache_alloc_layered")
    return h.value


def dkv_decode_layer(h, layer, x, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_decode_layer(h, layer, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), hidden,
                                  n_q_heads, _ptr(out), _stream(stream)), "dkv_decode_layer")


def dkv_prefill_layer(h, layer, x, T, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_prefill_layer(h, layer, _ptr(x), T, _ptr(wq), _ptr(wk), _ptr(wv), hidden,
                                   n_q_heads, _ptr(out), _stream(stream)), "dkv_prefill_layer")


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))(*[_ptr(t) for t in ts])
    return arr


def dkv_step_graph_capture(h, hidden, n_q_heads, xs, wqs, wks, wvs, outs):
    """Per-layer lists of device tensors; the arrays are copied into the graph."""
    arrs = [_ptr_array(v) for v in (xs, wqs, wks, wvs, outs)]
    _check(lib().dkv_step_graph_capture(h, hidden, n_q_heads,
                                        *[ctypes.cast(a, ctypes.c_void_p) for a in arrs]),
           "dkv_step_graph_capture")


def dkv_step_graph_launch(h, stream=None):
    _check(lib().dkv_step_graph_launch(h, _stream(stream)), "dkv_step_graph_launch")


def dkv_free(h):
    _check(lib().dkv_free(h), "dkv_free")


def dkv_cache_host_ptrs(h):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib().dkv_cache_host_ptrs(h, ctypes.byref(k), ctypes.byref(v)), "dkv_cache_host_ptrs")
    return k.value, v.value


def dkv_cache_device_ptrs(h):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(lib().dkv_cache_device_ptrs(h, ctypes.byref(k), ctypes.byref(v)),
           "dkv_cache_device_ptrs")
    return k.value, v.value


def dkv_cache_set_lengths(h, lens):
    a = np.ascontiguousarray(lens, dtype=np.int32)
    _check(lib().dkv_cache_set_lengths(h, a.ctypes.data), "dkv_cache_set_lengths")


def dkv_cache_get_lengths(h, batch):
    a = np.zeros(batch, np.int32)
    _check(lib().dkv_cache_get_lengths(h, a.ctypes.data), "dkv_cache_get_lengths")
    return a


def dkv_cache_info(h) -> dict:
    i = _CacheInfo()
    _check(lib().dkv_cache_info(h, ctypes.byref(i)), "dkv_cache_info")
    return {f: getattr(i, f) for f, _ in _CacheInfo._fields_}


def dkv_pci_numa_node(pci_bus_id: str, sysfs_root: str | None = None) -> int:
    """Host NUMA node of a PCI device (-1 if unknown); see include/dkv.h."""
    return lib().dkv_pci_numa_node(pci_bus_id.encode(),
                                   sysfs_root.encode() if sysfs_root else None)


def dkv_numa_probe(node: int) -> int:
    return lib().dkv_numa_probe(int(node))


def dkv_cache_reserve(h, n_q_heads, max_new_tokens):
    _check(lib().dkv_cache_reserve(h, n_q_heads, max_new_tokens), "dkv_cache_reserve")


def dkv_cache_set_tuning(h, splits=0, tile_n=0, stages=0):
    _check(lib().dkv_cache_set_tuning(h, splits, tile_n, stages), "dkv_cache_set_tuning")


def dkv_cache_debug_withhold(h, enable=True):
    _check(lib().dkv_cache_debug_withhold(h, int(bool(enable))), "dkv_cache_debug_withhold")


def dkv_cache_kernel_timing(h, enable=True):
    _check(lib().dkv_cache_kernel_timing(h, int(bool(enable))), "dkv_cache_kernel_timing")


def dkv_cache_last_kernel_ms(h) -> float:
    ms = ctypes.c_float()
    _check(lib().dkv_cache_last_kernel_ms(h, ctypes.byref(ms)), "dkv_cache_last_kernel_ms")
    return float(ms.value)


def dkv_decode(h, x, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_decode(h, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), hidden, n_q_heads,
                            _ptr(out), _stream(stream)), "dkv_decode")


def dkv_prefill(h, x, T, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_prefill(h, _ptr(x), T, _ptr(wq), _ptr(wk), _ptr(wv), hidden, n_q_heads,
                             _ptr(out), _stream(stream)), "dkv_prefill")


def dkv_sync_status(h, stream=None):
    _check(lib().dkv_sync_status(h, _stream(stream)), "dkv_sync_status")


def dkv_project(x, w, y, M, K, N, dtype="bf16", stream=None):
    _check(lib().dkv_project(_ptr(x), _ptr(w), _ptr(y), M, K, N, _DTYPE[dtype], _stream(stream)),
           "dkv_project")


def dkv_probe_read(src, nbytes, sink, stream=None):
    _check(lib().dkv_probe_read(_ptr(src), nbytes, _ptr(sink), _stream(stream)), "dkv_probe_read")


def dkv_probe_write(dst, nbytes, stream=None):
    _check(lib().dkv_probe_write(_ptr(dst), nbytes, _stream(stream)), "dkv_probe_write")


def dkv_probe_launch(grid, threads, smem_bytes, stream=None):
    _check(lib().dkv_probe_launch(grid, threads, smem_bytes, _stream(stream)), "dkv_probe_launch")


def dkv_attend_naive(h, q, n_q_heads, out, stream=None):
    _check(lib().dkv_attend_naive(h, _ptr(q), n_q_heads, _ptr(out), _stream(stream)),
           "dkv_attend_naive")


def dkv_decode_unfused(h, x, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_decode_unfused(h, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), hidden, n_q_heads,
                                    _ptr(out), _stream(stream)), "dkv_decode_unfused")


def dkv_decode_staged(h, x, wq, wk, wv, hidden, n_q_heads, out, k_stage, v_stage, stream=None):
    _check(lib().dkv_decode_staged(h, _ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), hidden, n_q_heads,
                                   _ptr(out), _ptr(k_stage), _ptr(v_stage), _stream(stream)),
           "dkv_decode_staged")


def dkv_prefill_staged(h, x, T, wq, wk, wv, hidden, n_q_heads, out, k_stage, v_stage,
                       stream=None):
    _check(lib().dkv_prefill_staged(h, _ptr(x), T, _ptr(wq), _ptr(wk), _ptr(wv), hidden,
                                    n_q_heads, _ptr(out), _ptr(k_stage), _ptr(v_stage),
                                    _stream(stream)),
           "dkv_prefill_staged")


def dkv_prefill_naive(h, x, T, wq, wk, wv, hidden, n_q_heads, out, stream=None):
    _check(lib().dkv_prefill_naive(h, _ptr(x), T, _ptr(wq), _ptr(wk), _ptr(wv), hidden,
                                   n_q_heads, _ptr(out), _stream(stream)),
           "dkv_prefill_naive")


def dkv_decode_noalloc(x, wq, wk, wv, k_cache, v_cache, lengths, batch, hidden, n_q_heads,
                       n_kv_heads, head_dim, max_tokens, dtype, out, stream=None):
    """dkv_decode on caller-owned buffers with no allocation (see include/dkv.h)."""
    lens = np.ascontiguousarray(lengths, dtype=np.int32).reshape(-1)
    if lens.size < batch:
        raise ValueError(f"lengths holds {lens.size} entries for a batch of {batch}")
    _check(lib().dkv_decode_noalloc(_ptr(x), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(k_cache),
                                    _ptr(v_cache), lens.ctypes.data, batch, hidden, n_q_heads,
                                    n_kv_heads, head_dim, max_tokens, _DTYPE[dtype], _ptr(out),
                                    _stream(stream)), "dkv_decode_noalloc")


def dkv_decode_noalloc_status(stream=None):
    """Status of the last dkv_decode_noalloc on the current device (raises on an error)."""
    _check(lib().dkv_decode_noalloc_status(_stream(stream)), "dkv_decode_noalloc_status")


def dkv_decode_noalloc_debug_withhold(enable=True):
    _check(lib().dkv_decode_noalloc_debug_withhold(int(bool(enable))),
           "dkv_decode_noalloc_debug_withhold")


class KVCache:
    """Owner of one dkv_cache handle, with numpy views of the pinned caches."""

    def __init__(self, batch, n_kv_heads, head_dim, max_tokens, dtype="bf16", kv_format="native"):
        """kv_format "e4m3": 8-bit E4M3 elements (views of uint8 bits; decode only)."""
        self.B, self.Hkv, self.D, self.S_max = batch, n_kv_heads, head_dim, max_tokens
        self.dtype, self.kv_format = dtype, kv_format
        self.h = dkv_cache_alloc_ex(batch, n_kv_heads, head_dim, max_tokens, dtype, kv_format)
        self._views((batch, n_kv_heads, max_tokens, head_dim))

    def _views(self, shape):
        kp, vp = dkv_cache_host_ptrs(self.h)
        n = int(np.prod(shape))
        el = ctypes.c_uint8 if self.kv_format == "e4m3" else ctypes.c_uint16
        self.k_host = np.ctypeslib.as_array((el * n).from_address(kp)).reshape(shape)
        self.v_host = np.ctypeslib.as_array((el * n).from_address(vp)).reshape(shape)

    def set_lengths(self, lens):
        dkv_cache_set_lengths(self.h, np.broadcast_to(np.asarray(lens, np.int32), (self.B,)))

    def lengths(self):
        return dkv_cache_get_lengths(self.h, self.B)

    def decode(self, x, wq, wk, wv, n_q_heads, out, stream=None):
        dkv_decode(self.h, x, wq, wk, wv, x.shape[-1], n_q_heads, out, stream)

    def prefill(self, x, wq, wk, wv, n_q_heads, out, stream=None):
        dkv_prefill(self.h, x, x.shape[1], wq, wk, wv, x.shape[-1], n_q_heads, out, stream)

    def sync(self, stream=None):
        dkv_sync_status(self.h, stream)

    def free(self):
        if self.h is not None:
            self.k_host = self.v_host = None
            dkv_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class PagedKVCache(KVCache):
    """A paged cache: numpy views of the K and V page pools
    ([num_pages, Hkv, page_tokens, D] uint16 each) and the page table."""

    def __init__(self, batch, n_kv_heads, head_dim, page_tokens, num_pages, max_pages_per_seq,
                 dtype="bf16", kv_format="native"):
        self.B, self.Hkv, self.D = batch, n_kv_heads, head_dim
        self.page_tokens, self.num_pages, self.max_pages = page_tokens, num_pages, max_pages_per_seq
        self.S_max = page_tokens * max_pages_per_seq
        self.dtype, self.kv_format = dtype, kv_format
        self.h = dkv_cache_alloc_ex(batch, n_kv_heads, head_dim, 0, dtype, kv_format, 1,
                                    page_tokens, num_pages, max_pages_per_seq)
        self._views((num_pages, n_kv_heads, page_tokens, head_dim))
        self.table = np.full((batch, max_pages_per_seq), -1, np.int32)

    def set_page_table(self, table):
        dkv_cache_set_page_table(self.h, table)
        self.table = np.array(table, dtype=np.int32, copy=True)


class LayeredKVCache(KVCache):
    """A whole model's caches: numpy views [layers, B, Hkv, S_max, D] (uint16)
    of the pinned K and V, per-layer decode / prefill and the captured step."""

    def __init__(self, layers, batch, n_kv_heads, head_dim, max_tokens, dtype="bf16",
                 kv_format="native"):
        self.L, self.B, self.Hkv, self.D, self.S_max = layers, batch, n_kv_heads, head_dim, max_tokens
        self.dtype, self.kv_format = dtype, kv_format
        self.h = dkv_cache_alloc_ex(batch, n_kv_heads, head_dim, max_tokens, dtype, kv_format,
                                    layers)
        self._views((layers, batch, n_kv_heads, max_tokens, head_dim))

    def decode_layer(self, layer, x, wq, wk, wv, n_q_heads, out, stream=None):
        dkv_decode_layer(self.h, layer, x, wq, wk, wv, x.shape[-1], n_q_heads, out, stream)

    def prefill_layer(self, layer, x, wq, wk, wv, n_q_heads, out, stream=None):
        dkv_prefill_layer(self.h, layer, x, x.shape[1], wq, wk, wv, x.shape[-1], n_q_heads, out,
                          stream)

    def capture_step(self, xs, wqs, wks, wvs, n_q_heads, outs):
        dkv_step_graph_capture(self.h, xs[0].shape[-1], n_q_heads, xs, wqs, wks, wvs, outs)

    def launch_step(self, stream=None):
        dkv_step_graph_launch(self.h, stream)
