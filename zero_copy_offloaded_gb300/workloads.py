"""Seeded synthetic workloads for the zero-copy KV-cache attention path.

This module only *builds inputs*: shapes, distributions and seeded random
streams.  It holds none of the method's arithmetic (no projection, no
softmax, no cache append), so both the CUDA path and the CPU oracle can draw
their inputs from it without sharing any computation.

Shapes follow the pages' evaluated models ("Paper Notes: DirectKV",
Experiments & Results: Llama-3.1-8B-shaped layers) and the decode/prefill
split of the Attention Fusion Engine ("Paper Notes: DirectKV", System
Architecture).  No dataset or trained weight is used: x ~ N(0,1),
W ~ N(0, 1/H), cached K/V ~ N(0,1) (or U(-2,2) for the fp16 MHA workload),
rounded to the storage dtype with round-to-nearest-even.

Notation: B batch, T new tokens per sequence (decode: T = 1), P cached
tokens before the call, H hidden, Hq / Hkv query / KV heads, D head_dim.
Layouts: x [B,T,H]; Wq [H, Hq*D]; Wk, Wv [H, Hkv*D] (row-major, K = X.Wk);
K and V caches [B][Hkv][S_max][D], S_max = P + T.
"""
from __future__ import annotations

import dataclasses
import numpy as np

BF16 = "bf16"
FP16 = "fp16"

# Fixed stream ids: one independent PCG64 stream per tensor.
_STREAM = {"x": 1, "wq": 2, "wk": 3, "wv": 4, "k": 5, "v": 6, "spike": 7}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    phase: str            # "decode" or "prefill"
    B: int
    H: int
    Hq: int
    Hkv: int
    D: int
    P: int                # cached tokens before the call
    T: int = 1            # new tokens per sequence
    dtype: str = BF16
    kv_dist: str = "normal"   # "normal" N(0,1) or "uniform2" U(-2,2)
    spike_frac: float = 0.0   # fraction of key rows scaled x8 per (b, kv head)
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def S_max(self) -> int:
        return self.P + self.T

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ---- algorithmic byte / flop counts (per call) -------------------------
    @property
    def esize(self) -> int:
        return 2

    def host_read_bytes(self) -> int:
        """Cached prefix K and V read once across the host link."""
        return 2 * self.B * self.Hkv * self.P * self.D * self.esize

    def host_write_bytes(self) -> int:
        """Appended K and V rows written once across the host link."""
        return 2 * self.B * self.Hkv * self.T * self.D * self.esize

    def attn_pairs(self) -> int:
        """(query, key) pairs per head summed over the batch, causal."""
        T, P = self.T, self.P
        return self.B * (T * P + T * (T + 1) // 2)

    def attn_flops(self) -> int:
        return 4 * self.Hq * self.D * self.attn_pairs()

    def proj_flops(self) -> int:
        return 2 * self.B * self.T * self.H * (self.Hq + 2 * self.Hkv) * self.D

    def flops(self) -> int:
        return self.attn_flops() + self.proj_flops()

    def hbm_min_bytes(self) -> int:
        """Weights + x + out, each touched once (prefill adds Q write+read)."""
        e = self.esize
        w = self.H * (self.Hq + 2 * self.Hkv) * self.D * e
        xo = self.B * self.T * (self.H + self.Hq * self.D) * e
        q = 2 * self.B * self.T * self.Hq * self.D * e if self.phase == "prefill" else 0
        return w + xo + q


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_decode", "decode", B=1, H=512, Hq=8, Hkv=2, D=64, P=2048),
        Workload("llama8b_decode", "decode", B=8, H=4096, Hq=32, Hkv=8, D=128, P=32768),
        Workload("llama8b_prefill", "prefill", B=1, H=4096, Hq=32, Hkv=8, D=128,
                 P=28672, T=4096),
        # a quarter-size chunked prefill (same heads), small enough for a
        # full profiler capture
        Workload("llama8b_prefill_quarter", "prefill", B=1, H=4096, Hq=32, Hkv=8, D=128,
                 P=7168, T=1024),
        Workload("longctx_b1_s16k", "decode", B=1, H=4096, Hq=32, Hkv=8, D=128,
                 P=16384, spike_frac=0.01),
        Workload("longctx_b1_s64k", "decode", B=1, H=4096, Hq=32, Hkv=8, D=128,
                 P=65536, spike_frac=0.01),
        Workload("longctx_b1_s128k", "decode", B=1, H=4096, Hq=32, Hkv=8, D=128,
                 P=131072, spike_frac=0.01),
        Workload("longctx_b4_s16k", "decode", B=4, H=4096, Hq=32, Hkv=8, D=128,
                 P=16384, spike_frac=0.01),
        Workload("longctx_b4_s64k", "decode", B=4, H=4096, Hq=32, Hkv=8, D=128,
                 P=65536, spike_frac=0.01),
        Workload("longctx_b4_s128k", "decode", B=4, H=4096, Hq=32, Hkv=8, D=128,
                 P=131072, spike_frac=0.01),
        Workload("mha_fp16_decode", "decode", B=16, H=2048, Hq=32, Hkv=32, D=64,
                 P=8192, dtype=FP16, kv_dist="uniform2"),
        Workload("mha_fp16_prefill", "prefill", B=2, H=2048, Hq=32, Hkv=32, D=64,
                 P=6144, T=2048, dtype=FP16, kv_dist="uniform2"),
    ]
}


def _rng(seed: int, stream: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _STREAM[stream], sub])))


def to_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> uint16 storage bits, round-to-nearest-even (input construction)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == FP16:
        return a.astype(np.float16).view(np.uint16)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 storage bits -> float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_dense(w: Workload):
    """x, Wq, Wk, Wv as uint16 bit arrays."""
    s = w.seed
    x = _rng(s, "x").standard_normal((w.B, w.T, w.H), dtype=np.float32)
    sd = np.float32(1.0 / np.sqrt(w.H))
    wq = _rng(s, "wq").standard_normal((w.H, w.Hq * w.D), dtype=np.float32) * sd
    wk = _rng(s, "wk").standard_normal((w.H, w.Hkv * w.D), dtype=np.float32) * sd
    wv = _rng(s, "wv").standard_normal((w.H, w.Hkv * w.D), dtype=np.float32) * sd
    return {k: to_bits(v, w.dtype) for k, v in dict(x=x, wq=wq, wk=wk, wv=wv).items()}


def fill_cache(w: Workload, k_out: np.ndarray, v_out: np.ndarray, s_max: int | None = None):
    """Fill rows [0, P) of K and V caches ([B][Hkv][s_max][D] uint16) in place.

    Rows at and beyond P are left untouched (the caller decides their value).
    Each (b, kv head) slice draws from its own sub-stream, so slices can be
    regenerated independently.
    """
    import concurrent.futures as cf
    import os
    s_max = s_max or w.S_max
    k4 = k_out.reshape(w.B, w.Hkv, s_max, w.D)
    v4 = v_out.reshape(w.B, w.Hkv, s_max, w.D)

    def one(bh):
        b, h = divmod(bh, w.Hkv)
        kk, vv = cache_slice(w, b, h)
        k4[b, h, : w.P] = kk
        v4[b, h, : w.P] = vv
    # the slices are independent streams: draw them on several threads
    n = w.B * w.Hkv
    with cf.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1, n))) as ex:
        list(ex.map(one, range(n)))


def cache_slice(w: Workload, b: int, h: int):
    """(K, V) rows [0, P) for sequence b, KV head h, as uint16 bits [P, D]."""
    sub = b * w.Hkv + h
    shape = (w.P, w.D)
    if w.kv_dist == "uniform2":
        kf = _rng(w.seed, "k", sub).uniform(-2.0, 2.0, shape).astype(np.float32)
        vf = _rng(w.seed, "v", sub).uniform(-2.0, 2.0, shape).astype(np.float32)
    else:
        kf = _rng(w.seed, "k", sub).standard_normal(shape, dtype=np.float32)
        vf = _rng(w.seed, "v", sub).standard_normal(shape, dtype=np.float32)
    if w.spike_frac > 0 and w.P > 0:
        n = int(round(w.spike_frac * w.P))
        idx = _rng(w.seed, "spike", sub).choice(w.P, size=n, replace=False)
        kf[idx] *= np.float32(8.0)
    return to_bits(kf, w.dtype), to_bits(vf, w.dtype)


def make_cache(w: Workload):
    """Fresh K, V caches [B,Hkv,S_max,D] (uint16), prefix filled, tail zero."""
    k = np.zeros((w.B, w.Hkv, w.S_max, w.D), np.uint16)
    v = np.zeros_like(k)
    fill_cache(w, k, v)
    return k, v


def small(name: str, **kw) -> Workload:
    """A named workload shrunk for oracle-speed tests (keeps heads/dtype)."""
    return WORKLOADS[name].with_(**kw)
