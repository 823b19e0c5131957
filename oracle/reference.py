"""ctypes wrapper around the fp64 C oracle, plus the end-to-end oracle step.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The end-to-end step follows "Paper Notes: DirectKV" (System Architecture,
KV Cache Manager and Attention Fusion Engine; Fundamental Underlying
Technologies, Kernel Fusion), in this order:
  1. q = x.Wq, k = x.Wk, v = x.Wv, each output accumulated in fp32 in
     sequential order and rounded once to the storage dtype;
  2. the new k, v rows are appended to the cache at rows [P, P+T);
  3. every query (absolute position P+t) attends in fp64 to keys 0..P+t of
     its KV head with softmax(q.k / sqrt(D)).v.
Query head h uses KV head h // G (contiguous groups; the pages do not fix
the mapping).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16 = 0
FP16 = 1
_DT = {"bf16": BF16, "fp16": FP16, BF16: BF16, FP16: FP16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libdkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
               "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L.dkv_oracle_decode.argtypes = [P, ctypes.c_int64, ctypes.c_int, P]
            L.dkv_oracle_round.argtypes = [P, ctypes.c_int64, ctypes.c_int, P]
            L.dkv_oracle_project.argtypes = [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                                             ctypes.c_int, P, P, P]
            L.dkv_oracle_decode_e4m3.argtypes = [P, ctypes.c_int64, P]
            L.dkv_oracle_round_e4m3.argtypes = [P, ctypes.c_int64, P]
            L.dkv_oracle_attend.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int, P, P,
                                            P, P, P]
            L.dkv_oracle_attend.restype = ctypes.c_int
            L.dkv_oracle_set_threads.argtypes = [ctypes.c_int]
            L.dkv_oracle_max_threads.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def set_threads(n: int) -> None:
    lib().dkv_oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().dkv_oracle_max_threads())


def decode_bits(bits: np.ndarray, dtype) -> np.ndarray:
    """uint16 storage bits -> exact float64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().dkv_oracle_decode(_p(b), b.size, _DT[dtype], _p(out))
    return out


def round_bits(v: np.ndarray, dtype) -> np.ndarray:
    """float64 values -> uint16 bits of the nearest bf16/fp16 (ties to even)."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, np.uint16)
    lib().dkv_oracle_round(_p(a), a.size, _DT[dtype], _p(out))
    return out


def project(x_bits: np.ndarray, w_bits: np.ndarray, dtype, exact: bool = False):
    """Y = X.W with fp32 sequential accumulation rounded to dtype.

    x_bits [rows, H], w_bits [H, N] uint16.  Returns uint16 [rows, N]
    (and the fp64 sum [rows, N] if exact)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    rows, H = x.shape
    H2, N = w.shape
    assert H == H2
    out = np.empty((rows, N), np.uint16)
    ex = np.empty((rows, N), np.float64) if exact else None
    lib().dkv_oracle_project(_p(x), rows, H, _p(w), N, _DT[dtype], _p(out), _p(ex), None)
    return (out, ex) if exact else out


def project_f32(x_bits: np.ndarray, w_bits: np.ndarray, dtype) -> np.ndarray:
    """The fp32 sequential sums of project() before their rounding (float64 holding
    fp32 values), for storage formats other than the inputs' dtype."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    rows, H = x.shape
    H2, N = w.shape
    assert H == H2
    f = np.empty((rows, N), np.float64)
    lib().dkv_oracle_project(_p(x), rows, H, _p(w), N, _DT[dtype], None, None, _p(f))
    return f


def decode_e4m3(bits: np.ndarray) -> np.ndarray:
    """uint8 E4M3 bits -> exact float64 values (NaN for the NaN codes)."""
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, np.float64)
    lib().dkv_oracle_decode_e4m3(_p(b), b.size, _p(out))
    return out


def round_e4m3(v: np.ndarray) -> np.ndarray:
    """float64 values -> uint8 bits of the nearest E4M3 value (ties to even),
    saturating at +-448."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, np.uint8)
    lib().dkv_oracle_round_e4m3(_p(a), a.size, _p(out))
    return out


def attend(K: np.ndarray, V: np.ndarray, Q: np.ndarray, pos, want_lse=False, want_weights=False):
    """fp64 softmax attention of Q rows [nq, D] over K, V [S, D]; row i sees keys 0..pos[i]."""
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    Q = np.ascontiguousarray(Q, dtype=np.float64).reshape(-1, K.shape[1])
    pos = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, np.int32), (Q.shape[0],)), dtype=np.int32)
    S, D = K.shape
    nq = Q.shape[0]
    out = np.empty((nq, D), np.float64)
    lse = np.empty(nq, np.float64) if want_lse else None
    wts = np.empty((nq, S), np.float64) if want_weights else None
    rc = lib().dkv_oracle_attend(D, S, _p(K), _p(V), nq, _p(Q), _p(pos), _p(out), _p(lse), _p(wts))
    if rc != 0:
        raise ValueError("query position outside the cache")
    res = [out]
    if want_lse:
        res.append(lse)
    if want_weights:
        res.append(wts)
    return res[0] if len(res) == 1 else tuple(res)


def step(x, wq, wk, wv, k_cache, v_cache, P, n_q_heads, dtype, rows=None, kv_format=None):
    """One decode/prefill call of the method, on the oracle.

    kv_format "e4m3": the caches hold 8-bit E4M3 bits (uint8) and the new K/V
    rows are the fp32 sums rounded once to E4M3; q stays in dtype.

    x [B,T,H] bits; wq [H,Hq*D]; wk, wv [H,Hkv*D]; k_cache, v_cache
    [B,Hkv,S_max,D] bits with rows [0,P) filled (P an int or per-sequence
    list).  rows: optional list of (b, t) query rows to attend (all if None).

    Returns dict: out {(b,t): [Hq,D] fp64} or [B,T,Hq,D] array when rows is
    None; k_new, v_new [B,T,Hkv,D] bits; q [B,T,Hq,D] bits; k_cache_after,
    v_cache_after (copies with the append applied).
    """
    B, T, H = x.shape
    _, Hkv, S_max, D = k_cache.shape
    Hq = n_q_heads
    G = Hq // Hkv
    Ps = np.broadcast_to(np.asarray(P, np.int64), (B,))
    xr = x.reshape(B * T, H)
    q = project(xr, wq, dtype).reshape(B, T, Hq, D)
    fp8 = kv_format == "e4m3"
    if fp8:
        k_new = round_e4m3(project_f32(xr, wk, dtype)).reshape(B, T, Hkv, D)
        v_new = round_e4m3(project_f32(xr, wv, dtype)).reshape(B, T, Hkv, D)
        kv_decode = decode_e4m3
    else:
        k_new = project(xr, wk, dtype).reshape(B, T, Hkv, D)
        v_new = project(xr, wv, dtype).reshape(B, T, Hkv, D)

        def kv_decode(bits):
            return decode_bits(bits, dtype)
    kc = k_cache.copy()
    vc = v_cache.copy()
    for b in range(B):
        p = int(Ps[b])
        if p + T > S_max:
            raise ValueError("cache capacity exceeded")
        kc[b, :, p:p + T] = k_new[b].transpose(1, 0, 2)
        vc[b, :, p:p + T] = v_new[b].transpose(1, 0, 2)
    want = [(b, t) for b in range(B) for t in range(T)] if rows is None else list(rows)
    outs = {}
    by_b = {}
    for (b, t) in want:
        by_b.setdefault(b, []).append(t)
    for b, ts in by_b.items():
        p = int(Ps[b])
        for kvh in range(Hkv):
            Kf = kv_decode(kc[b, kvh, : p + T])
            Vf = kv_decode(vc[b, kvh, : p + T])
            heads = list(range(kvh * G, (kvh + 1) * G))
            Qr = decode_bits(q[b][np.ix_(ts, heads)], dtype).reshape(-1, D)
            pos = np.repeat(np.asarray([p + t for t in ts], np.int32), G)
            o = attend(Kf, Vf, Qr, pos).reshape(len(ts), G, D)
            for i, t in enumerate(ts):
                outs.setdefault((b, t), np.zeros((Hq, D)))[kvh * G:(kvh + 1) * G] = o[i]
    if rows is None:
        out = np.zeros((B, T, Hq, D))
        for (b, t), o in outs.items():
            out[b, t] = o
    else:
        out = outs
    return dict(out=out, q=q, k_new=k_new, v_new=v_new, k_cache_after=kc, v_cache_after=vc)
