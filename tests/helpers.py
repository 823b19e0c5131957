"""Shared test plumbing: build a cache from a seeded workload, run the CUDA
path through the C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np

from zero_copy_offloaded_gb300 import workloads as wl

# Tolerances on the attention output versus the fp64 oracle: maximum absolute
# error and sum|gpu - ref| / sum|ref|.
MAX_ABS = 1e-2
MEAN_REL = 2e-3


def torch_dtype(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float16


def to_dev(bits: np.ndarray, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).cuda()


def to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def out_f64(t, dtype) -> np.ndarray:
    import oracle
    return oracle.decode_bits(to_bits(t), dtype)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in representable steps between two arrays of 16-bit float bits."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


# Tally of every projection comparison in this session (printed by conftest's
# terminal summary): elements, bit-exact, within 1 ulp, and those accepted
# only through the fp32 summation bound.
PROJECTION_TALLY = {"elements": 0, "bit_exact": 0, "within_1ulp": 0, "fp32_bound_only": 0,
                    "max_cancellation_ratio": 0.0}


def storage_ulp(v: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the 16-bit storage format at |v| (subnormal spacing below the
    smallest normal)."""
    p, emin = (8, -126) if dtype == "bf16" else (11, -14)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - (p - 1))


def assert_projection_close(got_bits, x_bits, w_bits, dtype, what=""):
    """A tensor-core projection against the oracle's fp32-sequential one.

    got_bits [rows, N], x_bits [rows, K], w_bits [K, N].  Each element is
    within 1 ulp of the oracle's, or within the fp32 summation error bound
    K * 2^-24 * sum|x_j w_j| (plus half an ulp) of the exact sum.  The second
    case is allowed only where the sum nearly cancels: any two fp32 sums of
    the same products lie within that bound of the exact sum, so their
    roundings can be more than 1 ulp apart only if the bound reaches a
    quarter of the storage ulp at the exact sum, i.e. |exact| is small next
    to sum|x_j w_j|.  Every element accepted that way is checked to be such a
    near-cancellation and counted.  Returns (bit-exact fraction, within-1-ulp
    fraction, number accepted only through the bound)."""
    import oracle
    ref, exact = oracle.project(x_bits, w_bits, dtype, exact=True)
    xf, wf = oracle.decode_bits(x_bits, dtype), oracle.decode_bits(w_bits, dtype)
    mag = np.abs(xf) @ np.abs(wf)
    bound = x_bits.shape[1] * 2.0 ** -24 * mag
    d = ulp_distance(got_bits, ref)
    g = oracle.decode_bits(got_bits, dtype)
    half_ulp = np.abs(g) * (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) + 1e-30
    near = d <= 1
    in_bound = np.abs(g - exact) <= bound + half_ulp
    ok = near | in_bound
    assert ok.all(), f"{what}: {(~ok).sum()} elements beyond 1 ulp and the fp32 error bound"
    fallback = ~near
    if fallback.any():
        cancels = bound[fallback] >= storage_ulp(exact[fallback], dtype) / 4
        assert cancels.all(), (
            f"{what}: {(~cancels).sum()} elements beyond 1 ulp where the sum does not cancel")
        ratio = float(np.max(np.abs(exact[fallback]) / np.maximum(mag[fallback], 1e-300)))
        PROJECTION_TALLY["max_cancellation_ratio"] = max(
            PROJECTION_TALLY["max_cancellation_ratio"], ratio)
    n_fb = int(fallback.sum())
    PROJECTION_TALLY["elements"] += int(d.size)
    PROJECTION_TALLY["bit_exact"] += int((d == 0).sum())
    PROJECTION_TALLY["within_1ulp"] += int(near.sum())
    PROJECTION_TALLY["fp32_bound_only"] += n_fb
    return float(np.mean(d == 0)), float(np.mean(near)), n_fb


def errors(got: np.ndarray, ref: np.ndarray):
    d = np.abs(got - ref)
    return float(d.max()), float(d.sum() / max(np.abs(ref).sum(), 1e-300))


def assert_close(got, ref, what=""):
    mx, mr = errors(got, ref)
    assert mx <= MAX_ABS and mr <= MEAN_REL, f"{what}: max_abs={mx:.3e} mean_rel={mr:.3e}"
    return mx, mr


def assert_close_beyond_rounding(got, ref, dtype, what=""):
    """The bars on the part of the error that the output's own rounding to
    `dtype` does not explain: |got - ref| - |round(ref) - ref| <= MAX_ABS and
    sum|got - ref| / sum|ref| <= MEAN_REL.

    For outputs of magnitude 4 and more a bf16 result is off the fp64 value
    by up to 2^-6 > MAX_ABS even when correctly rounded, so a flat max-abs bar
    cannot hold there; where |ref| < 2 (bf16) the two checks coincide to
    within 2^-8."""
    import oracle
    rounded = oracle.decode_bits(oracle.round_bits(ref, dtype), dtype)
    excess = np.abs(got - ref) - np.abs(rounded - ref)
    mx, mr = errors(got, ref)
    assert excess.max() <= MAX_ABS and mr <= MEAN_REL, (
        f"{what}: max_abs beyond rounding={excess.max():.3e} (raw {mx:.3e}) mean_rel={mr:.3e}")
    return float(excess.max()), mr


class Case:
    """A workload materialised on the GPU and in the host cache."""

    def __init__(self, w: wl.Workload, lens=None, s_max=None, tuning=None, page_tokens=0,
                 spare_pages=3, table_seed=0, kv_format="native"):
        """page_tokens > 0 builds a paged cache: the logical rows of every
        sequence go to pool pages drawn by a seeded permutation (spare pages
        stay in no table and hold the spare canary).  kv_format "e4m3": the
        prefix rows are the workload's values rounded to E4M3 (uint8 bits)."""
        import zero_copy_offloaded_gb300 as dkv
        self.w = w
        self.kv_format = kv_format
        fp8 = kv_format == "e4m3"
        self.canary = 0x5A if fp8 else 0x7E57       # rows past the append
        self.spare_canary = 0x33 if fp8 else 0x5A5A  # pool pages in no table
        el = np.uint8 if fp8 else np.uint16
        self.dense = wl.make_dense(w)
        self.s_max = s_max or w.S_max
        self.lens = np.broadcast_to(np.asarray(w.P if lens is None else lens, np.int64),
                                    (w.B,)).copy()
        self.page_tokens = page_tokens
        if page_tokens:
            npg = -(-self.s_max // page_tokens)
            self.s_max = npg * page_tokens
            perm = np.random.default_rng(table_seed).permutation(w.B * npg + spare_pages)
            self.table = perm[:w.B * npg].reshape(w.B, npg).astype(np.int32)
            self.spare = perm[w.B * npg:]
            self.cache = dkv.PagedKVCache(w.B, w.Hkv, w.D, page_tokens, len(perm), npg, w.dtype,
                                          kv_format)
            self.cache.k_host[...] = self.spare_canary
            self.cache.v_host[...] = self.spare_canary
            self.cache.set_page_table(self.table)
        else:
            self.cache = dkv.KVCache(w.B, w.Hkv, w.D, self.s_max, w.dtype, kv_format)
        # prefix rows: the workload's generator, truncated per sequence
        kc = np.zeros((w.B, w.Hkv, self.s_max, w.D), el)
        vc = np.zeros_like(kc)
        wp = w.with_(P=int(self.lens.max()))
        for b in range(w.B):
            for h in range(w.Hkv):
                kk, vv = wl.cache_slice(wp, b, h)
                if fp8:
                    import oracle
                    kk = oracle.round_e4m3(wl.bits_to_f32(kk, w.dtype).astype(np.float64))
                    vv = oracle.round_e4m3(wl.bits_to_f32(vv, w.dtype).astype(np.float64))
                n = int(self.lens[b])
                kc[b, h, :n] = kk[:n]
                vc[b, h, :n] = vv[:n]
        # canary pattern beyond the prefix: must be overwritten only by appends
        kc[:, :, :, :][np.broadcast_to(np.arange(self.s_max)[None, None, :, None]
                                       >= self.lens[:, None, None, None], kc.shape)] = self.canary
        vc[np.broadcast_to(np.arange(self.s_max)[None, None, :, None]
                           >= self.lens[:, None, None, None], vc.shape)] = self.canary
        if page_tokens:
            self._scatter(self.cache.k_host, kc)
            self._scatter(self.cache.v_host, vc)
        else:
            self.cache.k_host[...] = kc
            self.cache.v_host[...] = vc
        self.k0, self.v0 = kc, vc
        self.cache.set_lengths(self.lens.astype(np.int32))
        if tuning:
            dkv.dkv_cache_set_tuning(self.cache.h, **tuning)
        self.x = to_dev(self.dense["x"], w.dtype)
        self.wq = to_dev(self.dense["wq"], w.dtype)
        self.wk = to_dev(self.dense["wk"], w.dtype)
        self.wv = to_dev(self.dense["wv"], w.dtype)

    def _scatter(self, pool, logical):
        pt = self.page_tokens
        for b in range(self.w.B):
            for i, pg in enumerate(self.table[b]):
                pool[pg] = logical[b, :, i * pt:(i + 1) * pt]

    def _gather(self, pool):
        pt = self.page_tokens
        out = np.empty((self.w.B, self.w.Hkv, self.s_max, self.w.D), pool.dtype)
        for b in range(self.w.B):
            for i, pg in enumerate(self.table[b]):
                out[b, :, i * pt:(i + 1) * pt] = pool[pg]
        return out

    def k_logical(self):
        """The K cache as [B, Hkv, s_max, D] rows (gathered through the page table)."""
        return self._gather(self.cache.k_host) if self.page_tokens else self.cache.k_host

    def v_logical(self):
        return self._gather(self.cache.v_host) if self.page_tokens else self.cache.v_host

    def spare_pages_untouched(self):
        if not self.page_tokens:
            return True
        return bool(np.all(self.cache.k_host[self.spare] == self.spare_canary) and
                    np.all(self.cache.v_host[self.spare] == self.spare_canary))

    def out_tensor(self, T):
        import torch
        w = self.w
        return torch.empty((w.B, T, w.Hq, w.D), dtype=torch_dtype(w.dtype), device="cuda")

    def run_decode(self, x=None):
        out = self.out_tensor(1)
        x = self.x if x is None else x
        self.cache.decode(x.reshape(self.w.B, 1, self.w.H), self.wq, self.wk, self.wv, self.w.Hq,
                          out)
        self.cache.sync()
        return out

    def run_prefill(self, x=None):
        x = self.x if x is None else x
        out = self.out_tensor(x.shape[1])
        self.cache.prefill(x, self.wq, self.wk, self.wv, self.w.Hq, out)
        self.cache.sync()
        return out

    def oracle(self, x_bits=None, rows=None, k=None, v=None, lens=None):
        import oracle
        w = self.w
        return oracle.step(self.dense["x"] if x_bits is None else x_bits, self.dense["wq"],
                           self.dense["wk"], self.dense["wv"], self.k0 if k is None else k,
                           self.v0 if v is None else v, self.lens if lens is None else lens,
                           w.Hq, w.dtype, rows=rows,
                           kv_format="e4m3" if self.kv_format == "e4m3" else None)

    def free(self):
        self.cache.free()
