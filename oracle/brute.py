"""Pure-Python brute force for tiny shapes: the independent pin of the C oracle.

TEST INFRASTRUCTURE ONLY.  Written from the definitions on "Paper Notes:
DirectKV" (Kernel Fusion: K = X.Wk, V = X.Wv, softmax(Q.K^T/sqrt(d)).V) with
Python floats, fractions and explicit loops; shares nothing with
``dkv_oracle.c``.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def _fmt(dtype):
    # (exponent bits, stored mantissa bits)
    return (8, 7) if dtype in ("bf16", 0) else (5, 10)


def value_of(bits: int, dtype) -> Fraction | float:
    """Exact value of a 16-bit pattern as a Fraction (inf/nan as float)."""
    eb, mb = _fmt(dtype)
    bias = (1 << (eb - 1)) - 1
    s = -1 if bits >> 15 else 1
    e = (bits >> mb) & ((1 << eb) - 1)
    m = bits & ((1 << mb) - 1)
    if e == (1 << eb) - 1:
        return s * math.inf if m == 0 else math.nan
    if e == 0:
        return s * Fraction(m, 1) * Fraction(2) ** (1 - bias - mb)
    return s * Fraction(m + (1 << mb)) * Fraction(2) ** (e - bias - mb)


_TABLE = {}


def _finite_table(dtype):
    """All finite non-negative values with their bit patterns, sorted."""
    key = 0 if dtype in ("bf16", 0) else 1
    if key not in _TABLE:
        eb, mb = _fmt(dtype)
        vals = []
        for bits in range(0, 1 << 15):
            v = value_of(bits, dtype)
            if isinstance(v, Fraction) or v == 0:
                vals.append((Fraction(v), bits))
        vals.sort()
        _TABLE[key] = vals
    return _TABLE[key]


def nearest_bits(v, dtype) -> int:
    """Nearest representable value to v by enumeration; ties go to the even
    significand (even bit pattern); beyond max + half an ulp -> infinity."""
    import bisect

    eb, mb = _fmt(dtype)
    x = Fraction(v)
    sign = 0x8000 if (x < 0 or (x == 0 and math.copysign(1.0, float(v)) < 0)) else 0
    a = abs(x)
    table = _finite_table(dtype)
    vals = [t[0] for t in table]
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return sign | table[i][1]
    if i == len(vals):
        # above the largest finite: overflow threshold is max + ulp/2
        top, top_bits = table[-1]
        ulp = top - table[-2][0]
        if a >= top + ulp / 2:
            return sign | (((1 << eb) - 1) << mb)
        return sign | top_bits
    lo, lo_bits = table[i - 1]
    hi, hi_bits = table[i]
    dlo, dhi = a - lo, hi - a
    if dlo < dhi:
        return sign | lo_bits
    if dhi < dlo:
        return sign | hi_bits
    return sign | (lo_bits if lo_bits % 2 == 0 else hi_bits)


def e4m3_value(bits: int):
    """Exact value of an 8-bit E4M3 pattern (1 sign, 4 exponent bits with bias
    7, 3 mantissa bits; no infinities; exponent and mantissa all ones is NaN)."""
    s = -1 if bits & 0x80 else 1
    e = (bits >> 3) & 15
    m = bits & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * Fraction(m, 8) * Fraction(2) ** -6
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def e4m3_nearest(v) -> int:
    """Nearest E4M3 pattern by enumeration of the finite codes; ties go to the
    even mantissa; magnitudes past the largest finite value saturate to it."""
    x = Fraction(v)
    neg = x < 0 or (x == 0 and math.copysign(1.0, float(v)) < 0)
    a = abs(x)
    best = None
    for bits in range(0, 0x7F):  # non-negative finite codes
        d = abs(e4m3_value(bits) - a)
        if best is None or d < best[0] or (d == best[0] and bits % 2 == 0):
            best = (d, bits)
    top = 0x7E  # 448
    bits = top if a > e4m3_value(top) else best[1]
    return (0x80 | bits) if neg else bits


def f32_sums_seq(x_bits, w_bits, dtype):
    """x [H] bits, w [H][N] bits -> [N] floats: the fp32 sequential sums (unrounded)."""
    H = len(x_bits)
    N = len(w_bits[0])
    out = []
    for c in range(N):
        acc = 0.0
        for j in range(H):
            p = float(value_of(x_bits[j], dtype)) * float(value_of(w_bits[j][c], dtype))
            acc = f32(acc + p)
        out.append(acc)
    return out


def f32(x) -> float:
    """Round a Python float to the nearest IEEE single (ties to even)."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def project_seq_f32(x_bits, w_bits, dtype):
    """x [H] bits, w [H][N] bits -> [N] bits: fp32 sequential sum of exact products."""
    H = len(x_bits)
    N = len(w_bits[0])
    out = []
    for c in range(N):
        acc = 0.0
        for j in range(H):
            p = float(value_of(x_bits[j], dtype)) * float(value_of(w_bits[j][c], dtype))
            acc = f32(acc + p)
        out.append(nearest_bits(acc, dtype))
    return out


def project_exact(x_bits, w_bits, dtype):
    """Exact rational sum of products, per output column."""
    H = len(x_bits)
    N = len(w_bits[0])
    return [sum(value_of(x_bits[j], dtype) * value_of(w_bits[j][c], dtype) for j in range(H))
            for c in range(N)]


def attend(K, V, q, n_visible):
    """Per-element softmax attention with math.exp; K, V lists of [D] rows."""
    D = len(q)
    scale = 1.0 / math.sqrt(D)
    s = []
    for j in range(n_visible):
        dot = 0.0
        for d in range(D):
            dot += q[d] * K[j][d]
        s.append(dot * scale)
    m = max(s)
    e = [math.exp(v - m) for v in s]
    z = sum(e)
    o = [0.0] * D
    for j in range(n_visible):
        w = e[j] / z
        for d in range(D):
            o[d] += w * V[j][d]
    return o, [v / z for v in e]
