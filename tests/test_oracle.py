"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle fails it: a wrong
rounding rule (enumeration, golden ties), an fp64 instead of fp32 sum
(golden 'fp32_sequential_not_exact'), a wrong scale (golden
'scale_is_inverse_sqrt_d'), an off-by-one in the causal bound (golden
'causal_prefix_two_keys', brute force), a transposed operand (non-square
brute-force shapes), a wrong GQA mapping (GQA == repeated-KV MHA) and a
wrong append position (cache invariants, prefill == successive decodes).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import brute
from zero_copy_offloaded_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _num(v):
    if isinstance(v, (int, float)):
        return float(v)
    env = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln7": math.log(7)}
    if "/" in v and "*" not in v:
        a, b = v.split("/")
        return float(Fraction(int(a), int(b)))
    return float(eval(v, {"__builtins__": {}}, env))


# ---------------------------------------------------------------- rounding --

@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_decode_all_patterns(dt):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode_bits(bits, dt)
    for b in range(0, 1 << 16, 7):
        ref = brute.value_of(b, dt)
        if isinstance(ref, float) and math.isnan(ref):
            assert math.isnan(got[b])
        else:
            assert got[b] == float(ref), (dt, b)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_round_vs_enumeration(dt):
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(300) * 10.0 ** rng.integers(-9, 6, 300))
    # exact midpoints between neighbours -> ties
    for b in rng.integers(1, 0x7B00, 200):
        lo = brute.value_of(int(b), dt)
        hi = brute.value_of(int(b) + 1, dt)
        if isinstance(lo, Fraction) and isinstance(hi, Fraction):
            vals.append(float((lo + hi) / 2))
            vals.append(-float((lo + hi) / 2))
    big = 3.0e38 if dt == "bf16" else 65504.0
    vals += [0.0, -0.0, big, -big, big * 1.01, 1e-45, 2.0 ** -134, 2.0 ** -25, 65520.0, 65519.0]
    v = np.array(vals, np.float64)
    got = oracle.round_bits(v, dt)
    ref = [brute.nearest_bits(float(x), dt) for x in v]
    assert list(got) == ref


def test_round_matches_library_routines():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 5, 20000)
    # numpy float64 -> float16 is correctly rounded
    assert np.array_equal(oracle.round_bits(v, "fp16"), v.astype(np.float16).view(np.uint16))
    torch = pytest.importorskip("torch")
    f32 = v.astype(np.float32)
    tb = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bits(f32.astype(np.float64), "bf16"), tb)


def test_e4m3_decode_all_codes():
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(bits)
    for b in range(256):
        ref = brute.e4m3_value(b)
        if isinstance(ref, float) and math.isnan(ref):
            assert math.isnan(got[b]), b
        else:
            assert got[b] == float(ref), b
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_e4m3_round_vs_enumeration():
    rng = np.random.default_rng(17)
    vals = list(rng.standard_normal(400) * 2.0 ** rng.integers(-12, 10, 400))
    for b in range(0, 0x7E):  # every midpoint between neighbouring finite codes: ties
        lo, hi = brute.e4m3_value(b), brute.e4m3_value(b + 1)
        vals += [float((lo + hi) / 2), -float((lo + hi) / 2)]
    vals += [0.0, -0.0, 448.0, 447.9, 460.0, 464.0, 465.0, 1e6, -1e6, 2.0 ** -10, 2.0 ** -11]
    v = np.array(vals, np.float64)
    got = oracle.round_e4m3(v)
    assert list(got) == [brute.e4m3_nearest(float(x)) for x in v]


def test_project_f32_vs_bruteforce():
    rng = np.random.default_rng(23)
    H, N = 29, 4
    x = wl.to_bits(rng.standard_normal((2, H)).astype(np.float32), "bf16")
    w = wl.to_bits((rng.standard_normal((H, N)) / 5).astype(np.float32), "bf16")
    got = oracle.project_f32(x, w, "bf16")
    for r in range(2):
        ref = brute.f32_sums_seq(list(map(int, x[r])), [list(map(int, row)) for row in w], "bf16")
        assert list(got[r]) == ref
    # rounding the sums to the storage dtype is project() itself
    assert np.array_equal(oracle.round_bits(got, "bf16"), oracle.project(x, w, "bf16"))


def test_step_e4m3_cache():
    """With E4M3 caches the appended rows are the fp32 sums rounded to E4M3, and
    the attention runs over the decoded E4M3 values (checked against a step
    over the same values held in fp64 by hand)."""
    w = wl.Workload("t", "decode", B=1, H=32, Hq=4, Hkv=2, D=8, P=5, seed=3)
    d = wl.make_dense(w)
    rng = np.random.default_rng(4)
    kc = oracle.round_e4m3(rng.standard_normal((1, 2, 8, 8)))
    vc = oracle.round_e4m3(rng.standard_normal((1, 2, 8, 8)))
    ref = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], kc, vc, 5, 4, "bf16", kv_format="e4m3")
    xr = d["x"].reshape(1, 32)
    kn = oracle.round_e4m3(oracle.project_f32(xr, d["wk"], "bf16")).reshape(2, 8)
    assert np.array_equal(ref["k_new"][0, 0], kn)
    assert np.array_equal(ref["k_cache_after"][0, :, 5], kn)
    q = oracle.decode_bits(oracle.project(xr, d["wq"], "bf16"), "bf16").reshape(4, 8)
    K = oracle.decode_e4m3(ref["k_cache_after"][0])
    V = oracle.decode_e4m3(ref["v_cache_after"][0])
    for h in range(4):
        o, _ = brute.attend([list(r) for r in K[h // 2, :6]], [list(r) for r in V[h // 2, :6]],
                            list(q[h]), 6)
        np.testing.assert_allclose(ref["out"][0, 0, h], o, rtol=0, atol=1e-12)


# -------------------------------------------------------------- projection --

def test_project_golden():
    for case in json.load(open(GOLDEN))["project"]:
        x = np.array([case["x_bits"]], np.uint16)
        w = np.array(case["w_bits"], np.uint16)
        got, ex = oracle.project(x, w, case["dtype"], exact=True)
        assert list(got[0]) == case["out_bits"], case["name"]
        assert list(oracle.round_bits(ex[0], case["dtype"])) == case["exact_bits"], case["name"]


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_project_vs_bruteforce(dt):
    rng = np.random.default_rng(3)
    rows, H, N = 3, 37, 5
    x = wl.to_bits(rng.standard_normal((rows, H)).astype(np.float32), dt)
    w = wl.to_bits((rng.standard_normal((H, N)) / 6).astype(np.float32), dt)
    got, ex = oracle.project(x, w, dt, exact=True)
    for r in range(rows):
        seq = brute.project_seq_f32(list(map(int, x[r])), [list(map(int, row)) for row in w], dt)
        assert list(got[r]) == seq
        exact = brute.project_exact(list(map(int, x[r])), [list(map(int, row)) for row in w], dt)
        for c in range(N):
            assert abs(ex[r, c] - float(exact[c])) <= 1e-12 * max(1.0, abs(float(exact[c])))
            # fp32 sequential and exact sums round to the same or adjacent values
            eb = brute.nearest_bits(exact[c], dt)
            assert abs(int(got[r, c]) - eb) <= 1 or (got[r, c] & 0x7FFF) + (eb & 0x7FFF) <= 1


# --------------------------------------------------------------- attention --

def test_attend_golden():
    for case in json.load(open(GOLDEN))["attend"]:
        K = np.array([[_num(v) for v in r] for r in case["K"]])
        V = np.array([[_num(v) for v in r] for r in case["V"]])
        q = np.array([[_num(v) for v in case["q"]]])
        out, lse = oracle.attend(K, V, q, [case["pos"]], want_lse=True)
        np.testing.assert_allclose(out[0], [_num(v) for v in case["out"]], rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        assert abs(lse[0] - _num(case["lse"])) < 1e-12, case["name"]


def test_attend_vs_bruteforce():
    rng = np.random.default_rng(7)
    for D, S in [(4, 1), (4, 9), (8, 16), (6, 13)]:
        K = rng.standard_normal((S, D)) * 2
        V = rng.standard_normal((S, D))
        Q = rng.standard_normal((5, D)) * 2
        pos = rng.integers(0, S, 5)
        out, wts = oracle.attend(K, V, Q, pos, want_weights=True)
        for i in range(5):
            o, w = brute.attend(K.tolist(), V.tolist(), Q[i].tolist(), int(pos[i]) + 1)
            np.testing.assert_allclose(out[i], o, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(wts[i, : pos[i] + 1], w, rtol=1e-12, atol=1e-15)
            assert np.all(wts[i, pos[i] + 1:] == 0)


def test_attend_closed_forms():
    rng = np.random.default_rng(9)
    S, D = 50, 16
    K = rng.standard_normal((S, D))
    V = rng.standard_normal((S, D))
    # Q = 0: uniform weights -> mean of the visible V rows
    for p in [0, 7, 49]:
        out = oracle.attend(K, V, np.zeros((1, D)), [p])
        np.testing.assert_allclose(out[0], V[: p + 1].mean(0), rtol=1e-12, atol=1e-14)
    # one visible key -> exactly v_0
    out = oracle.attend(K, V, rng.standard_normal((3, D)) * 5, [0, 0, 0])
    np.testing.assert_array_equal(out, np.repeat(V[:1], 3, 0))
    # constant V -> that constant
    Vc = np.tile(rng.standard_normal(D), (S, 1))
    out = oracle.attend(K, Vc, rng.standard_normal((4, D)), [3, 10, 20, 49])
    np.testing.assert_allclose(out, np.tile(Vc[0], (4, 1)), rtol=1e-12)
    # weights sum to 1; a dominant key takes (almost) all the weight
    Q = rng.standard_normal((6, D))
    _, w = oracle.attend(K, V, Q, [49] * 6, want_weights=True)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)
    Kd = K.copy()
    Kd[17] = Q[0] * 40
    out = oracle.attend(Kd, V, Q[:1], [49])
    np.testing.assert_allclose(out[0], V[17], atol=1e-9)


# ------------------------------------------------------- end-to-end step --

def _small(name, **kw):
    return wl.small(name, **kw)


def test_step_cache_invariants():
    w = _small("tiny_decode", H=64, P=20, T=3)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    k[..., w.P + w.T:, :] = 0xABCD  # nothing lives there (S_max == P + T)
    r = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    ka, va = r["k_cache_after"], r["v_cache_after"]
    assert np.array_equal(ka[:, :, : w.P], k[:, :, : w.P])
    assert np.array_equal(va[:, :, : w.P], v[:, :, : w.P])
    assert np.array_equal(ka[:, :, w.P: w.P + w.T], r["k_new"].transpose(0, 2, 1, 3))
    assert np.array_equal(va[:, :, w.P: w.P + w.T], r["v_new"].transpose(0, 2, 1, 3))
    assert np.array_equal(r["k_new"].reshape(-1, w.Hkv * w.D),
                          oracle.project(d["x"].reshape(-1, w.H), d["wk"], w.dtype))


def test_step_gqa_equals_repeated_kv_mha():
    w = _small("tiny_decode", H=32, P=12, T=2, Hq=4, Hkv=2, D=8)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    G = w.G
    # MHA with every KV head repeated G times (weights columns and cache heads)
    rep = lambda a: np.repeat(a.reshape(w.H, w.Hkv, w.D), G, axis=1).reshape(w.H, -1)
    k2 = np.repeat(k, G, axis=1)
    v2 = np.repeat(v, G, axis=1)
    r1 = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    r2 = oracle.step(d["x"], d["wq"], rep(d["wk"]), rep(d["wv"]), k2, v2, w.P, w.Hq, w.dtype)
    np.testing.assert_array_equal(r1["out"], r2["out"])


def test_step_prefill_equals_successive_decodes():
    w = _small("tiny_decode", H=48, P=10, T=4, Hq=4, Hkv=2, D=8)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    r = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    kc, vc = k.copy(), v.copy()
    for t in range(w.T):
        rt = oracle.step(d["x"][:, t:t + 1], d["wq"], d["wk"], d["wv"], kc, vc, w.P + t, w.Hq,
                         w.dtype)
        np.testing.assert_allclose(rt["out"][:, 0], r["out"][:, t], rtol=1e-13, atol=1e-15)
        kc, vc = rt["k_cache_after"], rt["v_cache_after"]
    assert np.array_equal(kc, r["k_cache_after"]) and np.array_equal(vc, r["v_cache_after"])


def test_step_decode_key_permutation_invariance():
    w = _small("tiny_decode", H=32, P=30, Hq=4, Hkv=1, D=8)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    perm = np.random.default_rng(1).permutation(w.P)
    kp, vp = k.copy(), v.copy()
    kp[:, :, : w.P] = k[:, :, perm]
    vp[:, :, : w.P] = v[:, :, perm]
    r1 = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    r2 = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], kp, vp, w.P, w.Hq, w.dtype)
    np.testing.assert_allclose(r1["out"], r2["out"], rtol=1e-12, atol=1e-14)


def test_step_rows_subset_matches_full():
    w = _small("llama8b_prefill", H=64, P=40, T=6, Hq=4, Hkv=2, D=16)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    full = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype)
    sub = oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P, w.Hq, w.dtype,
                      rows=[(0, 0), (0, 5), (0, 2)])
    for (b, t), o in sub["out"].items():
        np.testing.assert_array_equal(o, full["out"][b, t])


def test_step_capacity_error():
    w = _small("tiny_decode", H=32, P=8, T=2, Hq=2, Hkv=1, D=4)
    d = wl.make_dense(w)
    k, v = wl.make_cache(w)
    with pytest.raises(ValueError):
        oracle.step(d["x"], d["wq"], d["wk"], d["wv"], k, v, w.P + 1, w.Hq, w.dtype)
