"""Layered caches (one pinned allocation holding every layer's K and V) and
captured decode steps (a CUDA graph that runs every layer, then advances the
lengths), through the C ABI, against the fp64 oracle layer by layer.

Bars as for the one-layer path: decode appends bit-exact, prefill appends
within 1 ulp or the fp32 summation bound, outputs max-abs <= 1e-2 and
mean-rel <= 2e-3; the lengths advance once per token, after the last layer."""
import numpy as np
import pytest

import zero_copy_offloaded_gb300 as dkv
from zero_copy_offloaded_gb300 import workloads as wl

from .helpers import assert_close, assert_projection_close, out_f64, to_dev, torch_dtype

pytestmark = pytest.mark.gpu


class Layers:
    """`layers` independent layers (own weights, own cache prefix) of one shape."""

    def __init__(self, layers, w: wl.Workload, lens, s_max):
        self.L, self.w, self.s_max = layers, w, s_max
        self.lens = np.asarray(lens, np.int64)
        self.cache = dkv.LayeredKVCache(layers, w.B, w.Hkv, w.D, s_max, w.dtype)
        self.dense, self.k0, self.v0 = [], [], []
        for l in range(layers):
            wl_l = w.with_(seed=w.seed + 101 * l)
            d = wl.make_dense(wl_l)
            kc = np.full((w.B, w.Hkv, s_max, w.D), 0x7E57, np.uint16)
            vc = kc.copy()
            wp = wl_l.with_(P=int(self.lens.max()))
            for b in range(w.B):
                for h in range(w.Hkv):
                    kk, vv = wl.cache_slice(wp, b, h)
                    n = int(self.lens[b])
                    kc[b, h, :n], vc[b, h, :n] = kk[:n], vv[:n]
            self.cache.k_host[l] = kc
            self.cache.v_host[l] = vc
            self.dense.append(d)
            self.k0.append(kc)
            self.v0.append(vc)
        self.cache.set_lengths(self.lens.astype(np.int32))
        self.dev = [{k: to_dev(d[k], w.dtype) for k in ("x", "wq", "wk", "wv")} for d in self.dense]

    def oracle(self, l, x_bits, k, v, lens):
        import oracle
        d = self.dense[l]
        return oracle.step(x_bits, d["wq"], d["wk"], d["wv"], k, v, lens, self.w.Hq, self.w.dtype)

    def free(self):
        self.cache.free()


def _decode_out(w):
    import torch
    return torch.empty((w.B, 1, w.Hq, w.D), dtype=torch_dtype(w.dtype), device="cuda")


def check_step(lay: Layers, outs, lens, label, canary=True):
    """One decode step of every layer against the oracle; the oracle's caches
    after the step become the reference for the next one."""
    w = lay.w
    for l in range(lay.L):
        xb = lay.dense[l]["x"][:, :1]
        ref = lay.oracle(l, xb, lay.k0[l], lay.v0[l], lens)
        got = out_f64(outs[l], w.dtype).reshape(w.B, w.Hq, w.D)
        assert_close(got, ref["out"].reshape(w.B, w.Hq, w.D), f"{label} layer {l}")
        kh, vh = lay.cache.k_host[l], lay.cache.v_host[l]
        for b in range(w.B):
            p = int(lens[b])
            assert np.array_equal(kh[b, :, p], ref["k_new"][b, 0]), f"{label} layer {l} k b={b}"
            assert np.array_equal(vh[b, :, p], ref["v_new"][b, 0]), f"{label} layer {l} v b={b}"
            if canary:
                assert np.all(kh[b, :, p + 1:] == 0x7E57)
        lay.k0[l], lay.v0[l] = ref["k_cache_after"], ref["v_cache_after"]


def test_layered_decode_layer_by_layer():
    w = wl.Workload("t", "decode", B=2, H=128, Hq=8, Hkv=2, D=128, P=300, seed=31)
    lay = Layers(3, w, [300, 77], 320)
    try:
        outs = [_decode_out(w) for _ in range(3)]
        for l in range(3):
            d = lay.dev[l]
            lay.cache.decode_layer(l, d["x"].reshape(w.B, 1, w.H), d["wq"], d["wk"], d["wv"], w.Hq,
                                   outs[l])
            # the lengths advance with the last layer only
            expect = [300, 77] if l < 2 else [301, 78]
            assert list(lay.cache.lengths()) == expect
        lay.cache.sync()
        check_step(lay, outs, lay.lens, "layered")
    finally:
        lay.free()


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [("bf16", 128, 32, 8), ("fp16", 64, 8, 8)])
def test_captured_step_replays(dtype, D, Hq, Hkv):
    """A captured two-layer step launched three times appends at the lengths
    of each step (the graph reads them from device memory), then ordinary
    per-layer calls and a relaunch continue from where the graph left off."""
    w = wl.Workload("t", "decode", B=3, H=128, Hq=Hq, Hkv=Hkv, D=D, P=200, dtype=dtype,
                    kv_dist="uniform2" if dtype == "fp16" else "normal", seed=41)
    lay = Layers(2, w, [200, 63, 64], 220)
    try:
        outs = [_decode_out(w) for _ in range(2)]
        xs = [d["x"].reshape(w.B, 1, w.H) for d in lay.dev]
        lay.cache.capture_step(xs, [d["wq"] for d in lay.dev], [d["wk"] for d in lay.dev],
                               [d["wv"] for d in lay.dev], w.Hq, outs)
        lens = lay.lens.copy()
        for step in range(3):
            lay.cache.launch_step()
            lay.cache.sync()
            check_step(lay, outs, lens, f"graph step {step}")
            lens = lens + 1
            assert list(lay.cache.lengths()) == list(lens)
        # per-layer calls outside the graph, then the graph again
        for l in range(2):
            d = lay.dev[l]
            lay.cache.decode_layer(l, xs[l], d["wq"], d["wk"], d["wv"], w.Hq, outs[l])
        lay.cache.sync()
        check_step(lay, outs, lens, "after graph")
        lens = lens + 1
        lay.cache.launch_step()
        lay.cache.sync()
        check_step(lay, outs, lens, "graph again")
        # a length set by hand is published before the next launch
        lens = np.array([5, 5, 5])
        lay.cache.set_lengths(lens.astype(np.int32))
        lay.k0 = [k.copy() for k in lay.k0]
        lay.cache.launch_step()
        lay.cache.sync()
        check_step(lay, outs, lens, "after set_lengths", canary=False)
    finally:
        lay.free()


def test_captured_steps_back_to_back():
    """Three captured three-layer steps launched with no synchronisation in
    between: inside a graph each layer's kernels are programmatic dependents of
    the previous layer's, and graphs follow one another on the stream.  Every
    step's appended rows, at their own lengths, and the last step's outputs
    match the oracle run step by step."""
    w = wl.Workload("t", "decode", B=2, H=256, Hq=8, Hkv=2, D=128, P=300, seed=43)
    lay = Layers(3, w, [300, 17], 320)
    try:
        outs = [_decode_out(w) for _ in range(lay.L)]
        xs = [d["x"].reshape(w.B, 1, w.H) for d in lay.dev]
        lay.cache.capture_step(xs, [d["wq"] for d in lay.dev], [d["wk"] for d in lay.dev],
                               [d["wv"] for d in lay.dev], w.Hq, outs)
        lens = lay.lens.copy()
        for _ in range(3):
            lay.cache.launch_step()
        lay.cache.sync()
        assert list(lay.cache.lengths()) == list(lens + 3)
        for step in range(3):
            for l in range(lay.L):
                ref = lay.oracle(l, lay.dense[l]["x"][:, :1], lay.k0[l], lay.v0[l], lens)
                kh, vh = lay.cache.k_host[l], lay.cache.v_host[l]
                for b in range(w.B):
                    p = int(lens[b])
                    assert np.array_equal(kh[b, :, p], ref["k_new"][b, 0]), f"step {step} layer {l}"
                    assert np.array_equal(vh[b, :, p], ref["v_new"][b, 0]), f"step {step} layer {l}"
                if step == 2:
                    got = out_f64(outs[l], w.dtype).reshape(w.B, w.Hq, w.D)
                    assert_close(got, ref["out"].reshape(w.B, w.Hq, w.D), f"last step layer {l}")
                lay.k0[l], lay.v0[l] = ref["k_cache_after"], ref["v_cache_after"]
            lens = lens + 1
        for l in range(lay.L):  # nothing written past the last step's rows
            for b in range(w.B):
                assert np.all(lay.cache.k_host[l][b, :, int(lens[b]):] == 0x7E57)
    finally:
        lay.free()


def test_layered_prefill_then_captured_decode():
    w = wl.Workload("t", "prefill", B=2, H=128, Hq=8, Hkv=2, D=128, P=100, T=60, seed=51)
    lay = Layers(2, w, [100, 30], 200)
    try:
        import torch
        for l in range(2):
            d = lay.dev[l]
            out = torch.empty((w.B, w.T, w.Hq, w.D), dtype=torch_dtype(w.dtype), device="cuda")
            lay.cache.prefill_layer(l, d["x"], d["wq"], d["wk"], d["wv"], w.Hq, out)
            lay.cache.sync()
            ref = lay.oracle(l, lay.dense[l]["x"], lay.k0[l], lay.v0[l], lay.lens)
            got = out_f64(out, w.dtype).reshape(w.B, w.T, w.Hq, w.D)
            assert_close(got, ref["out"], f"layered prefill layer {l}")
            for b in range(w.B):
                p = int(lay.lens[b])
                for name, host, wm in (("k", lay.cache.k_host[l], lay.dense[l]["wk"]),
                                       ("v", lay.cache.v_host[l], lay.dense[l]["wv"])):
                    g = host[b, :, p:p + w.T].transpose(1, 0, 2).reshape(w.T, w.Hkv * w.D)
                    assert_projection_close(g, lay.dense[l]["x"][b], wm, w.dtype,
                                            f"layer {l} {name} b={b}")
            # the oracle's caches after the prefill, with the GPU's appended rows
            # (the tensor-core projection may differ in the last bit)
            lay.k0[l] = lay.cache.k_host[l].copy()
            lay.v0[l] = lay.cache.v_host[l].copy()
        lens = lay.lens + w.T
        assert list(lay.cache.lengths()) == list(lens)
        wd = w.with_(phase="decode", T=1)
        outs = [_decode_out(wd) for _ in range(2)]
        xs = [d["x"][:, :1].contiguous() for d in lay.dev]
        lay.w = wd
        lay.dense = [{**d, "x": d["x"][:, :1]} for d in lay.dense]
        lay.cache.capture_step(xs, [d["wq"] for d in lay.dev], [d["wk"] for d in lay.dev],
                               [d["wv"] for d in lay.dev], w.Hq, outs)
        lay.cache.launch_step()
        lay.cache.sync()
        check_step(lay, outs, lens, "decode after layered prefill")
    finally:
        lay.free()


def test_layered_errors():
    c = dkv.LayeredKVCache(2, 1, 2, 64, 16)
    try:
        import torch
        x = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device="cuda")
        wq = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
        wk = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((1, 1, 4, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(dkv.DkvError) as ei:
            dkv.dkv_decode(c.h, x, wq, wk, wk, 64, 4, out)
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
        with pytest.raises(dkv.DkvError) as ei:
            c.decode_layer(2, x, wq, wk, wk, 4, out)
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
        with pytest.raises(dkv.DkvError) as ei:
            c.launch_step()
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
        info = dkv.dkv_cache_info(c.h)
        assert info["layers"] == 2 and info["host_pinned_bytes"] == 2 * 2 * 1 * 2 * 16 * 64 * 2
        c.set_lengths([16])
        with pytest.raises(dkv.DkvError) as ei:
            c.decode_layer(0, x, wq, wk, wk, 4, out)
        assert ei.value.name == "DKV_ERR_CAPACITY"
    finally:
        c.free()


def test_captured_step_discarded_when_the_workspace_grows():
    """A prefill that needs a larger workspace discards the captured step
    (its addresses would be stale): the launch asks for a new capture."""
    import torch
    w = wl.Workload("t", "decode", B=1, H=128, Hq=8, Hkv=2, D=64, P=100, seed=3)
    lay = Layers(2, w, [100], 1200)
    try:
        outs = [_decode_out(w) for _ in range(2)]
        xs = [d["x"].reshape(w.B, 1, w.H) for d in lay.dev]
        lay.cache.capture_step(xs, [d["wq"] for d in lay.dev], [d["wk"] for d in lay.dev],
                               [d["wv"] for d in lay.dev], w.Hq, outs)
        d = lay.dev[0]
        xp = torch.zeros((1, 1000, w.H), dtype=torch_dtype(w.dtype), device="cuda")
        op = torch.empty((1, 1000, w.Hq, w.D), dtype=torch_dtype(w.dtype), device="cuda")
        lay.cache.prefill_layer(0, xp, d["wq"], d["wk"], d["wv"], w.Hq, op)
        lay.cache.sync()
        with pytest.raises(dkv.DkvError) as ei:
            lay.cache.launch_step()
        assert ei.value.name == "DKV_ERR_INVALID_ARG"
    finally:
        lay.free()
