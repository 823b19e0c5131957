"""Multi-process host logic on CPU ranks (gloo, world size 2); no GPU.

* The timing reduction the benchmark uses under torchrun: barrier, max of the
  elapsed time over ranks, whole-job rate = units of all ranks / slowest time.
* Batch sharding (the replicas the fused path runs as): each rank steps its own
  block of sequences with no collective on the data path; the gathered outputs
  and caches equal one step over the whole batch.
* The key-range split with one exchange (all-gather of each rank's normalised
  partial output and log-sum-exp, then the log-sum-exp merge) equals attention
  over all keys: the merge the split-KV combine kernels perform, checked across
  real process boundaries.
"""
import os
import socket

import numpy as np
import pytest

import oracle
from zero_copy_offloaded_gb300 import ranks as rk
from zero_copy_offloaded_gb300 import workloads as wl

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

WORLD = 2


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _lse_merge(os_, lses):
    """o = sum_i e^(lse_i - L) o_i with L = log sum_i e^(lse_i) (natural log)."""
    lses = np.asarray(lses, np.float64)
    m = lses.max(axis=0)
    wts = np.exp(lses - m)
    return (wts[..., None] * np.asarray(os_, np.float64)).sum(axis=0) / wts.sum(axis=0)[..., None]


def _worker(rank, world, port, errfile):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    r = rk.Ranks.from_env()
    assert (r.world, r.rank, r.local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # -- timing reduction: the slowest rank's time, whole-job rate
        secs = [1.5, 2.5][rank]
        rk.barrier(dist)
        tmax = rk.max_over_ranks(secs, dist)
        assert tmax == 2.5
        assert rk.job_rate(8, world, tmax) == pytest.approx(8 * 2 / 2.5)

        # -- batch sharding: each rank steps its own sequences, no data-path collective
        w = wl.small("tiny_decode", B=3, P=40, H=64)
        dense = wl.make_dense(w)
        kc, vc = wl.make_cache(w)
        lo, hi = rk.shard(w.B, world, rank)
        mine = oracle.step(dense["x"][lo:hi], dense["wq"], dense["wk"], dense["wv"],
                           kc[lo:hi].copy(), vc[lo:hi].copy(), w.P, w.Hq, w.dtype)
        parts = [None] * world
        dist.all_gather_object(parts, {k: mine[k] for k in ("out", "k_cache_after", "v_cache_after")})
        whole = oracle.step(dense["x"], dense["wq"], dense["wk"], dense["wv"],
                            kc.copy(), vc.copy(), w.P, w.Hq, w.dtype)
        assert np.array_equal(np.concatenate([p["out"] for p in parts]), whole["out"])
        for key in ("k_cache_after", "v_cache_after"):
            assert np.array_equal(np.concatenate([p[key] for p in parts]), whole[key])

        # -- key-range split with one exchange of (o, lse)
        rng = np.random.default_rng(7)
        S, D, nq = 37, 16, 5
        K = rng.standard_normal((S, D))
        V = rng.standard_normal((S, D))
        Q = rng.standard_normal((nq, D))
        k0, k1 = rk.shard(S, world, rank)
        o_i, lse_i = oracle.attend(K[k0:k1], V[k0:k1], Q, k1 - k0 - 1, want_lse=True)
        gathered = [None] * world
        dist.all_gather_object(gathered, (o_i, lse_i))
        merged = _lse_merge([g[0] for g in gathered], [g[1] for g in gathered])
        o_all, lse_all = oracle.attend(K, V, Q, S - 1, want_lse=True)
        np.testing.assert_allclose(merged, o_all, rtol=0, atol=1e-13)
        # the merged log-sum-exp is the whole one
        lses = np.array([g[1] for g in gathered])
        m = lses.max(axis=0)
        np.testing.assert_allclose(m + np.log(np.exp(lses - m).sum(axis=0)), lse_all, rtol=0, atol=1e-12)
    except BaseException as e:  # the spawning test reads the first failure
        with open(f"{errfile}.{rank}", "w") as f:
            f.write(repr(e))
        raise
    finally:
        dist.destroy_process_group()


def test_ranks_from_env_and_shard():
    assert rk.Ranks.from_env({}) == rk.Ranks(1, 0, 0)
    assert rk.Ranks.from_env({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "1"}) == rk.Ranks(4, 3, 1)
    with pytest.raises(ValueError):
        rk.Ranks.from_env({"WORLD_SIZE": "2", "RANK": "2"})
    for n in (0, 1, 5, 8, 13):
        for world in (1, 2, 3, 8):
            blocks = [rk.shard(n, world, r) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(blocks, blocks[1:]))
            sizes = [hi - lo for lo, hi in blocks]
            assert max(sizes) - min(sizes) <= 1
    assert rk.max_over_ranks(3.0) == 3.0
    with pytest.raises(ValueError):
        rk.job_rate(1, 1, 0.0)


def test_two_gloo_ranks(tmp_path):
    oracle.build()  # once, before the ranks load it
    import torch.multiprocessing as mp

    errfile = str(tmp_path / "err")
    try:
        mp.spawn(_worker, args=(WORLD, _free_port(), errfile), nprocs=WORLD, join=True)
    except Exception:
        msgs = [open(f"{errfile}.{r}").read() for r in range(WORLD) if os.path.exists(f"{errfile}.{r}")]
        pytest.fail("rank failure: " + " | ".join(msgs))
