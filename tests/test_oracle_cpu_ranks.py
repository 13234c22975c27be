"""Pins for the CPU-rank ring (oracle/cpu_ranks.cpp, CPU only).

The threaded ring must give the bits of the single-threaded literal ring
(oracle/ring.py) for every kind, dtype, op, size and thread count, the worked
example's values, the ring's fold order (the discriminator), the byte counts of
the ring; and its bounded waits must turn an injected host fault -- a rank that
stalls, a rank that skips a send -- into a status, never a hang.
"""
from __future__ import annotations

import os
import time

import numpy as np
import pytest

from a2a_ring_ordered_gb300 import workloads
from oracle import cpu_ranks, ring

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_example_p4.txt")


def _inputs(dtype, p, n, seed):
    if dtype == "i32":
        rng = np.random.default_rng(seed)
        return [rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32) for _ in range(p)]
    return workloads.normal(p, n, 1.0, seed, dtype=dtype)


def _same(a, b):
    assert a.dtype == b.dtype and a.shape == b.shape
    assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_worked_example():
    g = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split(":", 1)
            g[k.strip()] = [float(t) for t in v.split()]
    x = [np.array(g[f"input {r}"], dtype=np.float32) for r in range(4)]
    outs, _, st, _ = cpu_ranks.ring("allreduce", x)
    assert st == cpu_ranks.OK
    for r in range(4):
        assert outs[r].tolist() == g["allreduce"]
    shards, _, st, _ = cpu_ranks.ring("reduce_scatter", x)
    assert [s.tolist() for s in shards] == [g[f"reduce_scatter {k}"] for k in range(4)]
    contrib = [np.array(g[f"all_gather_contrib {k}"], dtype=np.float32) for k in range(4)]
    outs, _, st, _ = cpu_ranks.ring("all_gather", contrib)
    assert all(o.tolist() == g["all_gather"] for o in outs)


def test_fold_order_discriminator():
    """Chunk 0 (p=4, n=4) folds x1 + x2 + x3 then x0: 2^24 + 1 + 1 - 2^24 = 0 in
    fp32 (each +1 is lost), where a fold starting at rank 0 would give 2."""
    x = [np.zeros(4, np.float32) for _ in range(4)]
    x[1][0], x[2][0], x[3][0], x[0][0] = 2.0**24, 1.0, 1.0, -(2.0**24)
    outs, _, st, _ = cpu_ranks.ring("allreduce", x, max_threads=4)
    assert st == cpu_ranks.OK
    assert all(o[0] == 0.0 for o in outs)


SHAPES = [(1, 5), (2, 4099), (3, 1001), (4, 13), (5, 3), (7, 7001), (16, 65543)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("p,n", SHAPES)
def test_equals_the_literal_ring(dtype, op, p, n):
    x = _inputs(dtype, p, n, seed=17 * p + n)
    want_ar, rs_b, ag_b = ring.ring_allreduce(x, dtype, op)
    want_rs, rs_only = ring.ring_reduce_scatter(x, dtype, op)
    want_ag, ag_only = ring.ring_all_gather(want_rs, dtype)
    for threads in sorted({1, 3, p}):
        outs, sent, st, used = cpu_ranks.ring("allreduce", x, dtype, op, max_threads=threads)
        assert st == cpu_ranks.OK and used == min(p, threads)
        for r in range(p):
            _same(outs[r], want_ar[r])
        assert sent == [a + b for a, b in zip(rs_b, ag_b)]
        shards, sent, st, _ = cpu_ranks.ring("reduce_scatter", x, dtype, op, max_threads=threads)
        assert st == cpu_ranks.OK and sent == rs_only
        for k in range(p):
            _same(shards[k], want_rs[k])
        outs, sent, st, _ = cpu_ranks.ring("all_gather", want_rs, dtype, max_threads=threads)
        assert st == cpu_ranks.OK and sent == ag_only
        for r in range(p):
            _same(outs[r], want_ag[r])


@pytest.mark.parametrize("p,n", [(8, 65536), (3, 1001), (2, 7)])
def test_bucket_equals_the_oracle_bucket(p, n):
    g = workloads.normal(p, n, 1e-3, seed=1)
    scale = float(np.float32(1.0 / p))
    want = ring.bucket_allreduce_scale_cast(g, scale)
    outs, _, st, _ = cpu_ranks.ring("bucket", g, scale=scale)
    assert st == cpu_ranks.OK
    for r in range(p):
        _same(outs[r], want[r])


@pytest.mark.parametrize("kind,step", [("allreduce", 1), ("allreduce", 5), ("reduce_scatter", 0),
                                       ("all_gather", 2)])
def test_a_stalled_rank_times_out(kind, step):
    """Rank 2 stops taking part at `step`: the others' barrier wait runs out
    and the collective returns TIMEOUT after about the timeout, not a hang."""
    p, n = 4, 1000
    x = workloads.normal(p, n, 1.0, seed=3)
    if kind == "all_gather":
        x = [v[off:off + ln] for v, (off, ln) in zip(x, ring.chunk_bounds(p, n))]
    t0 = time.perf_counter()
    outs, _, st, _ = cpu_ranks.ring(kind, x, max_threads=p, timeout_s=0.2, fault="stall", fault_rank=2,
                                    fault_step=step)
    dt = time.perf_counter() - t0
    assert st == cpu_ranks.TIMEOUT and outs is None
    assert dt < 5.0
    # the next collective runs normally
    outs, _, st, _ = cpu_ranks.ring(kind, x, max_threads=p)
    assert st == cpu_ranks.OK


@pytest.mark.parametrize("threads", [1, 2, 4])
def test_a_skipped_send_is_a_lost_message(threads):
    """Rank 1 skips its send of step 1: rank 2 finds no message of that step
    in its inbox and the collective returns LOST_MESSAGE."""
    p, n = 4, 1000
    x = workloads.normal(p, n, 1.0, seed=4)
    outs, _, st, _ = cpu_ranks.ring("allreduce", x, max_threads=threads, timeout_s=0.5, fault="skip_send",
                                    fault_rank=1, fault_step=1)
    assert st == cpu_ranks.LOST_MESSAGE and outs is None


def test_a_stall_with_several_ranks_per_thread():
    """8 ranks on 3 threads: the thread holding rank 5 stops; the other two
    time out instead of waiting for it."""
    x = workloads.normal(8, 4096, 1.0, seed=5)
    outs, _, st, used = cpu_ranks.ring("allreduce", x, max_threads=3, timeout_s=0.2, fault="stall",
                                       fault_rank=5, fault_step=9)
    assert st == cpu_ranks.TIMEOUT and used == 3


def test_invalid_arguments():
    x = workloads.normal(2, 8, 1.0, seed=6)
    assert cpu_ranks.ring("allreduce", x, max_threads=0)[2] == cpu_ranks.INVALID
    assert cpu_ranks.ring("allreduce", x, timeout_s=0.0)[2] == cpu_ranks.INVALID
    assert cpu_ranks.ring("bucket", x, op="max")[2] == cpu_ranks.INVALID
