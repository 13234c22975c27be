"""Pins for the literal ring oracle (CPU only).

Each test ties the oracle to something other than its own code: numpy's
array_split, exact integer arithmetic, a fold-order discriminator, the
identities of "Networks and Collective Communication" section 4.2, the byte
lower bounds of section 4.3, and the fp32 summation error bound.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

from a2a_ring_ordered_gb300 import workloads
from oracle import collectives, pointwise, ring
from oracle.bf16 import bf16_to_f32

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- chunk rule
@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 7, 8, 16, 72])
@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 13, 64, 255, 1000])
def test_chunk_rule_matches_numpy_array_split(p, n):
    bounds = ring.chunk_bounds(p, n)
    parts = np.array_split(np.arange(n), p)
    assert len(bounds) == p
    for (off, ln), part in zip(bounds, parts):
        assert ln == len(part)
        if ln:
            assert off == part[0]


# ------------------------------------------------------------- brute force
@pytest.mark.parametrize("p", [1, 2, 3, 4, 5, 6])
@pytest.mark.parametrize("n", list(range(0, 14)))
def test_allreduce_exact_integer_sums(p, n):
    """Integer-valued fp32 inputs: every fold order gives the exact sum, so each
    output element must equal the Python integer sum (comm_sim: "results all
    equal the numpy sum", section 5.2)."""
    rng = np.random.default_rng(1000 * p + n)
    x = [rng.integers(-50, 51, size=n).astype(np.float32) for _ in range(p)]
    outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
    for i in range(n):
        exact = sum(int(x[r][i]) for r in range(p))
        for r in range(p):
            assert outs[r][i] == exact
    shards, _ = ring.ring_reduce_scatter(x, "f32", "sum")
    for k, (off, ln) in enumerate(ring.chunk_bounds(p, n)):
        assert len(shards[k]) == ln
        for j in range(ln):
            assert shards[k][j] == sum(int(x[r][off + j]) for r in range(p))


@pytest.mark.parametrize("p", [2, 3, 5])
def test_int32_sum_wraps_like_twos_complement(p):
    n = 11
    rng = np.random.default_rng(p)
    x = [rng.integers(2**31 - 2**20, 2**31 - 1, size=n, dtype=np.int64).astype(np.int32)
         for _ in range(p)]
    outs, _, _ = ring.ring_allreduce(x, "i32", "sum")
    for i in range(n):
        total = sum(int(x[r][i]) for r in range(p)) % 2**32
        if total >= 2**31:
            total -= 2**32
        assert all(int(o[i]) == total for o in outs)


@pytest.mark.parametrize("op,fn", [("max", np.max), ("min", np.min)])
@pytest.mark.parametrize("p,n", [(3, 10), (8, 37), (1, 5)])
def test_max_min_match_numpy_reduction(op, fn, p, n):
    x = workloads.normal(p, n, 1.0, seed=7)
    outs, _, _ = ring.ring_allreduce(x, "f32", op)
    expect = fn(np.stack(x), axis=0)
    for o in outs:
        np.testing.assert_array_equal(o, expect)


# ------------------------------------------------------ fold-order pinning
def _discriminator(p: int, c: int, n: int | None = None) -> list[np.ndarray]:
    """Chunk c's element: x_{c+1} = 2^24, x_{c+2} = 1, x_{c+3} = 1 (p >= 4),
    x_c = -2^24, zero elsewhere.  Only the fold that starts at rank c+1 and
    walks forward gives 0; every other start or direction gives 1 or 2."""
    n = p if n is None else n
    off, _ = ring.chunk_bounds(p, n)[c]
    x = [np.zeros(n, dtype=np.float32) for _ in range(p)]
    x[(c + 1) % p][off] = 2.0**24
    x[(c + 2) % p][off] = 1.0
    if p >= 4:
        x[(c + 3) % p][off] = 1.0
    x[c][off] = -(2.0**24)
    return x


@pytest.mark.parametrize("p", [3, 4, 5, 8, 16])
def test_fold_order_discriminator(p):
    for c in range(p):
        x = _discriminator(p, c)
        off, _ = ring.chunk_bounds(p, p)[c]
        outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
        assert all(o[off] == 0.0 for o in outs), (p, c)
        # the discriminator really discriminates: other starts/directions differ
        vals = [x[r][off] for r in range(p)]
        for start in range(p):
            for step in (1, -1):
                acc = np.float32(vals[start])
                for j in range(1, p):
                    acc = np.float32(acc + np.float32(vals[(start + step * j) % p]))
                if (start, step) == ((c + 1) % p, 1):
                    assert acc == 0.0
                elif p > 3 or step == 1:
                    assert acc != 0.0, (p, c, start, step)


def test_fold_order_discriminator_ragged_chunks():
    p, n = 4, 10  # chunks of 3, 3, 2, 2
    for c in range(p):
        x = _discriminator(p, c, n)
        off, _ = ring.chunk_bounds(p, n)[c]
        outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
        assert all(o[off] == 0.0 for o in outs)
        assert pointwise.fold_at(x, np.array([off]))[0] == 0.0


# ------------------------------------------------------------- identities
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(1, 7), (2, 9), (4, 64), (5, 23), (8, 100), (16, 1000)])
def test_allreduce_equals_allgather_of_reducescatter(dtype, p, n):
    """Section 4.2: all-reduce = reduce-scatter + all-gather (bit for bit)."""
    if dtype == "i32":
        x = workloads.integer_valued(p, n, seed=p * n, dtype="i32")
    else:
        x = workloads.normal(p, n, 1.0, seed=p * n, dtype=dtype)
    ar, _, _ = ring.ring_allreduce(x, dtype, "sum")
    shards, _ = ring.ring_reduce_scatter(x, dtype, "sum")
    ag, _ = ring.ring_all_gather(shards, dtype)
    for a, b in zip(ar, ag):
        np.testing.assert_array_equal(a, b)
    # and every rank holds the same vector
    for a in ar[1:]:
        np.testing.assert_array_equal(a, ar[0])


def test_allreduce_equals_reduce_then_broadcast_integer():
    x = workloads.integer_valued(6, 31, seed=5)
    ar, _, _ = ring.ring_allreduce(x, "f32", "sum")
    red = collectives.reduce(x, root=2)[2]
    for a in ar:
        np.testing.assert_array_equal(a, red)


# ------------------------------------------------------------ byte counts
@pytest.mark.parametrize("dtype,e", [("f32", 4), ("bf16", 2), ("i32", 4)])
@pytest.mark.parametrize("p,n", [(1, 8), (2, 8), (4, 16), (5, 23), (8, 64), (7, 3)])
def test_byte_counters_closed_forms(dtype, e, p, n):
    if dtype == "i32":
        x = workloads.integer_valued(p, n, seed=3, dtype="i32")
    else:
        x = workloads.normal(p, n, 1.0, seed=3, dtype=dtype)
    _, rs, ag = ring.ring_allreduce(x, dtype, "sum")
    bounds = ring.chunk_bounds(p, n)
    for r in range(p):
        # RS: rank r sends every chunk but its own, as fp32/int32 partials
        assert rs[r] == (n - bounds[r][1]) * 4
        # AG: rank r sends every chunk but chunk r+1, in the data type
        assert ag[r] == (n - bounds[(r + 1) % p][1]) * e


@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_ring_meets_the_per_rank_lower_bounds(p):
    """Section 4.3: all-gather / reduce-scatter send at least (p-1)/p * n bytes
    per device, all-reduce at least 2(p-1)/p * n (Patarasuk & Yuan); the ring
    meets both exactly when p divides n (fp32: partials and data are 4 bytes)."""
    n = 64 * p
    nbytes = 4 * n
    x = workloads.normal(p, n, 1.0, seed=9)
    _, rs, ag = ring.ring_allreduce(x, "f32", "sum")
    shards, rs_only = ring.ring_reduce_scatter(x, "f32", "sum")
    _, ag_only = ring.ring_all_gather(shards, "f32")
    for r in range(p):
        assert rs_only[r] * p == (p - 1) * nbytes
        assert ag_only[r] * p == (p - 1) * nbytes
        assert (rs[r] + ag[r]) * p == 2 * (p - 1) * nbytes
    # and the number of steps is 2(p-1), each moving n/p per device
    assert rs[0] == (p - 1) * nbytes // p


# ------------------------------------------------------- accuracy bound
@pytest.mark.parametrize("p", [2, 4, 8, 16, 72])
def test_fp32_result_within_recursive_summation_bound(p):
    """|fl(sum) - sum| <= gamma_{p-1} * sum|x|, gamma_k = k u / (1 - k u),
    u = 2^-24: a dropped term or a wrong sign would break it."""
    n = 997
    x = workloads.normal(p, n, 1.0, seed=p)
    outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
    xs = np.stack(x).astype(np.float64)
    exact = xs.sum(axis=0)
    absum = np.abs(xs).sum(axis=0)
    u = 2.0**-24
    k = p - 1
    gamma = k * u / (1 - k * u)
    assert np.all(np.abs(outs[0].astype(np.float64) - exact) <= gamma * absum + 1e-300)


# ------------------------------------------------ pointwise vs literal
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("p,n", [(1, 5), (2, 3), (3, 17), (4, 1000), (6, 13), (8, 4099), (72, 300)])
def test_pointwise_matches_literal(dtype, op, p, n):
    if dtype == "i32":
        x = workloads.integer_valued(p, n, seed=11, lo=-2**30, hi=2**30, dtype="i32")
    else:
        x = workloads.normal(p, n, 1.0, seed=11, dtype=dtype)
    outs, _, _ = ring.ring_allreduce(x, dtype, op)
    got = pointwise.allreduce_at(x, np.arange(n), dtype, op)
    np.testing.assert_array_equal(outs[0], got)


# ------------------------------------------------------------- bf16 paths
def test_bf16_allreduce_integer_values_are_exact():
    p, n = 5, 40
    x = workloads.integer_valued(p, n, seed=2, lo=-20, hi=20, dtype="bf16")
    outs, _, _ = ring.ring_allreduce(x, "bf16", "sum")
    xs = np.stack([bf16_to_f32(v) for v in x]).astype(np.float64)
    exact = xs.sum(axis=0)  # |sum| <= 100: exactly representable in bf16
    np.testing.assert_array_equal(bf16_to_f32(outs[0]).astype(np.float64), exact)


def test_bf16_accumulates_in_fp32_not_per_hop():
    """256 + 1 + 1 + ... : rounding to bf16 at each hop would lose every 1
    (bf16 spacing at 256 is 2); fp32 accumulation keeps them."""
    p = 4
    from a2a_ring_ordered_gb300.workloads import to_bf16_bits

    vals = np.array([1.0, 256.0, 1.0, 1.0], dtype=np.float32)  # rank 1 starts chunk 0
    x = [to_bf16_bits(np.full(1, v, dtype=np.float32)) for v in vals]
    x = [np.concatenate([xi, np.zeros(3, np.uint16)]) for xi in x]
    outs, _, _ = ring.ring_allreduce(x, "bf16", "sum")
    assert bf16_to_f32(outs[0][:1])[0] == 260.0  # 259 rounds to 260 (ties to even)


def test_bucket_scale_cast_against_torch_cast():
    import torch

    p, n = 8, 257
    g = workloads.integer_valued(p, n, seed=4, lo=-3000, hi=3000)
    out = ring.bucket_allreduce_scale_cast(g, 1.0 / 8)
    exact = np.stack(g).astype(np.float64).sum(axis=0) / 8.0  # exact in fp32
    expect = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
    expect = expect.view(torch.int16).numpy().view(np.uint16)
    for o in out:
        np.testing.assert_array_equal(o, expect)


def test_zero_chain_equals_bf16_allreduce():
    p, n = 16, 16 * 37 + 5
    x = workloads.normal(p, n, 1e-2, seed=2, dtype="bf16")
    shards, gathered = ring.zero_rs_then_ag(x)
    ar, _, _ = ring.ring_allreduce(x, "bf16", "sum")
    for a, b in zip(ar, gathered):
        np.testing.assert_array_equal(a, b)
    assert [len(s) for s in shards] == [ln for _, ln in ring.chunk_bounds(p, n)]


# ---------------------------------------------------------------- shapes
def test_degenerate_shapes():
    # p = 1: no steps; the output is the input and nothing is sent
    x = workloads.normal(1, 9, 1.0, seed=0)
    outs, rs, ag = ring.ring_allreduce(x, "f32", "sum")
    np.testing.assert_array_equal(outs[0], x[0])
    assert rs == [0] and ag == [0]
    # n = 0: empty everywhere
    x = [np.zeros(0, np.float32) for _ in range(4)]
    outs, rs, ag = ring.ring_allreduce(x, "f32", "sum")
    assert all(len(o) == 0 for o in outs) and rs == [0] * 4 and ag == [0] * 4
    # n < p: some chunks are empty
    x = workloads.integer_valued(5, 3, seed=1)
    outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
    np.testing.assert_array_equal(outs[0], np.stack(x).sum(axis=0))
    with pytest.raises(ValueError):
        ring.ring_allreduce([np.zeros(3, np.float32), np.zeros(4, np.float32)])


def test_every_pair_of_small_p_and_n_runs():
    for p, n in itertools.product(range(1, 7), range(0, 9)):
        x = workloads.integer_valued(p, n, seed=p + 10 * n)
        outs, _, _ = ring.ring_allreduce(x, "f32", "sum")
        np.testing.assert_array_equal(outs[-1], np.stack(x).sum(axis=0) if n else np.zeros(0))
