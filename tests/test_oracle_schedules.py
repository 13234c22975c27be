"""Pins for the literal simulations of the other all-reduce schedules."""
from __future__ import annotations

import numpy as np
import pytest

from a2a_ring_ordered_gb300 import workloads
from oracle import ring, schedules

POW2 = [2, 4, 8, 16]


def _cases(schedule):
    ps = POW2 if schedule in ("recursive_doubling", "rabenseifner") else [1, 2, 3, 4, 5, 6, 7, 8, 13, 16]
    return [(p, n) for p in ps for n in (p, 3 * p + 1, 100)]


@pytest.mark.parametrize("schedule", schedules.SCHEDULES)
def test_exact_integer_sums_and_identical_outputs(schedule):
    for p, n in _cases(schedule):
        x = workloads.integer_valued(p, n, seed=p * 7 + n)
        out, _ = schedules.allreduce(schedule, x)
        exact = np.stack(x).astype(np.int64).sum(axis=0)
        for o in out:
            np.testing.assert_array_equal(o.astype(np.int64), exact, err_msg=f"{schedule} p={p} n={n}")


@pytest.mark.parametrize("schedule", schedules.SCHEDULES)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_every_device_gets_the_same_bits(schedule, dtype):
    p, n = 8, 1001
    x = (workloads.integer_valued(p, n, 3, lo=-2**30, hi=2**30, dtype="i32") if dtype == "i32"
         else workloads.normal(p, n, 1.0, 3, dtype=dtype))
    out, _ = schedules.allreduce(schedule, x, dtype)
    for o in out[1:]:
        np.testing.assert_array_equal(o, out[0])


def test_bytes_per_device_section_4_3_and_5_3():
    """p = 8: ring and Rabenseifner each send 1.75 n per device (the lower
    bound 2(p-1)/p n), recursive doubling sends 3 n (log2 p n)."""
    p, n = 8, 8 * 1000
    nbytes = 4 * n
    x = workloads.normal(p, n, 1.0, 1)
    _, rs, ag = ring.ring_allreduce(x)
    _, rab = schedules.rabenseifner(x)
    _, rd = schedules.recursive_doubling(x)
    for r in range(p):
        assert (rs[r] + ag[r]) * 4 == 7 * nbytes     # 1.75 n
        assert rab[r] * 4 == 7 * nbytes
        assert rd[r] == 3 * nbytes


@pytest.mark.parametrize("p", [2, 4, 16])
def test_rabenseifner_meets_the_lower_bound(p):
    n = p * 37
    _, sent = schedules.rabenseifner(workloads.normal(p, n, 1.0, 2))
    assert all(s * p == 2 * (p - 1) * 4 * n for s in sent)


def test_tree_and_naive_are_unbalanced():
    """Section 4.3: the tree and naive algorithms load the devices near the root."""
    p, n = 8, 64
    x = workloads.normal(p, n, 1.0, 4)
    _, tree = schedules.binomial_tree(x)
    _, nv = schedules.naive(x)
    e = 4 * n
    # binomial tree: 0 broadcasts 3 times; 4 sends once up, twice down; 2 and 6 once
    # up, once down; the odd devices only send up
    assert tree == [3 * e, 1 * e, 2 * e, 1 * e, 3 * e, 1 * e, 2 * e, 1 * e]
    assert nv == [7 * e] + [e] * 7


# hand-derived values (fp32, round to nearest even; 2^24 + 1 rounds to 2^24):
#   A = (2^24, 1, -2^24, 1):
#     recursive doubling / tree: (x0 + x1) + (x2 + x3) = 2^24 + (-2^24 + 1) = 1
#     Rabenseifner (pairs at distance 2 first): (x0 + x2) + (x1 + x3) = 0 + 2 = 2
#     naive (rank order): ((x0 + x1) + x2) + x3 = (2^24 - 2^24) + 1 = 1
#   B = (1, 2^24, 1, -2^24):
#     recursive doubling / tree: (1 + 2^24) + (1 - 2^24) = 2^24 - 16777215 = 1
#     Rabenseifner: (x0 + x2) + (x1 + x3) = 2 + 0 = 2
#     naive: ((1 + 2^24) + 1) - 2^24 = 2^24 - 2^24 = 0
DISCRIMINATORS = {
    "A": ([2.0**24, 1.0, -(2.0**24), 1.0], {"recursive_doubling": 1.0, "binomial_tree": 1.0,
                                            "rabenseifner": 2.0, "naive": 1.0}),
    "B": ([1.0, 2.0**24, 1.0, -(2.0**24)], {"recursive_doubling": 1.0, "binomial_tree": 1.0,
                                            "rabenseifner": 2.0, "naive": 0.0}),
}


@pytest.mark.parametrize("case", ["A", "B"])
@pytest.mark.parametrize("schedule", schedules.SCHEDULES)
def test_pairing_discriminators(case, schedule):
    vals, want = DISCRIMINATORS[case]
    x = [np.full(4, v, dtype=np.float32) for v in vals]  # every element of every chunk
    out, _ = schedules.allreduce(schedule, x)
    for o in out:
        assert (o == want[schedule]).all(), (schedule, case, o)


def test_bf16_partials_travel_in_fp32():
    p = 4
    vals = np.array([256.0, 1.0, 1.0, 1.0], dtype=np.float32)
    x = [workloads.to_bf16_bits(np.full(4, v, dtype=np.float32)) for v in vals]
    from oracle.bf16 import bf16_to_f32
    for s in schedules.SCHEDULES:
        out, _ = schedules.allreduce(s, x, "bf16")
        assert (bf16_to_f32(out[0]) == 260.0).all(), s  # 259 -> 260 (ties to even) once


def test_power_of_two_required():
    with pytest.raises(ValueError):
        schedules.recursive_doubling(workloads.normal(6, 10, 1.0, 0))
    with pytest.raises(ValueError):
        schedules.rabenseifner(workloads.normal(3, 10, 1.0, 0))


# ------------------------------------------------- hierarchical / 2-D ring
# Hand-derived (fp32, nearest even; 2^24 + 1 rounds to 2^24).
#   p = 6, groups of 3: group 0 = (-2^24, 2^24, 1), group 1 = zeros.  Chunk l
#   of the group ring starts at local rank l + 1:
#     l = 0: (2^24 + 1) - 2^24 = 0;  l = 1: (1 - 2^24) + 2^24 = 1;
#     l = 2: (-2^24 + 2^24) + 1 = 1; the 2-group ring adds zeros.
#   p = 6, groups of 2: group partials (-2^24, 2^24, 1); sub-chunk m of the
#   ring over the groups starts at group m + 1:
#     m = 0: (2^24 + 1) - 2^24 = 0;  m = 1: (1 - 2^24) + 2^24 = 1;
#     m = 2: (-2^24 + 2^24) + 1 = 1.
HIER_CASES = [
    (3, [-(2.0**24), 2.0**24, 1.0, 0.0, 0.0, 0.0], [0, 0, 1, 1, 1, 1]),
    (2, [-(2.0**24), 0.0, 2.0**24, 0.0, 1.0, 0.0], [0, 1, 1, 0, 1, 1]),
]


@pytest.mark.parametrize("group,vals,want", HIER_CASES)
def test_hierarchical_fold_order_by_hand(group, vals, want):
    x = [np.full(6, v, dtype=np.float32) for v in vals]
    out, _ = schedules.hierarchical(x, group)
    for o in out:
        np.testing.assert_array_equal(o, np.array(want, dtype=np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(1, 5), (4, 1), (6, 23), (8, 1000), (12, 37)])
def test_hierarchical_with_one_level_is_the_ring(dtype, p, n):
    """One group of p, or p groups of one: the two-level ring is the flat ring."""
    x = (workloads.integer_valued(p, n, 5, lo=-2**30, hi=2**30, dtype="i32") if dtype == "i32"
         else workloads.normal(p, n, 1.0, 5, dtype=dtype))
    want, _, _ = ring.ring_allreduce(x, dtype)
    for group in (1, p):
        out, _ = schedules.hierarchical(x, group, dtype)
        for o, w in zip(out, want):
            np.testing.assert_array_equal(o, w)


@pytest.mark.parametrize("p,group", [(4, 2), (6, 3), (6, 2), (8, 4), (16, 8), (12, 4)])
def test_hierarchical_exact_integer_sums_and_identical_outputs(p, group):
    for n in (p, 3 * p + 1, 100, 1):
        x = workloads.integer_valued(p, n, seed=p + n)
        out, _ = schedules.hierarchical(x, group)
        exact = np.stack(x).astype(np.int64).sum(axis=0)
        for o in out:
            np.testing.assert_array_equal(o.astype(np.int64), exact)
    y = workloads.normal(p, 501, 1.0, 9, dtype="bf16")
    out, _ = schedules.hierarchical(y, group, "bf16")
    for o in out[1:]:
        np.testing.assert_array_equal(o, out[0])


def test_hierarchical_differs_from_the_flat_ring():
    """Same data as the first hand case: the flat 6-ring starts chunk 0 at rank 1."""
    x = [np.full(6, v, dtype=np.float32) for v in HIER_CASES[0][1]]
    flat, _, _ = ring.ring_allreduce(x)
    hier, _ = schedules.hierarchical(x, 3)
    assert not np.array_equal(flat[0], hier[0])


def test_hierarchical_bytes_section_6_3():
    """p = 16 as 2 nodes x 8 GPUs, n divisible by everything: each GPU sends
    2 (a-1)/a n inside its node and 2 (N-1)/N n/8 across nodes (fp32)."""
    p, a, n = 16, 8, 16 * 64
    x = workloads.normal(p, n, 1.0, 3)
    _, sent = schedules.hierarchical(x, a)
    b = p // a
    intra = 2 * (a - 1) * n // a
    inter = 2 * (b - 1) * (n // a) // b
    assert all(s == 4 * (intra + inter) for s in sent)


def test_hierarchical_group_must_divide_p():
    with pytest.raises(ValueError):
        schedules.hierarchical(workloads.normal(6, 10, 1.0, 0), 4)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,group,n", [(6, 3, 23), (6, 2, 100), (16, 8, 1001), (8, 4, 5), (12, 1, 37),
                                       (12, 12, 37), (9, 3, 2)])
def test_pointwise_hierarchical_matches_the_literal_simulation(dtype, p, group, n):
    from oracle import pointwise
    x = (workloads.integer_valued(p, n, 2, lo=-2**30, hi=2**30, dtype="i32") if dtype == "i32"
         else workloads.normal(p, n, 1.0, 2, dtype=dtype))
    want, _ = schedules.hierarchical(x, group, dtype)
    idx = np.arange(n)
    got = pointwise.hierarchical_at_columns([v[idx] for v in x], idx, n, group, dtype)
    np.testing.assert_array_equal(got, want[0])
    sub = np.array([0, n - 1, n // 2], dtype=np.int64)
    got = pointwise.hierarchical_at_columns([v[sub] for v in x], sub, n, group, dtype)
    np.testing.assert_array_equal(got, want[0][sub])
