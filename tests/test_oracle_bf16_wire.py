"""Pins for the ring's bf16-wire variant (partials rounded to bf16 at every hop)."""
from __future__ import annotations

import numpy as np
import pytest

from a2a_ring_ordered_gb300 import workloads
from oracle import pointwise, ring
from oracle.bf16 import bf16_to_f32


def _bf16(vals):
    return workloads.to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_per_hop_rounding_by_hand():
    """p = 3, one element per chunk, rank values (2^-8, 1, 2^-8).  bf16 has 8
    significant bits, so 1 + 2^-8 is a tie that rounds to 1 (even):
      chunk 0 starts at rank 1: bf16(1 + 2^-8) = 1, bf16(1 + 2^-8) = 1
      chunk 1 starts at rank 2: bf16(2^-8 + 2^-8) = 2^-7, bf16(2^-7 + 1) = 1 + 2^-7
      chunk 2 starts at rank 0: bf16(2^-8 + 1) = 1, bf16(1 + 2^-8) = 1
    With fp32 partials every chunk is 1 + 2^-7, rounded once."""
    x = [_bf16([2.0**-8] * 3), _bf16([1.0] * 3), _bf16([2.0**-8] * 3)]
    wire, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    fp32, _, _ = ring.ring_allreduce(x, "bf16")
    for o in wire:
        np.testing.assert_array_equal(bf16_to_f32(o), [1.0, 1.0 + 2.0**-7, 1.0])
    for o in fp32:
        np.testing.assert_array_equal(bf16_to_f32(o), [1.0 + 2.0**-7] * 3)


@pytest.mark.parametrize("p,n", [(1, 5), (2, 7), (3, 10), (5, 13), (8, 100)])
def test_small_integers_stay_exact(p, n):
    """Every partial of small integers is a bf16 integer (|sum| <= 256), so
    per-hop rounding changes nothing: the exact sum."""
    rng = np.random.default_rng(p * 31 + n)
    vals = [rng.integers(-256 // p, 256 // p + 1, size=n).astype(np.float32) for _ in range(p)]
    out, _, _ = ring.ring_allreduce([_bf16(v) for v in vals], "bf16", wire="bf16")
    exact = np.sum(np.stack(vals).astype(np.float64), axis=0)
    for o in out:
        np.testing.assert_array_equal(bf16_to_f32(o).astype(np.float64), exact)


@pytest.mark.parametrize("op", ["max", "min"])
def test_order_free_ops_are_unchanged(op):
    x = workloads.normal(6, 101, 1.0, 3, dtype="bf16")
    a, _, _ = ring.ring_allreduce(x, "bf16", op, wire="bf16")
    b, _, _ = ring.ring_allreduce(x, "bf16", op)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_reduce_scatter_sends_two_bytes_per_element():
    p, n = 8, 8 * 125
    x = workloads.normal(p, n, 1.0, 4, dtype="bf16")
    _, sent = ring.ring_reduce_scatter(x, "bf16", wire="bf16")
    assert sent == [(n - n // p) * 2] * p  # (p-1)/p n elements of 2 bytes


def test_error_within_the_per_hop_bound():
    """Each hop's rounding moves the partial by at most half a bf16 ulp
    (2^-8 relative, nearest-even), so the result is within
    2^-8 * sum of |partials| (plus fp32 add error, far smaller) of the exact
    sum; the fp32-partial result, rounded once, is within 2^-8 |sum| + fp32."""
    p, n = 8, 2000
    x = workloads.normal(p, n, 1.0, 5, dtype="bf16")
    vals = np.stack([bf16_to_f32(v).astype(np.float64) for v in x])
    out, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    got = bf16_to_f32(out[0]).astype(np.float64)
    bounds = ring.chunk_bounds(p, n)
    for c, (off, ln) in enumerate(bounds):
        order = [(c + j) % p for j in range(1, p + 1)]
        partial_abs = np.zeros(ln)
        run = np.zeros(ln)
        for k, r in enumerate(order):
            run = run + vals[r, off:off + ln]
            if k >= 1:
                partial_abs += np.abs(run)
        err = np.abs(got[off:off + ln] - run)
        assert np.all(err <= 2.0**-8 * partial_abs * 1.01 + 1e-30)


@pytest.mark.parametrize("p,n", [(3, 3), (4, 1001), (7, 50)])
def test_pointwise_matches_literal(p, n):
    x = workloads.normal(p, n, 1.0, 6, dtype="bf16")
    want, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    idx = np.arange(n)
    got = pointwise.allreduce_at_columns([v[idx] for v in x], idx, n, "bf16", wire="bf16")
    np.testing.assert_array_equal(got, want[0])


def test_bf16_wire_needs_bf16_data():
    with pytest.raises(ValueError):
        ring.ring_allreduce(workloads.normal(2, 4, 1.0, 0), "f32", wire="bf16")
