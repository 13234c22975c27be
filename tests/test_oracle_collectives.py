"""Pins for the oracle's primitive definitions and the pages' worked example."""
from __future__ import annotations

import numpy as np
import pytest

from a2a_ring_ordered_gb300 import workloads
from oracle import collectives, ring


def _f(v):
    return np.asarray(v, dtype=np.float32)


def test_worked_example_all_primitives(worked_example):
    """Section 4.1's 4-device example; expected outputs derived by hand."""
    g = worked_example
    x = workloads.worked_example(4)
    for d in range(4):
        np.testing.assert_array_equal(x[d], _f(g[f"input {d}"]))

    ar, _, _ = ring.ring_allreduce(x, "f32", "sum")
    for d in range(4):
        np.testing.assert_array_equal(ar[d], _f(g["allreduce"]))

    shards, _ = ring.ring_reduce_scatter(x, "f32", "sum")
    for k in range(4):
        np.testing.assert_array_equal(shards[k], _f(g[f"reduce_scatter {k}"]))

    contrib = [x[d][d:d + 1].copy() for d in range(4)]  # block d of [10d+j] is 10d+d = 11d
    for d in range(4):
        np.testing.assert_array_equal(contrib[d], _f(g[f"all_gather_contrib {d}"]))
    gathered, _ = ring.ring_all_gather(contrib, "f32")
    for d in range(4):
        np.testing.assert_array_equal(gathered[d], _f(g["all_gather"]))
    np.testing.assert_array_equal(collectives.all_gather(contrib)[0], _f(g["all_gather"]))

    a2a = collectives.all_to_all(x)
    for j in range(4):
        np.testing.assert_array_equal(a2a[j], _f(g[f"all_to_all {j}"]))

    for d in range(4):
        np.testing.assert_array_equal(collectives.broadcast(x, 0)[d], _f(g["broadcast_root0"]))
    red = collectives.reduce(x, 0)
    np.testing.assert_array_equal(red[0], _f(g["reduce_root0"]))
    assert all(r is None for r in red[1:])


def test_worked_example_whole_vector_all_gather():
    """The other reading of section 4.1's all-gather: each device contributes its
    whole vector; everyone gets the 16-element concatenation."""
    x = workloads.worked_example(4)
    gathered, _ = ring.ring_all_gather(x, "f32")
    expect = np.concatenate(x)
    for g in gathered:
        np.testing.assert_array_equal(g, expect)


@pytest.mark.parametrize("p,n", [(1, 3), (2, 8), (4, 4), (3, 10), (8, 1000), (5, 3)])
def test_all_to_all_twice_is_identity(p, n):
    """Section 4.2: all-to-all applied twice returns the original (transpose of a transpose)."""
    x = workloads.normal(p, n, 1.0, seed=p + n)
    back = collectives.all_to_all(collectives.all_to_all(x))
    for a, b in zip(x, back):
        np.testing.assert_array_equal(a, b)


def test_all_to_all_is_a_block_transpose_by_brute_force():
    p, n = 3, 7  # blocks of 3, 2, 2
    x = [np.array([100 * i + k for k in range(n)], dtype=np.float32) for i in range(p)]
    out = collectives.all_to_all(x)
    bounds = ring.chunk_bounds(p, n)
    for j in range(p):
        expect = []
        for i in range(p):
            off, ln = bounds[j]
            expect += [100 * i + k for k in range(off, off + ln)]
        np.testing.assert_array_equal(out[j], _f(expect))


def _tagged_rows(counts, row_elems):
    """Row values encode (source, destination, row index) so placement is unique."""
    p = counts.shape[0]
    send = []
    for s in range(p):
        rows = []
        for d in range(p):
            for k in range(int(counts[s][d])):
                rows.append(np.full(row_elems, s * 10_000 + d * 100 + k, dtype=np.int32))
        send.append(np.concatenate(rows) if rows else np.zeros(0, np.int32))
    return send


@pytest.mark.parametrize("p,row_elems", [(1, 3), (3, 1), (4, 5), (8, 2)])
def test_all_to_allv_placement_by_brute_force(p, row_elems):
    rng = np.random.default_rng(p)
    counts = rng.integers(0, 5, size=(p, p))
    counts[0, :] = 0  # a source that sends nothing
    send = _tagged_rows(counts, row_elems)
    recv = collectives.all_to_allv(send, counts, row_elems)
    for d in range(p):
        expect = []
        for s in range(p):  # source order
            for k in range(int(counts[s][d])):
                expect += [s * 10_000 + d * 100 + k] * row_elems
        np.testing.assert_array_equal(recv[d], np.array(expect, dtype=np.int32))


def test_moe_dispatch_then_combine_is_identity():
    """Section 4.2 / 7.4: MoE dispatches with all-to-all and combines with a
    second one; with counts transposed the second returns every token home."""
    counts, rng = workloads.moe_counts(p=8, tokens_per_rank=512, seed=3)
    hidden = 16
    send = workloads.moe_tokens(counts, hidden, rng, dtype="bf16")
    recv = collectives.all_to_allv(send, counts, hidden)
    assert [len(r) // hidden for r in recv] == list(counts.sum(axis=0))
    back = collectives.all_to_allv(recv, counts.T, hidden)
    for a, b in zip(send, back):
        np.testing.assert_array_equal(a, b)


def test_moe_counts_draw_is_zipf_skewed():
    counts, _ = workloads.moe_counts()
    assert counts.shape == (8, 8)
    assert (counts.sum(axis=1) == 16384).all()
    recv = counts.sum(axis=0)
    assert list(recv) == sorted(recv, reverse=True)  # expert 0 is the hot one
    pi = workloads.moe_zipf_probs()
    assert abs(pi[0] - 0.4286) < 1e-4 and abs(pi.sum() - 1) < 1e-12


@pytest.mark.parametrize("p,n", [(1, 5), (4, 4), (4, 10), (8, 1001), (16, 3)])
def test_broadcast_equals_scatter_then_all_gather(p, n):
    """Section 4.2 (Van de Geijn): broadcast = scatter + all-gather."""
    x = workloads.normal(p, n, 1.0, seed=n)
    root = p - 1
    parts = collectives.scatter(x[root], p)
    gathered, _ = ring.ring_all_gather(parts, "f32")
    for a, b in zip(collectives.broadcast(x, root), gathered):
        np.testing.assert_array_equal(a, b)


def test_scatter_gather_are_inverse():
    data = np.arange(23, dtype=np.float32)
    parts = collectives.scatter(data, 5)
    np.testing.assert_array_equal(collectives.gather(parts, root=3)[3], data)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(1, 5), (3, 10), (4, 4), (8, 1001)])
def test_ring_reduce_equals_allreduce_on_the_root(dtype, p, n):
    """all-reduce = reduce + broadcast (section 4.2 family): the root's reduce
    result is bit-identical to every rank's all-reduce result."""
    x = (workloads.integer_valued(p, n, 5, dtype="i32") if dtype == "i32"
         else workloads.normal(p, n, 1.0, 5, dtype=dtype))
    ar, _, _ = ring.ring_allreduce(x, dtype)
    for root in {0, p - 1}:
        red = collectives.reduce_ring(x, root, dtype)
        np.testing.assert_array_equal(red[root], ar[0])
        assert all(red[r] is None for r in range(p) if r != root)


def test_ring_reduce_integer_values_exact():
    x = workloads.integer_valued(6, 37, 2)
    red = collectives.reduce_ring(x, 2)[2]
    np.testing.assert_array_equal(red, np.stack(x).sum(axis=0))


@pytest.mark.parametrize("p,sp,H,D", [(1, 3, 2, 4), (2, 5, 4, 8), (4, 3, 8, 16), (8, 2, 16, 4)])
def test_ulysses_exchange_by_brute_force_and_inverse(p, sp, H, D):
    """Element (s, t, h, d) of the sequence shards lands at (r = h // (H/p),
    row s*sp + t, head h % (H/p), d) -- checked element by element -- and the
    inverse exchange restores every shard."""
    x = [np.arange(sp * H * D, dtype=np.float32) + 10_000 * s for s in range(p)]
    y = collectives.ulysses_seq_to_heads(x, H, D)
    hp = H // p
    for s in range(p):
        for t in range(sp):
            for h in range(H):
                r = h // hp
                got = y[r].reshape(p * sp, hp, D)[s * sp + t, h % hp]
                want = x[s].reshape(sp, H, D)[t, h]
                np.testing.assert_array_equal(got, want)
    back = collectives.ulysses_heads_to_seq(y, H, D)
    for a, b in zip(x, back):
        np.testing.assert_array_equal(a, b)


def test_ulysses_is_an_all_to_all_of_contiguous_segments():
    """With one token per shard and D = 1 the exchange is the plain block
    transpose of section 4.1."""
    p = 4
    x = workloads.normal(p, p, 1.0, 0)  # shard s: [1 token, H = p heads, D = 1]
    np.testing.assert_array_equal(np.concatenate(collectives.ulysses_seq_to_heads(x, p, 1)),
                                  np.concatenate(collectives.all_to_all(x)))


@pytest.mark.parametrize("p", [1, 2, 3, 5, 7])
@pytest.mark.parametrize("n", [0, 1, 4, 13, 23])
def test_pointwise_sources_match_the_whole_buffer_collectives(p, n):
    """The per-element source maps (used to check huge outputs at sampled
    positions) agree at every position with the whole-buffer all-gather (and
    the literal ring all-gather) and the block-transpose all-to-all, on inputs
    whose every value names its rank and position."""
    from oracle import pointwise

    x = [np.arange(n, dtype=np.int64) + 1000 * r for r in range(p)]
    parts = [x[k][off:off + ln] for k, (off, ln) in enumerate(ring.chunk_bounds(p, n))]
    ag = collectives.all_gather(parts)
    ring_ag, _ = ring.ring_all_gather([v.astype(np.int32) for v in parts], "i32")
    idx = np.arange(n, dtype=np.int64)
    k, pos = pointwise.all_gather_source(p, n, idx)
    got = np.array([parts[a][b] for a, b in zip(k, pos)], dtype=np.int64)
    for r in range(p):
        np.testing.assert_array_equal(got, ag[r])
        np.testing.assert_array_equal(got.astype(np.int32), ring_ag[r])
    a2a = collectives.all_to_all(x)
    for j in range(p):
        m = len(a2a[j])
        src, spos = pointwise.all_to_all_source(p, n, j, np.arange(m, dtype=np.int64))
        got = np.array([x[a][b] for a, b in zip(src, spos)], dtype=np.int64)
        np.testing.assert_array_equal(got, a2a[j])


@pytest.mark.parametrize("p,seed", [(1, 0), (3, 1), (5, 2), (8, 3)])
def test_all_to_allv_source_matches_the_whole_buffer_exchange(p, seed):
    """The per-row source map agrees with ``collectives.all_to_allv`` at every
    received row, with empty blocks among the counts; every value names its
    source rank and row."""
    from oracle import pointwise

    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 4, size=(p, p))
    counts[rng.random((p, p)) < 0.3] = 0
    row = 3
    send = [np.repeat(np.arange(counts[s].sum(), dtype=np.int64) + 1000 * s, row) for s in range(p)]
    recv = collectives.all_to_allv(send, counts, row)
    for d in range(p):
        m = len(recv[d]) // row
        src, srow = pointwise.all_to_allv_source(counts, d, np.arange(m, dtype=np.int64))
        got = np.array([send[a][b * row] for a, b in zip(src, srow)], dtype=np.int64)
        np.testing.assert_array_equal(got, recv[d][::row])
