"""Seeded random parity cases across the primitives: sizes, rank counts,
dtypes, ops, alignments (buffers shifted off the 16-byte grid) and in-place
forms drawn at random, every result compared with the oracle element by
element, every output's guard bands checked."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import GUARD, Guarded, assert_equal, ccl, to_dev, to_host
from oracle import collectives, ring, schedules

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _draw(seed):
    rng = np.random.default_rng(seed)
    p = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 33]))
    n = int(rng.choice([1, 3, p, 17 * p + 5, 4096 + 7, int(rng.integers(1, 200_000))]))
    dtype = str(rng.choice(["f32", "bf16", "i32"]))
    shift = int(rng.integers(0, 2))  # 1: every buffer one element off the 16-byte grid
    return rng, p, n, dtype, shift


def _inputs(dtype, p, n, seed):
    if dtype == "i32":
        return workloads.integer_valued(p, n, seed, lo=-2**31, hi=2**31 - 1, dtype="i32")
    return workloads.normal(p, n, 1.0, seed, dtype=dtype)


def _placed(values, dtype, shift):
    bufs = [Guarded(len(v), dtype, offset=GUARD + shift) for v in values]
    for b, v in zip(bufs, values):
        if len(v):
            b.view.copy_(to_dev(v, dtype))
    return bufs


@pytest.mark.parametrize("seed", range(CASES))
def test_random_allreduce_family(lib, seed):
    rng, p, n, dtype, shift = _draw(seed)
    x = _inputs(dtype, p, n, seed)
    op = str(rng.choice(["sum", "max", "min"]))
    send = _placed(x, dtype, shift)
    in_place = bool(rng.integers(0, 2))
    outs = send if in_place else [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    want, _, _ = ring.ring_allreduce(x, dtype, op)
    lib.ccl_allreduce([b.view for b in send], [o.view for o in outs], op=op)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"AR seed {seed} p={p} n={n} {op} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_reduce_scatter_and_all_gather(lib, seed):
    rng, p, n, dtype, shift = _draw(100 + seed)
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, shift)
    lens = [ln for _, ln in ring.chunk_bounds(p, n)]
    shards = [Guarded(ln, dtype, offset=GUARD + int(rng.integers(0, 2))) for ln in lens]
    want_rs, _ = ring.ring_reduce_scatter(x, dtype, "sum")
    lib.ccl_reduce_scatter([b.view for b in send], [s.view for s in shards])
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], dtype, f"RS seed {seed} p={p} n={n} rank {k}")
        assert shards[k].guards_intact()
    full = [Guarded(n, dtype, offset=GUARD + shift) for _ in range(p)]
    lib.ccl_all_gather([s.view for s in shards], [f.view for f in full])
    want_ag, _ = ring.ring_all_gather(want_rs, dtype)
    for r in range(p):
        assert_equal(to_host(full[r].view), want_ag[r], dtype, f"AG seed {seed} p={p} n={n} rank {r}")
        assert full[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_other_fold_orders(lib, seed):
    rng, p, n, dtype, shift = _draw(200 + seed)
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, shift)
    outs = [Guarded(n, dtype, offset=GUARD + shift) for _ in range(p)]
    choices = ["binomial_tree", "naive", "hierarchical"]
    if p & (p - 1) == 0:
        choices += ["recursive_doubling", "rabenseifner"]
    sched = str(rng.choice(choices))
    if sched == "hierarchical":
        group = int(rng.choice([g for g in range(1, p + 1) if p % g == 0]))
        want, _ = schedules.hierarchical(x, group, dtype)
        lib.ccl_allreduce_hierarchical([b.view for b in send], [o.view for o in outs], group)
    else:
        want, _ = schedules.allreduce(sched, x, dtype)
        lib.ccl_allreduce_schedule([b.view for b in send], [o.view for o in outs], sched)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"{sched} seed {seed} p={p} n={n} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_bf16_wire(lib, seed):
    rng, p, n, _, shift = _draw(300 + seed)
    x = _inputs("bf16", p, n, seed)
    send = _placed(x, "bf16", shift)
    outs = [Guarded(n, "bf16", offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    want, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    lib.ccl_allreduce_bf16_wire([b.view for b in send], [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], "bf16", f"bf16 wire seed {seed} p={p} n={n} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_rooted(lib, seed):
    rng, p, n, dtype, shift = _draw(400 + seed)
    x = _inputs(dtype, p, n, seed)
    root = int(rng.integers(0, p))
    send = _placed(x, dtype, shift)
    # broadcast
    outs = [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    lib.ccl_broadcast(send[root].view, [o.view for o in outs], root=root)
    for r, w in enumerate(collectives.broadcast(x, root)):
        assert_equal(to_host(outs[r].view), w, dtype, f"broadcast seed {seed} rank {r}")
        assert outs[r].guards_intact()
    # reduce (the ring's bits on the root)
    red = Guarded(n, dtype, offset=GUARD + shift)
    lib.ccl_reduce([b.view for b in send], red.view, root=root)
    want_root = collectives.reduce_ring(x, root, dtype)[root]
    assert_equal(to_host(red.view), want_root, dtype, f"reduce seed {seed} p={p} n={n}")
    assert red.guards_intact()
    # scatter then gather back
    parts = [Guarded(ln, dtype, offset=GUARD + int(rng.integers(0, 2))) for _, ln in ring.chunk_bounds(p, n)]
    lib.ccl_scatter(send[root].view, [g.view for g in parts], root=root)
    for k, w in enumerate(collectives.scatter(x[root], p)):
        assert_equal(to_host(parts[k].view), w, dtype, f"scatter seed {seed} rank {k}")
        assert parts[k].guards_intact()
    back = Guarded(n, dtype, offset=GUARD + shift)
    lib.ccl_gather([g.view for g in parts], back.view, root=root)
    assert_equal(to_host(back.view), x[root], dtype, f"gather seed {seed}")
    assert back.guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_all_to_allv(lib, seed):
    rng = np.random.default_rng(500 + seed)
    p = int(rng.choice([1, 2, 3, 5, 8, 13]))
    row = int(rng.choice([1, 2, 3, 7, 8, 64, 129]))
    dtype = str(rng.choice(["f32", "bf16", "i32"]))
    counts = rng.integers(0, int(rng.choice([2, 9, 300])), size=(p, p))
    send_np = [_inputs(dtype, 1, max(int(counts[s].sum()) * row, 1), seed + s)[0][: int(counts[s].sum()) * row]
               for s in range(p)]
    want = collectives.all_to_allv(send_np, counts, row)
    send = _placed(send_np, dtype, int(rng.integers(0, 2)))
    outs = [Guarded(int(counts[:, d].sum()) * row, dtype, offset=GUARD + int(rng.integers(0, 3))) for d in range(p)]
    lib.ccl_all_to_allv([b.view for b in send], counts, [o.view for o in outs], row)
    for d in range(p):
        assert_equal(to_host(outs[d].view), want[d], dtype, f"a2av seed {seed} p={p} row={row} rank {d}")
        assert outs[d].guards_intact()
    # combine with the transposed counts returns every source's rows
    back = [torch.empty_like(b.view) for b in send]
    lib.ccl_all_to_allv([o.view for o in outs], counts.T.copy(), back, row)
    for s in range(p):
        assert_equal(to_host(back[s]), send_np[s], dtype, f"a2av combine seed {seed} rank {s}")
