"""Other all-reduce schedules, simulated literally (oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

"Networks and Collective Communication" section 5.2:

* recursive doubling (p a power of two): at step k device i exchanges its
  whole data with device i XOR 2^k and adds; log2 p steps;
* Rabenseifner: a recursive-halving reduce-scatter (each step a device swaps
  half of the range it is still reducing with its partner and adds the half
  it keeps), then a recursive-doubling all-gather; bytes like the ring,
  steps like the tree;
* binary (binomial) tree: reduce to the root along a binomial tree, then
  broadcast back along it, 2 ceil(log2 p) steps;
* naive: everyone sends to the root, the root sends the sum to everyone.

Section 6.3 (hierarchical all-reduce) and section 6.1 (two-dimensional
all-reduce) add a two-level ring: p = a * b devices in b groups of a (the a
GPUs of a node, or one row of an a x b torus); a ring reduce-scatter inside
every group, a ring all-reduce across the groups among the devices with the
same index inside their group, then a ring all-gather inside every group.

Readings taken where the pages are silent: a receiver computes (received partial) +
(own value) -- IEEE addition is commutative, so only the pairing matters;
the halving step pairs devices at distance p/2 first and a device keeps the
lower half of its range when its bit for that distance is clear, so device i
ends owning chunk i (the ring's chunk rule); the tree's root is device 0 and
at step k device i (a multiple of 2^(k+1)) receives from i + 2^k; the naive
root adds the arrivals in rank order.  bf16 data travels as fp32 partials
and is rounded once by the owner (or root) before the gather / broadcast
phase, as in the ring.  Per-device bytes sent are counted in the size that
travels.
"""
from __future__ import annotations

import math

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16_rne
from .ring import (_check, _finish_chunk, chunk_bounds, combine, ring_all_gather_phase,
                   ring_reduce_scatter_phase)

SCHEDULES = ("recursive_doubling", "rabenseifner", "binomial_tree", "naive")


def _widen(xi, dtype):
    return bf16_to_f32(xi) if dtype == "bf16" else xi.copy()


def _finish(v, dtype):
    if dtype == "bf16":
        return f32_to_bf16_rne(v)
    return v.astype(np.int32 if dtype == "i32" else np.float32, copy=True)


def _e(dtype):
    return 2 if dtype == "bf16" else 4


def _pow2(p):
    if p & (p - 1):
        raise ValueError("this schedule needs p to be a power of two")


def recursive_doubling(x, dtype="f32", op="sum"):
    """Returns (outputs, bytes_sent)."""
    p, n = _check(x, dtype)
    _pow2(p)
    work = [_widen(v, dtype) for v in x]
    sent = [0] * p
    for k in range(int(math.log2(p))):
        msgs = [w.copy() for w in work]  # every device sends its whole data at once
        for i in range(p):
            sent[i] += n * 4
        for i in range(p):
            work[i] = combine(msgs[i ^ (1 << k)], work[i], op)
    return [_finish(w, dtype) for w in work], sent


def rabenseifner(x, dtype="f32", op="sum"):
    """Recursive-halving reduce-scatter then recursive-doubling all-gather."""
    p, n = _check(x, dtype)
    _pow2(p)
    bounds = chunk_bounds(p, n)

    def span(lo, hi):  # element range of chunks [lo, hi)
        return bounds[lo][0], (bounds[hi - 1][0] + bounds[hi - 1][1]) if hi > lo else bounds[lo][0]

    work = [_widen(v, dtype) for v in x]
    lo, hi = [0] * p, [p] * p
    sent = [0] * p
    d = p // 2
    while d >= 1:
        msgs = []
        for i in range(p):
            mid = (lo[i] + hi[i]) // 2
            keep = (lo[i], mid) if (i & d) == 0 else (mid, hi[i])
            give = (mid, hi[i]) if (i & d) == 0 else (lo[i], mid)
            a, b = span(*give)
            msgs.append((give, work[i][a:b].copy()))
            sent[i] += (b - a) * 4
            lo[i], hi[i] = keep
        for i in range(p):
            give, data = msgs[i ^ d]
            assert give == (lo[i], hi[i])  # the partner sends exactly the half this device keeps
            a, b = span(*give)
            work[i][a:b] = combine(data, work[i][a:b], op)
        d //= 2
    assert all(lo[i] == i and hi[i] == i + 1 for i in range(p))
    want = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    out = []
    for i in range(p):
        o = np.zeros(n, dtype=want)
        a, b = span(i, i + 1)
        o[a:b] = _finish(work[i][a:b], dtype)
        out.append(o)
    d = 1
    while d < p:
        msgs = []
        for i in range(p):
            a, b = span(lo[i], hi[i])
            msgs.append(((lo[i], hi[i]), out[i][a:b].copy()))
            sent[i] += (b - a) * _e(dtype)
        for i in range(p):
            (plo, phi), data = msgs[i ^ d]
            a, b = span(plo, phi)
            out[i][a:b] = data
            lo[i], hi[i] = min(lo[i], plo), max(hi[i], phi)
        d *= 2
    return out, sent


def binomial_tree(x, dtype="f32", op="sum"):
    """Reduce to device 0 along a binomial tree, then broadcast back along it."""
    p, n = _check(x, dtype)
    levels = math.ceil(math.log2(p)) if p > 1 else 0
    work = [_widen(v, dtype) for v in x]
    sent = [0] * p
    for k in range(levels):
        step = 1 << k
        for i in range(0, p, 2 * step):
            src = i + step
            if src < p:
                work[i] = combine(work[src].copy(), work[i], op)
                sent[src] += n * 4
    result = _finish(work[0], dtype)
    out = [None] * p
    out[0] = result
    for k in reversed(range(levels)):
        step = 1 << k
        for i in range(0, p, 2 * step):
            dst = i + step
            if dst < p:
                out[dst] = out[i].copy()
                sent[i] += n * _e(dtype)
    return out, sent


def naive(x, dtype="f32", op="sum"):
    """Everyone sends to device 0, which folds the arrivals in rank order and
    sends the result to everyone."""
    p, n = _check(x, dtype)
    sent = [0] * p
    acc = _widen(x[0], dtype)
    for i in range(1, p):
        acc = combine(_widen(x[i], dtype), acc, op)
        sent[i] += n * 4
    result = _finish(acc, dtype)
    out = [result.copy() for _ in range(p)]
    sent[0] += (p - 1) * n * _e(dtype)
    return out, sent


def hierarchical(x, group, dtype="f32", op="sum"):
    """Two-level ring all-reduce over b = p / group groups of `group`
    consecutive ranks (group g = ranks g*a .. g*a + a - 1, a = group).

    Readings taken where the pages are silent: every ring is the ring of ``oracle.ring``
    (rank order inside its ring, chunk rule, chunk c starts after its owner);
    device (g, l) owns chunk l of the a chunks after step 1; in step 2 the
    ring over the groups for chunk l has group g at position g and cuts that
    chunk into b sub-chunks by the same chunk rule, sub-chunk m owned by group
    m; partial sums travel in fp32 (int32) through both reduce-scatters and
    the owner of a sub-chunk rounds bf16 once, before the all-gathers.
    Returns (outputs, bytes_sent).
    """
    p, n = _check(x, dtype)
    a = int(group)
    if a < 1 or p % a:
        raise ValueError("group must divide p")
    b = p // a
    want = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    part = "i32" if dtype == "i32" else "f32"  # what partials travel as
    sent = [0] * p
    # 1. reduce-scatter inside every group
    work = [None] * p
    for g in range(b):
        w, s = ring_reduce_scatter_phase([x[g * a + l] for l in range(a)], dtype, op)
        for l in range(a):
            work[g * a + l] = w[l]
            sent[g * a + l] += s[l]
    out = [np.zeros(n, dtype=want) for _ in range(p)]
    # 2. all-reduce of chunk l across the groups (a rings, one per local index)
    for l, (off, ln) in enumerate(chunk_bounds(a, n)):
        w2, s2 = ring_reduce_scatter_phase([work[g * a + l][off:off + ln] for g in range(b)], part, op)
        bufs = []
        for g, (o2, l2) in enumerate(chunk_bounds(b, ln)):
            buf = np.zeros(ln, dtype=want)
            buf[o2:o2 + l2] = _finish_chunk(w2[g][o2:o2 + l2], dtype)
            bufs.append(buf)
        s3 = ring_all_gather_phase(bufs, dtype)
        for g in range(b):
            sent[g * a + l] += s2[g] + s3[g]
            out[g * a + l][off:off + ln] = bufs[g]
    # 3. all-gather inside every group
    for g in range(b):
        s4 = ring_all_gather_phase([out[g * a + l] for l in range(a)], dtype)
        for l in range(a):
            sent[g * a + l] += s4[l]
    return out, sent


def allreduce(schedule: str, x, dtype="f32", op="sum"):
    fn = {"recursive_doubling": recursive_doubling, "rabenseifner": rabenseifner,
          "binomial_tree": binomial_tree, "naive": naive}[schedule]
    return fn(x, dtype, op)
