"""The ring-ordered fold written per output element (oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Following the ring of "Networks and Collective Communication" section 5.1
with the readings of ``oracle/ring.py``: element i lies in chunk c; chunk c's
partial starts at rank c+1 and collects ranks c+2, ..., p-1, 0, ..., c in that
order, each receiver combining the received partial with its own value.  The
all-gather phase only copies, so every rank's output at i is that fold.

This evaluates the fold for an explicit set of indices, so that huge buffers
can be checked at sampled positions.  It is checked against the literal
simulator ``oracle.ring`` in ``tests/test_oracle_ring.py``.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16_rne
from .ring import chunk_bounds, combine


def chunk_of(p: int, n: int, idx: np.ndarray) -> np.ndarray:
    """Chunk number of each index (by scanning the chunk table)."""
    bounds = chunk_bounds(p, n)
    starts = np.array([off for off, _ in bounds], dtype=np.int64)
    ends = np.array([off + ln for off, ln in bounds], dtype=np.int64)
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= n):
        raise IndexError("index out of range")
    out = np.empty(idx.shape, dtype=np.int64)
    for c in range(p):
        if ends[c] > starts[c]:
            sel = (idx >= starts[c]) & (idx < ends[c])
            out[sel] = c
    return out


def fold_columns(cols: list[np.ndarray], idx: np.ndarray, n: int, dtype: str = "f32",
                 op: str = "sum", wire: str = "fp32"):
    """The fold at indices ``idx`` of n-element rank buffers, given only the
    sampled values: ``cols[r][j]`` is rank r's element ``idx[j]``.  With
    ``wire="bf16"`` every hop's new partial is rounded to bf16 (the ring's
    bf16-wire variant, ``oracle.ring``)."""
    p = len(cols)
    idx = np.asarray(idx, dtype=np.int64)
    chunks = chunk_of(p, n, idx)
    acc_dtype = np.int32 if dtype == "i32" else np.float32
    out = np.empty(idx.shape, dtype=acc_dtype)

    def value(rank, mask):
        v = cols[rank][mask]
        return bf16_to_f32(v) if dtype == "bf16" else v.astype(acc_dtype, copy=True)

    for c in range(p):
        mask = chunks == c
        if not mask.any():
            continue
        acc = value((c + 1) % p, mask)
        for j in range(2, p + 1):
            acc = combine(acc, value((c + j) % p, mask), op)
            if wire == "bf16":
                acc = bf16_to_f32(f32_to_bf16_rne(acc))
        out[mask] = acc
    return out


def fold_at(x: list[np.ndarray], idx: np.ndarray, dtype: str = "f32", op: str = "sum"):
    """Reduced value at each index in ``idx`` (fp32/int32 accumulator, unrounded)."""
    idx = np.asarray(idx, dtype=np.int64)
    return fold_columns([xr[idx] for xr in x], idx, len(x[0]), dtype, op)


def allreduce_at(x: list[np.ndarray], idx: np.ndarray, dtype: str = "f32", op: str = "sum"):
    """All-reduce output (any rank) at the given indices, in the output dtype."""
    acc = fold_at(x, idx, dtype, op)
    return f32_to_bf16_rne(acc) if dtype == "bf16" else acc


def allreduce_at_columns(cols: list[np.ndarray], idx: np.ndarray, n: int, dtype: str = "f32",
                         op: str = "sum", wire: str = "fp32"):
    """All-reduce output at ``idx`` from sampled columns (see ``fold_columns``)."""
    acc = fold_columns(cols, idx, n, dtype, op, wire)
    return f32_to_bf16_rne(acc) if dtype == "bf16" else acc


def bucket_at(grads: list[np.ndarray], idx: np.ndarray, scale: float):
    """DDP bucket output (any rank) at the given indices: bf16(fold * scale)."""
    acc = fold_at(grads, idx, "f32", "sum")
    return f32_to_bf16_rne(acc * np.float32(scale))


def hierarchical_at_columns(cols: list[np.ndarray], idx: np.ndarray, n: int, group: int,
                            dtype: str = "f32"):
    """The two-level ring fold ("Networks and Collective Communication"
    sections 6.3 and 6.1; the readings of ``oracle.schedules.hierarchical``)
    at indices ``idx``, in the output dtype: element i lies in chunk l of the
    a = group chunks and in sub-chunk m of that chunk's b = p / a pieces; each
    group's value is its ring fold from local rank l + 1 to l, and the group
    values are folded from group m + 1 to m.  Checked against the literal
    simulation in ``tests/test_oracle_schedules.py``."""
    p = len(cols)
    a = int(group)
    if a < 1 or p % a:
        raise ValueError("group must divide p")
    b = p // a
    idx = np.asarray(idx, dtype=np.int64)
    acc_dtype = np.int32 if dtype == "i32" else np.float32
    out = np.empty(idx.shape, dtype=acc_dtype)
    level1 = chunk_bounds(a, n)
    l_of = chunk_of(a, n, idx)

    def value(rank, mask):
        v = cols[rank][mask]
        return bf16_to_f32(v) if dtype == "bf16" else v.astype(acc_dtype, copy=True)

    for l in range(a):
        in_l = l_of == l
        if not in_l.any():
            continue
        off, ln = level1[l]
        m_of = np.full(idx.shape, -1, dtype=np.int64)
        m_of[in_l] = chunk_of(b, ln, idx[in_l] - off)
        for m in range(b):
            mask = in_l & (m_of == m)
            if not mask.any():
                continue
            tot = None
            for gi in range(1, b + 1):
                g = (m + gi) % b
                part = value(g * a + (l + 1) % a, mask)
                for li in range(2, a + 1):
                    part = combine(part, value(g * a + (l + li) % a, mask), "sum")
                tot = part if tot is None else combine(tot, part, "sum")
            out[mask] = tot
    return f32_to_bf16_rne(out) if dtype == "bf16" else out


def all_gather_source(p: int, n: int, idx: np.ndarray):
    """Where the all-gather's output element ``idx`` comes from ("Networks and
    Collective Communication" section 4.1: rank k contributes block k, which
    lands at off(k) of every rank's output): the contributing rank k (the
    chunk holding idx) and the position idx - off(k) in its block."""
    idx = np.asarray(idx, dtype=np.int64)
    k = chunk_of(p, n, idx)
    offs = np.array([off for off, _ in chunk_bounds(p, n)], dtype=np.int64)
    return k, idx - offs[k]


def all_to_all_source(p: int, n: int, j: int, idx: np.ndarray):
    """Where rank j's all-to-all output element ``idx`` comes from (section
    4.1, the transpose: rank j receives block j of every rank, in source
    order, so its output is p blocks of len(j)): the source rank
    idx // len(j) and the position off(j) + idx mod len(j) in its buffer."""
    idx = np.asarray(idx, dtype=np.int64)
    off, ln = chunk_bounds(p, n)[j]
    if idx.size and (idx.min() < 0 or idx.max() >= p * ln):
        raise IndexError("index out of range")
    return idx // ln, off + idx % ln


def all_to_allv_source(counts: np.ndarray, d: int, rows: np.ndarray):
    """Where destination d's received row ``rows`` comes from in the
    row-granular all-to-allv (the layout of ``oracle.collectives.all_to_allv``:
    d holds its blocks in source order, source s holds its blocks in
    destination order): the source rank s and the row of s's send buffer."""
    counts = np.asarray(counts, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    recv_start = np.concatenate([[0], np.cumsum(counts[:, d])])      # d's block from s starts here
    if rows.size and (rows.min() < 0 or rows.max() >= recv_start[-1]):
        raise IndexError("row out of range")
    src = np.searchsorted(recv_start, rows, side="right") - 1
    send_start = np.concatenate([np.zeros((counts.shape[0], 1), np.int64), np.cumsum(counts, axis=1)], axis=1)
    return src, send_start[src, d] + (rows - recv_start[src])
