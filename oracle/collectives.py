"""Collective primitives by their definitions (oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

"Networks and Collective Communication" section 4.1 and "dist_train",
"Collective Communication Primitives":

* broadcast  -- the root's data is copied to everyone;
* reduce     -- element-wise sum, result only on the root;
* scatter    -- the root holds [x_1, ..., x_p]; rank k receives x_k;
* gather     -- rank k holds x_k; the root receives [x_1, ..., x_p];
* all-gather -- every rank contributes one block and everyone gets the whole
                concatenation;
* all-to-all -- device i's block j goes to device j (rows = devices, columns
                = blocks: a transpose); MoE expert parallelism dispatches
                tokens with it.

Blocks follow the same chunk rule as the ring (``oracle.ring.chunk_bounds``).
The all-to-allv form (reading 9) carries whole rows: ``counts[s][d]`` rows go
from source s to destination d; a source's buffer holds its blocks in
destination order, a destination's buffer receives them in source order.
"""
from __future__ import annotations

import numpy as np

from .ring import chunk_bounds


def broadcast(x: list[np.ndarray], root: int = 0) -> list[np.ndarray]:
    return [x[root].copy() for _ in x]


def reduce(x: list[np.ndarray], root: int = 0) -> list[np.ndarray | None]:
    """Element-wise sum, only on the root.  The pages fix no order for it; this
    sums in rank order 0..p-1 (used only with exactly representable sums)."""
    acc = x[0].copy()
    for xi in x[1:]:
        acc = acc + xi
    return [acc if r == root else None for r in range(len(x))]


def reduce_ring(x: list[np.ndarray], root: int = 0, dtype: str = "f32", op: str = "sum"):
    """Reduce built as the ring's reduce-scatter followed by a gather of the
    shards to the root (the pages fix no order for reduce; this reading gives
    the root exactly the ring all-reduce's bits).  Returns one entry per
    rank: the result at index ``root``, None for the other ranks."""
    from .ring import ring_reduce_scatter

    shards, _ = ring_reduce_scatter(x, dtype, op)
    whole = np.concatenate(shards) if shards else np.zeros(0)
    return [whole if r == root else None for r in range(len(x))]


def scatter(data: np.ndarray, p: int) -> list[np.ndarray]:
    """Root's buffer cut into p chunks; rank k receives chunk k."""
    return [data[off:off + ln].copy() for off, ln in chunk_bounds(p, len(data))]


def gather(parts: list[np.ndarray], root: int = 0) -> list[np.ndarray | None]:
    whole = np.concatenate(parts)
    return [whole if r == root else None for r in range(len(parts))]


def all_gather(parts: list[np.ndarray]) -> list[np.ndarray]:
    whole = np.concatenate(parts)
    return [whole.copy() for _ in parts]


def all_to_all(x: list[np.ndarray]) -> list[np.ndarray]:
    """recv[j] = concat_i (block j of x[i]) -- the block transpose."""
    p = len(x)
    blocks = [[xi[off:off + ln] for off, ln in chunk_bounds(p, len(xi))] for xi in x]
    return [np.concatenate([blocks[i][j] for i in range(p)]) for j in range(p)]


def all_to_allv(send: list[np.ndarray], counts: np.ndarray, row_elems: int) -> list[np.ndarray]:
    """Row-granular all-to-all with per-pair counts (MoE dispatch).

    send[s] holds sum_d counts[s][d] rows, its block for d starting at row
    sum_{d' < d} counts[s][d']; recv[d] holds sum_s counts[s][d] rows, the
    block from s starting at row sum_{s' < s} counts[s'][d].  Combine is the
    same call on the received buffers with counts transposed.
    """
    counts = np.asarray(counts, dtype=np.int64)
    p = counts.shape[0]
    if counts.shape != (p, p) or len(send) != p:
        raise ValueError("counts must be p x p")
    blocks = []
    for s in range(p):
        if len(send[s]) != counts[s].sum() * row_elems:
            raise ValueError(f"send[{s}] has the wrong length")
        row = []
        start = 0
        for d in range(p):
            ln = int(counts[s][d]) * row_elems
            row.append(send[s][start:start + ln])
            start += ln
        blocks.append(row)
    return [np.concatenate([blocks[s][d] for s in range(p)]) if p else np.zeros(0)
            for d in range(p)]


def ulysses_seq_to_heads(x: list[np.ndarray], heads: int, head_dim: int) -> list[np.ndarray]:
    """Sequence-parallel attention's all-to-all ("LLM Distributed Training
    Collectives", Sequence Parallelism / Ulysses): rank r holds sequence shard r
    with every head, shape [S/p, H, D]; afterwards rank r holds the whole
    sequence for head group r, [S, H/p, D]:
        y_r[s * S/p + t, h, :] = x_s[t, r * H/p + h, :]."""
    p = len(x)
    if heads % p:
        raise ValueError("heads must be a multiple of p")
    hp = heads // p
    xs = [xi.reshape(-1, heads, head_dim) for xi in x]
    return [np.concatenate([xs[s][:, r * hp:(r + 1) * hp, :] for s in range(p)], axis=0).reshape(-1)
            for r in range(p)]


def ulysses_heads_to_seq(y: list[np.ndarray], heads: int, head_dim: int) -> list[np.ndarray]:
    """The inverse exchange: [S, H/p, D] per head group back to [S/p, H, D] per
    sequence shard: x_s[t, r * H/p + h, :] = y_r[s * S/p + t, h, :]."""
    p = len(y)
    hp = heads // p
    ys = [yi.reshape(-1, hp, head_dim) for yi in y]
    sp = ys[0].shape[0] // p
    return [np.concatenate([ys[r][s * sp:(s + 1) * sp] for r in range(p)], axis=1).reshape(-1)
            for s in range(p)]
