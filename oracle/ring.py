"""Literal ring simulator: reduce-scatter, all-gather, all-reduce (oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

The ring, as the pages give it ("Networks and Collective Communication"
section 5.1 and Exercise 2; "dist_train", "Ring Algorithm"; "LLM Distributed
Training Collectives", "Ring AllReduce"):

* the p devices form a logical ring, every device talks only to its next
  neighbour, and each device's data is cut into p chunks;
* reduce-scatter phase, p-1 steps: at every step every device passes one
  partial sum (one chunk) to the next device, which adds its own chunk to
  it; after p-1 steps every device holds one fully reduced chunk;
* all-gather phase, p-1 steps: at every step every device passes the
  complete chunk it received most recently to the next device;
* every device sends n/p per step, 2(p-1) steps in all.

Readings taken where the pages are silent:

1. Chunk split when p does not divide n: numpy's ``array_split`` rule --
   the first (n mod p) chunks get floor(n/p)+1 elements, the rest floor(n/p).
   (The pages' simulator is numpy.)
2. Direction and ownership: rank r sends to rank r+1 (mod p).  In RS step s
   (s = 0..p-2) rank r sends its partial of chunk (r-s-1) mod p and the
   receiver adds its own chunk to it.  Chunk c therefore starts at rank c+1
   and ends at rank c, so after the phase rank k holds chunk k, which matches
   "process k gets sum_i x_i^(k)" (dist_train, Reduce-Scatter).  In AG step s
   rank r sends chunk (r-s) mod p.
3. bf16 inputs: the partial travels and accumulates in fp32; the owner rounds
   its finished chunk to bf16 once (nearest-even) and the AG phase moves bf16.
   The variant ``wire="bf16"`` sends the partial as bf16 instead: every hop
   adds in fp32 and rounds the new partial to bf16 (nearest-even) before it
   travels on, so the reduce-scatter moves 2 bytes per element.
4. MAX/MIN (not on the pages; extras of the library): the receiver keeps its
   own value when it is strictly greater (smaller), else the received partial.

The simulation is literal: at each step all outgoing messages are copied
first (every device sends at once), then every receiver combines.  Each
device's count of bytes sent is kept, in the element size that travels.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16_rne

DTYPES = ("f32", "bf16", "i32")
OPS = ("sum", "max", "min")


# ---------------------------------------------------------------- chunk rule
def chunk_bounds(p: int, n: int) -> list[tuple[int, int]]:
    """(offset, length) of each of the p chunks of an n-element buffer (reading 1)."""
    if p < 1 or n < 0:
        raise ValueError("need p >= 1 and n >= 0")
    base, extra = divmod(n, p)
    bounds = []
    off = 0
    for c in range(p):
        ln = base + (1 if c < extra else 0)
        bounds.append((off, ln))
        off += ln
    return bounds


# ------------------------------------------------------------- element types
def _check(x: list[np.ndarray], dtype: str) -> tuple[int, int]:
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {DTYPES}")
    p = len(x)
    if p < 1:
        raise ValueError("need at least one rank")
    n = len(x[0])
    want = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    for xi in x:
        if xi.ndim != 1 or len(xi) != n or xi.dtype != want:
            raise ValueError("every rank buffer must be 1-D, of the same length and dtype")
    return p, n


def _widen(xi: np.ndarray, dtype: str) -> np.ndarray:
    """The value a rank starts its partial with (fp32 for f32/bf16, int32 for i32)."""
    if dtype == "bf16":
        return bf16_to_f32(xi)
    return xi.copy()


def combine(received: np.ndarray, own: np.ndarray, op: str) -> np.ndarray:
    """What a receiving rank computes from the partial it got and its own chunk."""
    if op == "sum":
        return received + own  # fp32 add (or int32 add, which wraps)
    if op == "max":
        return np.where(own > received, own, received)
    if op == "min":
        return np.where(own < received, own, received)
    raise ValueError(f"op must be one of {OPS}")


def _wire_size_rs(dtype: str, wire: str = "fp32") -> int:
    if wire == "bf16":
        return 2  # bf16 partials
    return 4  # fp32 partials (f32 and bf16) or int32 partials


def _check_wire(dtype: str, wire: str) -> None:
    if wire not in ("fp32", "bf16"):
        raise ValueError("wire must be 'fp32' or 'bf16'")
    if wire == "bf16" and dtype != "bf16":
        raise ValueError("a bf16 wire needs bf16 data")


def _elem_size(dtype: str) -> int:
    return 2 if dtype == "bf16" else 4


# ------------------------------------------------------------------ RS phase
def ring_reduce_scatter_phase(x: list[np.ndarray], dtype: str = "f32", op: str = "sum",
                              wire: str = "fp32"):
    """Run the p-1 reduce-scatter steps on copies of the rank buffers.

    Returns (work, bytes_sent): ``work[r]`` is rank r's full working buffer
    after the phase (fp32 for f32/bf16, int32 for i32); its chunk r is the
    complete reduction.  ``bytes_sent[r]`` counts the bytes rank r sent.
    """
    p, n = _check(x, dtype)
    if op not in OPS:
        raise ValueError(f"op must be one of {OPS}")
    _check_wire(dtype, wire)
    bounds = chunk_bounds(p, n)
    wire_bytes = _wire_size_rs(dtype, wire)
    work = [_widen(xi, dtype) for xi in x]
    sent = [0] * p
    for s in range(p - 1):
        # every rank sends at once: copy all outgoing partials first
        messages = []
        for r in range(p):
            c = (r - s - 1) % p
            off, ln = bounds[c]
            messages.append((c, work[r][off:off + ln].copy()))
            sent[r] += ln * wire_bytes
        for r in range(p):
            c, msg = messages[r]
            dst = (r + 1) % p
            off, ln = bounds[c]
            part = combine(msg, work[dst][off:off + ln], op)
            if wire == "bf16":  # the new partial is what travels: round it now
                part = bf16_to_f32(f32_to_bf16_rne(part))
            work[dst][off:off + ln] = part
    return work, sent


def _finish_chunk(values: np.ndarray, dtype: str) -> np.ndarray:
    """The owner's finished chunk in the output dtype (one bf16 rounding)."""
    if dtype == "bf16":
        return f32_to_bf16_rne(values)
    return values.astype({"f32": np.float32, "i32": np.int32}[dtype], copy=True)


def ring_reduce_scatter(x: list[np.ndarray], dtype: str = "f32", op: str = "sum", wire: str = "fp32"):
    """Reduce-scatter: rank k gets chunk k of the ring-ordered reduction.

    Returns (shards, bytes_sent); ``shards[k]`` has len(chunk k) elements of
    the input dtype.
    """
    work, sent = ring_reduce_scatter_phase(x, dtype, op, wire)
    bounds = chunk_bounds(len(x), len(x[0]))
    shards = []
    for k, (off, ln) in enumerate(bounds):
        shards.append(_finish_chunk(work[k][off:off + ln], dtype))
    return shards, sent


# ------------------------------------------------------------------ AG phase
def ring_all_gather_phase(bufs: list[np.ndarray], dtype: str = "f32"):
    """Run the p-1 all-gather steps in place on full-size rank buffers.

    On entry rank r's chunk r is valid; on return every rank holds every
    chunk.  Returns bytes_sent per rank.
    """
    p = len(bufs)
    n = len(bufs[0])
    bounds = chunk_bounds(p, n)
    e = _elem_size(dtype)
    sent = [0] * p
    for s in range(p - 1):
        messages = []
        for r in range(p):
            c = (r - s) % p
            off, ln = bounds[c]
            messages.append((c, bufs[r][off:off + ln].copy()))
            sent[r] += ln * e
        for r in range(p):
            c, msg = messages[r]
            dst = (r + 1) % p
            off, ln = bounds[c]
            bufs[dst][off:off + ln] = msg
    return sent


def ring_all_gather(shards: list[np.ndarray], dtype: str = "f32"):
    """All-gather: rank k contributes chunk k (len(k) elements); every rank gets
    the concatenation.  Returns (outputs, bytes_sent)."""
    p = len(shards)
    n = sum(len(s) for s in shards)
    bounds = chunk_bounds(p, n)
    for k, (off, ln) in enumerate(bounds):
        if len(shards[k]) != ln:
            raise ValueError(f"rank {k} must contribute {ln} elements (chunk rule)")
    want = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    bufs = []
    for k, (off, ln) in enumerate(bounds):
        b = np.zeros(n, dtype=want)  # bytes outside chunk k are not valid yet
        b[off:off + ln] = shards[k]
        bufs.append(b)
    sent = ring_all_gather_phase(bufs, dtype)
    return bufs, sent


# ------------------------------------------------------------------ all-reduce
def ring_allreduce(x: list[np.ndarray], dtype: str = "f32", op: str = "sum", wire: str = "fp32"):
    """All-reduce = the RS phase then the AG phase on the same working buffers.

    Returns (outputs, bytes_sent_rs, bytes_sent_ag).  For bf16 the owner of
    each chunk rounds it to bf16 between the phases (reading 3).
    """
    work, sent_rs = ring_reduce_scatter_phase(x, dtype, op, wire)
    p, n = len(x), len(x[0])
    bounds = chunk_bounds(p, n)
    want = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    bufs = []
    for r in range(p):
        b = np.zeros(n, dtype=want)
        off, ln = bounds[r]
        b[off:off + ln] = _finish_chunk(work[r][off:off + ln], dtype)
        bufs.append(b)
    sent_ag = ring_all_gather_phase(bufs, dtype)
    return bufs, sent_rs, sent_ag


# ------------------------------------------------ DDP bucket: scale and cast
def bucket_allreduce_scale_cast(grads: list[np.ndarray], scale: float):
    """DDP gradient bucket: ring all-reduce of fp32 gradients, times ``scale``
    (1/p for an average) in fp32, rounded once to bf16 (nearest-even).

    "dist_train", Communication-Computation Overlap: DDP buckets gradients
    (bucket_cap_mb=25) and all-reduces each bucket; the 1/p average and the
    bf16 output are the fused epilogue.  Returns per-rank uint16 bf16 bits.
    """
    summed, _, _ = ring_allreduce(grads, "f32", "sum")
    s = np.float32(scale)
    return [f32_to_bf16_rne(v * s) for v in summed]


def zero_rs_then_ag(x_bf16: list[np.ndarray]):
    """ZeRO chain: reduce-scatter of bf16 gradients with fp32 accumulation,
    then all-gather of the bf16 shards.  Returns (shards, gathered)."""
    shards, _ = ring_reduce_scatter(x_bf16, "bf16", "sum")
    gathered, _ = ring_all_gather(shards, "bf16")
    return shards, gathered
