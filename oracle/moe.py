"""MoE expert-parallel dispatch / combine with routing (oracle).

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

"Networks and Collective Communication" section 7.4: with expert parallelism
every MoE layer does two all-to-alls -- dispatch (each token goes to the
devices holding the experts it chose) and combine (the expert outputs come
back) -- each device sending about tokens x k x d x bytes x (EP-1)/EP; the
DeepSeek-V3 recipe dispatches in FP8 and combines in BF16.

Readings taken where the pages are silent:

* expert e lives on rank e // (E / p); a token that chose k experts is sent as
  k rows, one per choice (the page's tokens x k accounting);
* destination d receives its rows grouped by source rank (ascending), then by
  token, then by choice (a stable order); ``slot`` is a row's index among the
  rows that its source sends to the same destination, so its row in d's
  buffer is sum_{s' < s} counts[s'][d] + slot;
* FP8 dispatch quantises each row in blocks of 128 elements, the per-tile
  scaling of the DeepSeek-V3 Technical Report that section 7.4 points to
  (its fine-grained quantisation, section 3.3): the block's scaling factor
  scale = amax / 448 maps the largest magnitude onto e4m3's largest finite
  value, quantisation divides by it and dequantisation multiplies by it, so
  code = e4m3(x / scale) (fp32 divisions, each correctly rounded; e4m3
  rounded to nearest even with saturation to +-448).  The report does not
  print the formula; dividing by the factor is the plain meaning of a scaling
  factor that dequantisation multiplies by.  scale travels as fp32; an
  all-zero block gets scale = 1;
* combine: token t's output = bf16( sum_j w[t][j] * y_j ) accumulated in fp32
  in choice order, each product and each sum rounded (no fused multiply-add);
* expert ids outside [0, E) route nowhere (slot -1) and contribute nothing.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16_rne

FP8_MAX = 448.0
FP8_BLOCK = 128


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """fp32 -> float8 e4m3 (1 sign, 4 exponent bits, bias 7, 3 mantissa bits,
    no infinities, 0x7F/0xFF = NaN), round to nearest even, finite values
    saturating at +-448.  Returns uint8 codes."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << 7
    code = np.zeros(x.shape, dtype=np.int64)
    sub = a < 2.0**-6
    # subnormals and zero: multiples of 2^-9 (q = 8 is the smallest normal, 2^-6)
    code[sub] = np.rint(a[sub] / 2.0**-9).astype(np.int64)
    nrm = ~sub & np.isfinite(a)
    m, ex = np.frexp(np.where(nrm, a, 1.0))  # a = m * 2^ex, m in [0.5, 1), exact
    e = ex.astype(np.int64) - 1
    frac = 2.0 * m - 1.0  # [0, 1), exact
    q = np.rint(frac * 8.0).astype(np.int64)
    carry = q == 8
    e = e + carry
    q = np.where(carry, 0, q)
    normal_code = ((e + 7) << 3) | q
    code[nrm] = normal_code[nrm]
    code = np.minimum(code, 0x7E)  # saturate finite values at 448
    code[np.isinf(a)] = 0x7E
    out = code.astype(np.uint8) | sign
    out[np.isnan(x)] = 0x7F
    return out


def e4m3_to_f32(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 7
    v = np.where(e == 0, m * 2.0**-9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return (s * v).astype(np.float32)


def route(expert_ids: list[np.ndarray], p: int, num_experts: int):
    """Returns (counts[p][p] int64, slots per source (int32 per item, -1 when the
    id is out of range), destinations per source (int64, -1 likewise))."""
    if num_experts % p:
        raise ValueError("num_experts must be a multiple of p")
    epr = num_experts // p
    counts = np.zeros((p, p), dtype=np.int64)
    slots, dests = [], []
    for s in range(p):
        ids = np.asarray(expert_ids[s], dtype=np.int64)
        d = np.where((ids >= 0) & (ids < num_experts), ids // epr, -1)
        slot = np.full(ids.shape, -1, dtype=np.int32)
        seen = np.zeros(p, dtype=np.int64)
        for i, di in enumerate(d):  # items in (token, choice) order
            if di >= 0:
                slot[i] = seen[di]
                seen[di] += 1
        counts[s] = seen
        slots.append(slot)
        dests.append(d)
    return counts, slots, dests


def _row_offsets(counts: np.ndarray) -> np.ndarray:
    """base[s][d] = rows of destination d that come from sources before s."""
    return np.vstack([np.zeros((1, counts.shape[1]), dtype=np.int64),
                      np.cumsum(counts, axis=0)[:-1]])


def quantize_rows_fp8(rows_f32: np.ndarray):
    """Per 128-element block: scale = amax / 448 (1 for an all-zero block),
    code = e4m3(x / scale).  Returns (codes uint8, scales float32)."""
    r, h = rows_f32.shape
    blocks = rows_f32.reshape(r, h // FP8_BLOCK, FP8_BLOCK)
    amax = np.abs(blocks).max(axis=2).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(FP8_MAX), np.float32(1.0)).astype(np.float32)
    q = f32_to_e4m3((blocks / scale[:, :, None]).astype(np.float32))
    return q.reshape(r, h), scale


def dispatch(tokens: list[np.ndarray], expert_ids: list[np.ndarray], p: int, k: int,
             num_experts: int, hidden: int, fp8: bool = False):
    """tokens[s]: (T*hidden) bf16 bits.  Returns per destination (rows, scales
    or None, expert id per row), and (counts, slots)."""
    counts, slots, dests = route(expert_ids, p, num_experts)
    base = _row_offsets(counts)
    rows_per_dest = counts.sum(axis=0)
    recv = [np.zeros((int(m), hidden), dtype=np.uint8 if fp8 else np.uint16) for m in rows_per_dest]
    scales = [np.zeros((int(m), hidden // FP8_BLOCK), dtype=np.float32) for m in rows_per_dest] if fp8 else None
    recv_expert = [np.full(int(m), -1, dtype=np.int32) for m in rows_per_dest]
    for s in range(p):
        x = tokens[s].reshape(-1, hidden)
        ids = np.asarray(expert_ids[s]).reshape(-1)
        for i in range(ids.size):
            d = dests[s][i]
            if d < 0:
                continue
            pos = base[s][d] + slots[s][i]
            row = x[i // k]
            if fp8:
                q, sc = quantize_rows_fp8(bf16_to_f32(row)[None, :])
                recv[d][pos] = q[0]
                scales[d][pos] = sc[0]
            else:
                recv[d][pos] = row
            recv_expert[d][pos] = ids[i]
    return recv, scales, recv_expert, counts, slots


def combine(expert_out: list[np.ndarray], expert_ids: list[np.ndarray], weights: list[np.ndarray],
            p: int, k: int, num_experts: int, hidden: int):
    """expert_out[d]: (rows, hidden) bf16 bits in dispatch layout.  Returns per
    source (T*hidden) bf16 bits."""
    counts, slots, dests = route(expert_ids, p, num_experts)
    base = _row_offsets(counts)
    out = []
    for s in range(p):
        ids = np.asarray(expert_ids[s]).reshape(-1)
        w = np.asarray(weights[s], dtype=np.float32).reshape(-1)
        T = ids.size // k
        res = np.zeros((T, hidden), dtype=np.uint16)
        for t in range(T):
            acc = None
            for j in range(k):
                i = t * k + j
                d = dests[s][i]
                if d < 0:
                    continue
                y = bf16_to_f32(expert_out[d][base[s][d] + slots[s][i]])
                prod = (np.float32(w[i]) * y).astype(np.float32)
                acc = prod if acc is None else (acc + prod).astype(np.float32)
            res[t] = f32_to_bf16_rne(acc if acc is not None else np.zeros(hidden, np.float32))
        out.append(res.reshape(-1))
    return out
