"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws numbers.  It holds none of the collectives' arithmetic:
no fold, no chunk rule, no rounding of results.  Both sides of every parity
check consume the exact bytes produced here.

Workloads (sizes follow the pages' examples):

* ``worked_example``  -- 4 devices, device d holds [10d, 10d+1, 10d+2, 10d+3]
  ("Networks and Collective Communication", section 4.1).
* ``normal``          -- N(0, sigma) per rank; sigma is a standard deviation.
  Used for the p=4 fp32 case (sigma 1, seed 0), the 25 MB DDP bucket
  (p=8, sigma 1e-3, seed 1; "dist_train", DDP bucketing, bucket_cap_mb=25)
  and the 192 MiB ZeRO gradients (p=16, bf16, sigma 1e-2, seed 2).
* ``uniform``         -- U(-1, 1) per rank for the message-size sweep (seed 4).
* ``moe_counts`` / ``moe_tokens`` -- MoE dispatch: p=8 ranks, each sends
  16,384 tokens whose destination expert is drawn from a Zipf(1.2) law over
  8 experts (one expert per rank, the same hot expert for every source).

bf16 values are produced by drawing fp32 and converting with torch's own
round-to-nearest-even cast (a library routine), then returned as raw uint16
bit patterns so that numpy code can hold them.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "worked_example",
    "normal",
    "uniform",
    "integer_valued",
    "to_bf16_bits",
    "moe_zipf_probs",
    "moe_counts",
    "moe_tokens",
]


def worked_example(p: int = 4, dtype=np.float32) -> list[np.ndarray]:
    """Device d holds [10d, 10d+1, ..., 10d+p-1] (section 4.1 uses p = 4)."""
    return [np.array([10 * d + j for j in range(p)], dtype=dtype) for d in range(p)]


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 via torch's cast; returns the uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32, copy=False)
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(f"unsupported dtype {dtype!r}")


def normal(p: int, n: int, sigma: float, seed: int, dtype: str = "f32") -> list[np.ndarray]:
    """p rank buffers of n values ~ N(0, sigma), drawn in rank order from one stream."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(p):
        x = rng.standard_normal(n, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        out.append(_finish(x, dtype))
    return out


def uniform(p: int, n: int, seed: int, dtype: str = "f32") -> list[np.ndarray]:
    """p rank buffers of n values ~ U(-1, 1), drawn in rank order from one stream."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(p):
        x = rng.random(n, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)
        out.append(_finish(x, dtype))
    return out


def integer_valued(p: int, n: int, seed: int, lo: int = -1000, hi: int = 1000,
                   dtype: str = "f32") -> list[np.ndarray]:
    """Small integers, so any fold order gives the exact sum (|sum| << 2^24)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(p):
        x = rng.integers(lo, hi + 1, size=n)
        if dtype == "i32":
            out.append(x.astype(np.int32))
        else:
            out.append(_finish(x.astype(np.float32), dtype))
    return out


def moe_zipf_probs(experts: int = 8, s: float = 1.2) -> np.ndarray:
    """pi_e proportional to (e+1)^-s, e = 0..experts-1."""
    w = (np.arange(experts, dtype=np.float64) + 1.0) ** (-s)
    return w / w.sum()


def moe_counts(p: int = 8, tokens_per_rank: int = 16384, s: float = 1.2,
               seed: int = 3) -> tuple[np.ndarray, np.random.Generator]:
    """counts[src][dst] token rows; row s ~ Multinomial(tokens_per_rank, pi).

    Returns the counts and the generator, so that the token payload is drawn
    from the same stream right after the counts.
    """
    rng = np.random.default_rng(seed)
    pi = moe_zipf_probs(p, s)
    counts = np.stack([rng.multinomial(tokens_per_rank, pi) for _ in range(p)]).astype(np.int64)
    return counts, rng


def moe_tokens(counts: np.ndarray, hidden: int, rng: np.random.Generator,
               dtype: str = "bf16") -> list[np.ndarray]:
    """Per source rank: sum_d counts[s][d] rows of `hidden` values ~ N(0, 1), flat."""
    out = []
    for s in range(counts.shape[0]):
        rows = int(counts[s].sum())
        x = rng.standard_normal(rows * hidden, dtype=np.float32)
        out.append(_finish(x, dtype))
    return out


def moe_topk_routing(p: int, tokens: int, k: int, num_experts: int, s: float = 1.2,
                     seed: int = 3) -> list[np.ndarray]:
    """Per source: (tokens, k) int32 distinct expert ids, drawn without
    replacement with Zipf(s) popularity over the experts (Gumbel top-k)."""
    rng = np.random.default_rng(seed)
    logw = np.log((np.arange(num_experts, dtype=np.float64) + 1.0) ** (-s))
    out = []
    for _ in range(p):
        g = rng.gumbel(size=(tokens, num_experts)) + logw
        out.append(np.argsort(-g, axis=1)[:, :k].astype(np.int32))
    return out


def moe_gate_weights(p: int, tokens: int, k: int, seed: int = 4) -> list[np.ndarray]:
    """Per source: (tokens, k) positive float32 gate weights summing to ~1 per token."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(p):
        w = rng.random((tokens, k)) + 0.05
        out.append((w / w.sum(axis=1, keepdims=True)).astype(np.float32))
    return out
