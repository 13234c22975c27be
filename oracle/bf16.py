"""bf16 <-> fp32 conversions for the oracle (test infrastructure only).

bf16 is the top 16 bits of an IEEE binary32.  Widening is exact (append 16
zero bits).  Narrowing rounds to nearest, ties to even, by the published bit
method: add 0x7FFF plus the lowest kept bit, then drop the low 16 bits.  A NaN
stays a NaN (its top bits are kept and the quiet bit is set), and finite
values that round past the largest bf16 become +-inf, as IEEE rounding does.

Pinned in ``tests/test_oracle_bf16.py`` against torch's own fp32 -> bf16 cast
on a grid that includes exact ties, subnormals, overflow and infinities.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening: uint16 bit patterns -> float32 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16, nearest-even; returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    rounded = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(np.ascontiguousarray(x, dtype=np.float32))
    if nan.any():
        quiet = ((u >> np.uint32(16)) | np.uint32(0x0040)).astype(np.uint16)
        rounded = np.where(nan, quiet, rounded)
    return rounded
