"""Pin the oracle's fp32 -> bf16 rounding against torch's own cast."""
from __future__ import annotations

import numpy as np
import torch

from oracle.bf16 import bf16_to_f32, f32_to_bf16_rne


def _torch_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _grid() -> np.ndarray:
    rng = np.random.default_rng(0)
    specials = np.array(
        [0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
         3.4028235e38, 1e-45, -1e-45, 1.17549435e-38, 5.9e-39, 65504.0],
        dtype=np.float32,
    )
    # exact ties: a bf16 value plus exactly half an ulp (low 16 bits = 0x8000),
    # with both parities of the kept lsb
    base = rng.integers(0, 2**31, size=4096, dtype=np.uint32) & np.uint32(0x7F7F0000)
    ties = (base | np.uint32(0x8000)).view(np.float32)
    near = np.concatenate([(base | np.uint32(0x7FFF)).view(np.float32),
                           (base | np.uint32(0x8001)).view(np.float32)])
    rand = rng.integers(0, 2**32, size=200_000, dtype=np.uint32).view(np.float32)
    rand = rand[~np.isnan(rand)]
    return np.concatenate([specials, ties, -ties, near, rand])


def test_rne_matches_torch_cast():
    x = _grid()
    np.testing.assert_array_equal(f32_to_bf16_rne(x), _torch_bits(x))


def test_nan_stays_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    assert np.isnan(bf16_to_f32(f32_to_bf16_rne(x))).all()


def test_widening_is_exact_and_round_trips():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    bits = bits[~np.isnan(bf16_to_f32(bits))]
    f = bf16_to_f32(bits)
    np.testing.assert_array_equal(f32_to_bf16_rne(f), bits)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(f, t)
