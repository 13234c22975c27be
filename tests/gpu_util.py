"""Helpers for the GPU parity tests: host<->device moves, guard bands, bf16 ulps."""
from __future__ import annotations

import numpy as np
import torch

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
NP_DT = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}
GUARD = 64  # elements of guard band on each side of an output (keeps 16-byte alignment)


def ccl():
    """The binding, with the library built first if it is out of date."""
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl as mod

    return mod


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


class Guarded:
    """A device buffer of n elements with sentinel-filled guard bands around it.

    ``view`` is the buffer handed to the library, starting ``offset`` elements
    into the storage (offset GUARD keeps 16-byte alignment; GUARD+1 breaks it).
    """

    def __init__(self, n: int, dtype: str, offset: int = GUARD):
        self.n, self.offset, self.dtype = n, offset, dtype
        total = n + offset + GUARD
        self.store = torch.empty(total, dtype=TORCH_DT[dtype], device="cuda")
        # sentinel: an fp32 / bf16 / int32 bit pattern the collectives never produce here
        self.store.view(torch.int16 if dtype == "bf16" else torch.int32).fill_(0x5A5A if dtype == "bf16" else 0x5A5A5A5A)
        self.sentinel = to_host(self.store[:1])[0]
        self.view = self.store[offset:offset + n]

    def guards_intact(self) -> bool:
        h = to_host(self.store)
        before, after = h[:self.offset], h[self.offset + self.n:]
        s = self.sentinel
        if self.dtype == "f32":
            return bool((before.view(np.int32) == s.view(np.int32)).all()
                        and (after.view(np.int32) == s.view(np.int32)).all())
        return bool((before == s).all() and (after == s).all())


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in bf16 units in the last place (bit patterns, monotone ordering)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))


def assert_bf16_close(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    """The contract: at most 1 bf16 ulp from the oracle; the design is bit-exact,
    so the number of differing elements is asserted to be zero too."""
    d = bf16_ulp_diff(got, want)
    assert d.max(initial=0) <= 1, f"{what}: max bf16 ulp difference {d.max()}"
    assert int((d != 0).sum()) == 0, f"{what}: {(d != 0).sum()} elements differ by 1 ulp"


def assert_equal(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "") -> None:
    if dtype == "bf16":
        assert_bf16_close(got, want, what)
    elif dtype == "f32":
        # bit-exact, NaN payloads included
        np.testing.assert_array_equal(got.view(np.int32), want.view(np.int32), err_msg=what)
    else:
        np.testing.assert_array_equal(got, want, err_msg=what)


def sample_indices(n: int, p: int, count: int, seed: int) -> np.ndarray:
    """Random indices plus every chunk edge and both buffer ends."""
    from oracle.ring import chunk_bounds

    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, n, size=count)]
    edges = []
    for off, ln in chunk_bounds(p, n):
        edges += [off - 1, off, off + 1, off + ln - 1, off + ln]
    edges += [0, 1, n - 2, n - 1]
    idx.append(np.array([e for e in edges if 0 <= e < n], dtype=np.int64))
    return np.unique(np.concatenate(idx))
