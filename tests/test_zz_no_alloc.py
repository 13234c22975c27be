"""The allocation-free reduce-scatter (ccl_ring_reduce_scatter_literal_noalloc).

Some callers of this library cannot allocate device memory -- code inside an
allocator callback, or under a host application that owns all device memory
-- so they cannot provide the workspace the literal reduce-scatter needs.
This entry point uses the library's built-in static scratch instead.  These
tests check that two calls in a row give exactly what the workspace entry
point gives, and that sizes beyond the scratch are refused up front.  The
file is named to be collected last.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import assert_equal, to_dev, to_host

SCRATCH_ELEMS = (32 << 20) // 4  # p*n limit: 32 MiB of fp32 working buffers


def _lib():
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl

    return ccl


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    lib = _lib()
    cases = [("f32", 8, 1_000_003, 1), ("bf16", 16, 500_001, 2)]  # each near the 32 MiB limit
    assert all(p * n <= SCRATCH_ELEMS for _, p, n, _ in cases)
    for dtype, p, n, seed in cases:
        x = workloads.normal(p, n, 1.0, seed=seed, dtype=dtype)
        send = [to_dev(v, dtype) for v in x]
        sizes = [lib.ccl_chunk_bounds(p, n, k)[1] for k in range(p)]
        want = [torch.empty(s, dtype=send[0].dtype, device="cuda") for s in sizes]
        got = [torch.full((s,), 7, dtype=send[0].dtype, device="cuda") for s in sizes]
        sent_want = lib.ccl_ring_reduce_scatter_literal(send, want)
        sent_got = lib.ccl_ring_reduce_scatter_literal_noalloc(send, got)
        torch.cuda.synchronize()
        assert sent_got == sent_want
        for k in range(p):
            assert_equal(to_host(got[k]), to_host(want[k]), dtype, f"{dtype} shard {k}")


def test_noalloc_refuses_sizes_beyond_the_static_scratch():
    """Refused on the host before any CUDA call (runs without a GPU too)."""
    lib = _lib()
    p, n = 8, SCRATCH_ELEMS // 8 + 1
    base = 0x7F0000000000
    send = (ctypes.c_void_p * p)(*[base + r * (1 << 26) for r in range(p)])
    recv = (ctypes.c_void_p * p)(*[base + (1 << 32) + r * (1 << 26) for r in range(p)])
    fn = lib.LIB.ccl_ring_reduce_scatter_literal_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                   ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                   ctypes.c_void_p]
    st = fn(send, recv, p, n, lib.CCL_F32, lib.CCL_SUM, None, None)
    assert st == lib.CCL_ERR_INVALID_ARG
    assert "static scratch" in lib.ccl_last_error()
