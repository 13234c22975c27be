"""The allocation-free reduce-scatter (ccl_ring_reduce_scatter_literal_noalloc).

Some callers of this library cannot allocate device memory -- code inside an
allocator callback, or under a host application that owns all device memory
-- so they cannot provide the workspace the literal reduce-scatter needs.
This entry point uses the library's built-in static scratch instead.  These
tests check two calls in a row against the workspace entry point and against
the oracle's literal ring (shards and per-rank bytes sent), calls whose
working buffers end exactly on the scratch's last byte, and that sizes beyond
the scratch are refused up front.  The file is named to be collected last.
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


def _inputs(dtype, p, n, seed):
    if dtype == "i32":  # the full int32 range: the sums wrap (two's complement)
        return workloads.integer_valued(p, n, seed, lo=-(2**31), hi=2**31 - 1, dtype="i32")
    return workloads.normal(p, n, 1.0, seed=seed, dtype=dtype)


def _shards(lib, send, p, n, fill):
    sizes = [lib.ccl_chunk_bounds(p, n, k)[1] for k in range(p)]
    return [torch.full((s,), fill, dtype=send[0].dtype, device="cuda") for s in sizes]


# (dtype, p, n, seed): the first two near the limit, the last three with
# p*n exactly 8,388,608 (the last rank's working buffer ends on the array's
# final byte)
CASES = [("f32", 8, 1_000_003, 1), ("bf16", 16, 500_001, 2),
         ("f32", 8, 1_048_576, 3), ("bf16", 16, 524_288, 4), ("i32", 4, 2_097_152, 5)]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,p,n,seed", CASES)
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls_in_a_row(dtype, p, n, seed):
    from oracle import ring

    lib = _lib()
    assert p * n <= SCRATCH_ELEMS
    # two calls in a row on different inputs: the second must not see the
    # first one's leftovers in the shared scratch
    for call, s in enumerate((seed, seed + 100)):
        x = _inputs(dtype, p, n, s)
        send = [to_dev(v, dtype) for v in x]
        want = _shards(lib, send, p, n, 0)
        got = _shards(lib, send, p, n, 7)
        sent_want = lib.ccl_ring_reduce_scatter_literal(send, want)
        sent_got = lib.ccl_ring_reduce_scatter_literal_noalloc(send, got)
        torch.cuda.synchronize()
        oracle_shards, oracle_sent = ring.ring_reduce_scatter(x, dtype, "sum")
        assert sent_got == sent_want == [int(b) for b in oracle_sent], f"call {call}: bytes sent"
        for k in range(p):
            h = to_host(got[k])
            assert_equal(h, to_host(want[k]), dtype, f"call {call} {dtype} shard {k} vs workspace")
            assert_equal(h, oracle_shards[k], dtype, f"call {call} {dtype} shard {k} vs oracle")


def _raw_call(lib, p, n, dtype_code):
    base = 0x7F0000000000
    send = (ctypes.c_void_p * p)(*[base + r * (1 << 26) for r in range(p)])
    recv = (ctypes.c_void_p * p)(*[base + (1 << 32) + r * (1 << 26) for r in range(p)])
    fn = lib.LIB.ccl_ring_reduce_scatter_literal_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                   ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                   ctypes.c_void_p]
    return fn(send, recv, p, n, dtype_code, lib.CCL_SUM, None, None)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_noalloc_refuses_sizes_beyond_the_static_scratch(dtype):
    """Refused on the host before any CUDA call (runs without a GPU too).
    The working buffers are fp32 / int32 whatever the dtype (bf16 partials
    travel in fp32), so p*n = limit + 1 is refused for bf16 as well."""
    lib = _lib()
    code = {"f32": lib.CCL_F32, "bf16": lib.CCL_BF16, "i32": lib.CCL_I32}[dtype]
    for p, n in ((8, SCRATCH_ELEMS // 8 + 1), (1, SCRATCH_ELEMS + 1), (3, (SCRATCH_ELEMS + 2) // 3)):
        assert p * n > SCRATCH_ELEMS
        st = _raw_call(lib, p, n, code)
        assert st == lib.CCL_ERR_INVALID_ARG
        assert "static scratch" in lib.ccl_last_error()
