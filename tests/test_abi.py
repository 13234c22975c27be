"""The C ABI without a GPU: build, load, exported symbols, host-side checks.

No call here reaches a kernel launch: every argument set is rejected on the
host (or is a no-op), which is exactly what the ABI promises to do before any
CUDA call.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import ring


@pytest.fixture(scope="module")
def lib():
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl

    return ccl


def declared_functions() -> list[str]:
    text = open(os.path.join(ROOT, "include", "ccl.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ccl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["ccl_allreduce", "ccl_reduce_scatter", "ccl_all_gather", "ccl_all_to_allv",
                 "ccl_bucket_allreduce_scale_cast", "ccl_ring_allreduce_literal",
                 "ccl_ring_reduce_scatter_literal", "ccl_ring_all_gather_literal",
                 "ccl_chunk_bounds", "ccl_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ccl.h but not exported"


def test_binding_names_match_the_c_abi(lib):
    for name in declared_functions():
        assert callable(getattr(lib, name)), f"binding lacks {name}"


def test_abi_version_and_status_strings(lib):
    assert lib.ccl_abi_version() == 1
    for st in range(5):  # OK, INVALID_ARG, UNSUPPORTED, CUDA, TIMEOUT
        assert lib.ccl_status_string(st).startswith("CCL_")
    assert "unknown" in lib.ccl_status_string(99)


@pytest.mark.parametrize("p", [1, 2, 3, 4, 7, 8, 16, 72, 128])
@pytest.mark.parametrize("n", [0, 1, 5, 13, 1000, 6553600, 100663296])
def test_chunk_bounds_match_the_oracle(lib, p, n):
    expect = ring.chunk_bounds(p, n)
    for c in range(p):
        assert lib.ccl_chunk_bounds(p, n, c) == expect[c]


def test_chunk_bounds_rejects_bad_arguments(lib):
    for p, c in [(0, 0), (129, 0), (4, 4), (4, -1)]:
        with pytest.raises(lib.CclError) as e:
            lib.ccl_chunk_bounds(p, 10, c)
        assert e.value.status == lib.CCL_ERR_INVALID_ARG


# ------------------------------------------------ host-side rejection paths
def lib_ptr_array(vals):
    a = (ctypes.c_void_p * max(1, len(vals)))()
    for i, v in enumerate(vals):
        a[i] = v
    return a


BASE = 0x7F0000000000  # fake device addresses: never dereferenced by a rejected call


def _call_ar(lib, send, recv, p, n, dt=0, op=0):
    return lib.LIB.ccl_allreduce(lib_ptr_array(send), lib_ptr_array(recv), p, n, dt, op, None)


def test_allreduce_rejects_bad_p_dtype_op(lib):
    s = [BASE + i * 4096 for i in range(4)]
    r = [BASE + 65536 + i * 4096 for i in range(4)]
    assert _call_ar(lib, s, r, 0, 16) == lib.CCL_ERR_INVALID_ARG
    assert _call_ar(lib, s, r, 129, 16) == lib.CCL_ERR_INVALID_ARG
    assert _call_ar(lib, s, r, 4, 16, dt=7) == lib.CCL_ERR_INVALID_ARG
    assert _call_ar(lib, s, r, 4, 16, op=9) == lib.CCL_ERR_INVALID_ARG
    assert lib.LIB.ccl_allreduce(None, lib_ptr_array(r), 4, 16, 0, 0, None) == lib.CCL_ERR_INVALID_ARG
    assert "NULL" in lib.ccl_last_error()


def test_allreduce_rejects_null_and_misaligned_pointers(lib):
    s = [BASE + i * 4096 for i in range(4)]
    r = [BASE + 65536 + i * 4096 for i in range(4)]
    assert _call_ar(lib, [s[0], 0, s[2], s[3]], r, 4, 16) == lib.CCL_ERR_INVALID_ARG
    assert _call_ar(lib, s, [r[0] + 2, r[1], r[2], r[3]], 4, 16) == lib.CCL_ERR_INVALID_ARG  # f32 at +2
    assert "aligned" in lib.ccl_last_error()


def test_allreduce_rejects_overlaps_but_not_exact_in_place(lib):
    s = [BASE + i * 4096 for i in range(4)]
    r = [BASE + 65536 + i * 4096 for i in range(4)]
    # two outputs overlapping
    assert _call_ar(lib, s, [r[0], r[0] + 8, r[2], r[3]], 4, 16) == lib.CCL_ERR_INVALID_ARG
    # an output overlapping another rank's input
    assert _call_ar(lib, s, [s[1], r[1], r[2], r[3]], 4, 16) == lib.CCL_ERR_INVALID_ARG
    # an output partially overlapping its own input
    assert _call_ar(lib, s, [s[0] + 16, r[1], r[2], r[3]], 4, 16) == lib.CCL_ERR_INVALID_ARG
    assert "overlap" in lib.ccl_last_error()


def test_zero_length_calls_are_noops(lib):
    s = [BASE + i * 4096 for i in range(4)]
    r = [BASE + 65536 + i * 4096 for i in range(4)]
    assert _call_ar(lib, s, r, 4, 0) == lib.CCL_OK
    assert _call_ar(lib, [0] * 4, [0] * 4, 4, 0) == lib.CCL_OK
    assert lib.LIB.ccl_reduce_scatter(lib_ptr_array(s), lib_ptr_array(r), 4, 0, 0, 0, None) == 0
    assert lib.LIB.ccl_all_gather(lib_ptr_array(s), lib_ptr_array(r), 4, 0, 1, None) == 0
    assert lib.LIB.ccl_bucket_allreduce_scale_cast(lib_ptr_array(s), lib_ptr_array(r), 4, 0,
                                                   0.25, None) == 0
    counts = (ctypes.c_size_t * 16)()
    assert lib.LIB.ccl_all_to_allv(lib_ptr_array(s), counts, lib_ptr_array(r), 4, 8, 1, None) == 0
    sent = (ctypes.c_uint64 * 4)(7, 7, 7, 7)
    assert lib.LIB.ccl_ring_allreduce_literal(lib_ptr_array(s), lib_ptr_array(r), 4, 0, 0, 0,
                                              sent, None, 0, None) == 0
    assert list(sent) == [0, 0, 0, 0]


def test_reduce_scatter_in_place_rule(lib):
    p, n, e = 4, 10, 4  # chunks 3, 3, 2, 2 at offsets 0, 3, 6, 8
    s = [BASE + i * 4096 for i in range(p)]
    offs = [o for o, _ in ring.chunk_bounds(p, n)]
    good = [s[k] + offs[k] * e for k in range(p)]
    bad = list(good)
    bad[2] = s[2]  # overlaps send[2] but not at off(2)
    st = lib.LIB.ccl_reduce_scatter(lib_ptr_array(s), lib_ptr_array(bad), p, n, 0, 0, None)
    assert st == lib.CCL_ERR_INVALID_ARG
    # a shard of length 0 may be NULL, a non-empty one may not
    p2, n2 = 5, 3
    s2 = [BASE + i * 4096 for i in range(p2)]
    r2 = [BASE + 65536 + i * 4096 for i in range(p2)]
    r2[1] = 0
    assert lib.LIB.ccl_reduce_scatter(lib_ptr_array(s2), lib_ptr_array(r2), p2, n2, 0, 0,
                                      None) == lib.CCL_ERR_INVALID_ARG


def test_bucket_rejects_in_place_and_bad_alignment(lib):
    p, n = 8, 64
    g = [BASE + i * 4096 for i in range(p)]
    o = [BASE + 65536 + i * 4096 for i in range(p)]
    assert lib.LIB.ccl_bucket_allreduce_scale_cast(lib_ptr_array(g), lib_ptr_array(g), p, n,
                                                   0.125, None) == lib.CCL_ERR_INVALID_ARG
    o_bad = list(o)
    o_bad[3] += 1  # bf16 output at an odd address
    assert lib.LIB.ccl_bucket_allreduce_scale_cast(lib_ptr_array(g), lib_ptr_array(o_bad), p, n,
                                                   0.125, None) == lib.CCL_ERR_INVALID_ARG


def test_all_to_allv_rejects_overlapping_receivers(lib):
    p, row = 2, 4
    counts = (ctypes.c_size_t * 4)(1, 1, 1, 1)
    s = [BASE, BASE + 4096]
    r = [BASE + 65536, BASE + 65536 + 8]  # each receives 2 rows of 16 bytes: overlap
    assert lib.LIB.ccl_all_to_allv(lib_ptr_array(s), counts, lib_ptr_array(r), p, row, 0,
                                   None) == lib.CCL_ERR_INVALID_ARG


def test_all_to_all_checks(lib):
    p = 4
    s = [BASE + i * 4096 for i in range(p)]
    r = [BASE + 65536 + i * 4096 for i in range(p)]
    assert lib.LIB.ccl_all_to_all(lib_ptr_array(s), lib_ptr_array(r), p, 0, 0, None) == lib.CCL_OK
    assert lib.LIB.ccl_all_to_all(lib_ptr_array(s), lib_ptr_array(r), 0, 8, 0, None) == lib.CCL_ERR_INVALID_ARG
    # each destination receives 4 blocks of 4 f32 (64 bytes): 32 bytes apart overlaps
    r_bad = [BASE + 65536 + i * 32 for i in range(p)]
    assert lib.LIB.ccl_all_to_all(lib_ptr_array(s), lib_ptr_array(r_bad), p, 16, 0,
                                  None) == lib.CCL_ERR_INVALID_ARG


def test_literal_workspace_sizes_and_checks(lib):
    ws = lib.LIB.ccl_ring_literal_workspace_bytes
    assert ws(lib.CCL_KIND_ALLREDUCE, 4, 100, lib.CCL_F32) == 0
    assert ws(lib.CCL_KIND_ALLREDUCE, 4, 100, lib.CCL_BF16) == 4 * 100 * 4
    assert ws(lib.CCL_KIND_REDUCE_SCATTER, 4, 100, lib.CCL_I32) == 4 * 100 * 4
    assert ws(lib.CCL_KIND_ALL_GATHER, 4, 100, lib.CCL_BF16) == 0
    assert ws(lib.CCL_KIND_ALLREDUCE, 0, 100, lib.CCL_BF16) == 0
    p, n = 4, 100
    s = [BASE + i * 4096 for i in range(p)]
    r = [BASE + 65536 + i * 4096 for i in range(p)]
    sent = (ctypes.c_uint64 * p)()
    # bf16 needs a workspace: NULL and too small are rejected
    st = lib.LIB.ccl_ring_allreduce_literal(lib_ptr_array(s), lib_ptr_array(r), p, n, 1, 0, sent,
                                            None, 0, None)
    assert st == lib.CCL_ERR_INVALID_ARG
    st = lib.LIB.ccl_ring_allreduce_literal(lib_ptr_array(s), lib_ptr_array(r), p, n, 1, 0, sent,
                                            BASE + 2**20, 100, None)
    assert st == lib.CCL_ERR_INVALID_ARG
    # workspace overlapping an input
    st = lib.LIB.ccl_ring_allreduce_literal(lib_ptr_array(s), lib_ptr_array(r), p, n, 1, 0, sent,
                                            s[0], p * n * 4, None)
    assert st == lib.CCL_ERR_INVALID_ARG


def test_importing_binding_without_library_fails_loudly(tmp_path):
    """The product path has no fallback: a missing library is an ImportError."""
    import subprocess
    import sys

    code = f"import sys; sys.path.insert(0, {ROOT!r}); import a2a_ring_ordered_gb300.ccl"
    env = dict(os.environ, CCL_LIBRARY=str(tmp_path / "missing" / "libccl.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    assert r.returncode != 0 and "ImportError" in r.stderr and "no fallback" in r.stderr
