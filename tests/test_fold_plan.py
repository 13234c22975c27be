"""Host checks of the fused fold kernel's variant choice (``ccl_fold_plan``).

Runs without a GPU (the plan is host code; the SM count is passed in).  The
guard walks the size classes of every (kind, dtype, p) and requires that each
variant the plan can pick has a GPU parity case in ``fold_variants.CASES`` for
that kind and dtype, so a new variant or a moved threshold cannot leave a
kernel instantiation untested.
"""
from __future__ import annotations

import pytest

import fold_variants

SM_COUNTS = (132, 144, 148, 152, 160)


def _lib():
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl

    return ccl


def _sizes():
    out = {0, 1, 2, 3}
    for k in range(1, 32):
        for base in (1 << k, 3 << (k - 1)):
            out.update((base - 1, base, base + 1))
    return sorted(out)


def _reachable(lib, dtype, kind):
    seen = set()
    for p in range(1, 17):
        for n in _sizes():
            for sms in SM_COUNTS:
                seen.add(lib.ccl_fold_plan(p, n, dtype, "sum", kind=kind, sm_count=sms))
    return seen


@pytest.mark.parametrize("kind", fold_variants.KINDS)
def test_every_reachable_fold_variant_has_a_gpu_case(kind):
    lib = _lib()
    dtypes = ("f32",) if kind == "bucket" else ("f32", "bf16", "i32")
    for dt in dtypes:
        reach = _reachable(lib, dt, kind)
        covered = {plan for (k, d, _, _, plan) in fold_variants.CASES if k == kind and d == dt}
        missing = reach - covered
        assert not missing, f"{kind} {dt}: variants {sorted(missing)} have no GPU parity case"


@pytest.mark.parametrize("case", fold_variants.CASES, ids=fold_variants.case_id)
def test_gpu_cases_select_their_variant_on_a_152_sm_device(case):
    kind, dt, p, n, plan = case
    lib = _lib()
    assert lib.ccl_fold_plan(p, n, dt, "sum", kind=kind, sm_count=152) == plan
    assert n % p != 0 or p == 1, "cases keep ragged chunk edges"


def test_max_min_and_unaligned_calls_take_the_general_kernel():
    lib = _lib()
    for dt in ("f32", "bf16", "i32"):
        for p in (1, 2, 4, 8):
            assert lib.ccl_fold_plan(p, 1 << 24, dt, "max", sm_count=152) == (0, 0)
            assert lib.ccl_fold_plan(p, 1 << 24, dt, "min", sm_count=152) == (0, 0)
            assert lib.ccl_fold_plan(p, 1 << 24, dt, "sum", aligned=False, sm_count=152) == (0, 0)


def test_fold_plan_rejects_bad_arguments():
    lib = _lib()
    with pytest.raises(lib.CclError):
        lib.ccl_fold_plan(0, 10)
    with pytest.raises(lib.CclError):
        lib.ccl_fold_plan(129, 10)
    with pytest.raises(lib.CclError):
        lib.ccl_fold_plan(4, 10, "bf16", kind="bucket")
    with pytest.raises(lib.CclError):
        lib.ccl_fold_plan(4, 10, "f32", "max", kind="bucket")
    with pytest.raises(ValueError):
        lib.ccl_fold_plan(4, 10, "f32", kind="gather")


def test_small_chunk_kernel_boundaries():
    """(-1, 0): 17 - 32 ranks while p x (chunk + 1) stays within 2048
    elements; more than 32 ranks for chunks of at most 1536 elements while
    the grid (segments of 4096 // p elements per chunk, x p chunks) holds at
    most 4 CTAs per SM for every two of the vector kernels' 16-rank rounds.
    Any op and alignment."""
    lib = _lib()
    for op in ("sum", "max", "min"):
        for aligned in (True, False):
            plan = lambda p, n, sms=152: lib.ccl_fold_plan(p, n, "f32", op, aligned=aligned, sm_count=sms)
            assert plan(16, 16 * 10) != (-1, 0)                 # 16 ranks: one round already
            assert plan(17, 17 * 119) == (-1, 0)                # 17 x 120 = 2040
            assert plan(17, 17 * 121) != (-1, 0)                # 17 x 122 = 2074
            assert plan(32, 32 * 63) == (-1, 0)                 # 32 x 64 = 2048
            assert plan(32, 32 * 64) != (-1, 0)
            # p = 33 (3 rounds): segments of 124, at most 608 CTAs; the 1536 cap binds first
            assert plan(33, 33 * 1535 + 32) == (-1, 0)          # chunks of 1535 and 1536
            assert plan(33, 33 * 1536) != (-1, 0)               # q + 1 = 1537
            # p = 48 (3 rounds): segments of 85, 12 per chunk (576 CTAs) still in, 13 (624) not
            assert plan(48, 48 * 1019) == (-1, 0)
            assert plan(48, 48 * 1020) != (-1, 0)
            # p = 72 (5 rounds, two waves of 4 CTAs per SM): segments of 56, 16 per chunk (1152 CTAs)
            assert plan(72, 72 * 895) == (-1, 0)
            assert plan(72, 72 * 896) != (-1, 0)
            assert plan(72, 72 * 895, sms=132) != (-1, 0)      # 1056 CTAs at most on 132 SMs
            assert plan(72, 72 * 783, sms=132) == (-1, 0)      # 14 segments, 1008 CTAs
            # p = 128 (8 rounds, four waves): segments of 32, 19 per chunk (2432 CTAs)
            assert plan(128, 128 * 607) == (-1, 0)
            assert plan(128, 128 * 608) != (-1, 0)
    assert lib.ccl_fold_plan(72, 1000, "f32", "sum", kind="bucket", sm_count=152) == (-1, 0)
