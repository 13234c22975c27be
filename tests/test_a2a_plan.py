"""Host checks of the all-to-all kernel's variant choice (``ccl_all_to_all_plan``,
``ccl_all_to_allv_plan``).

Runs without a GPU: the plan reads buffer addresses only for their 16-byte
phase, and the SM count is passed in.  The guard walks plain and table calls
over p, sizes, row lengths, count ranges and buffer offsets, and requires
that every (form, shift, stage, tile) the plan can pick has a GPU parity
case in ``a2a_variants.CASES``, so a new variant or a moved threshold cannot
leave a kernel instantiation untested.
"""
from __future__ import annotations

import numpy as np
import pytest

import a2a_variants as av


def _lib():
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl

    return ccl


def _addresses(p, off, e, base=0):
    # distinct 1 GiB-aligned allocations, the buffer GUARD + off elements in
    return [(base + i + 1) * (1 << 30) + (av.GUARD + off) * e for i in range(p)]


def _plan(lib, case, sms=152):
    kind, dt, p, size, _, _, so, ro, _ = case
    e = av.ELEM_BYTES[dt]
    send, recv = _addresses(p, so, e), _addresses(p, ro, e, base=256)
    if kind == "plain":
        return lib.ccl_all_to_all_plan(send, recv, size, dt, sm_count=sms)
    return lib.ccl_all_to_allv_plan(send, av.counts_of(case), recv, size, dt, sm_count=sms)


@pytest.mark.parametrize("case", av.CASES, ids=av.case_id)
def test_gpu_cases_select_their_variant_on_a_152_sm_device(case):
    lib = _lib()
    form, shift, stage, launches, tile = _plan(lib, case)
    assert (form, shift, stage, tile) == case[-1]
    assert launches == 1


def _reachable(lib):
    seen = set()
    for dt in ("f32", "bf16"):
        e = av.ELEM_BYTES[dt]
        for p in (2, 3, 5, 8, 16, 17, 24, 40, 72, 100, 128):
            for so, ro in ((0, 0), (0, 1), (1, 0), (1, 1), (0, 8)):
                send, recv = _addresses(p, so, e), _addresses(p, ro, e, base=256)
                for n in (7, 100, 1000, 4096, 10_000, 65_536, 100_003, 1 << 20, 1 << 22, 1 << 24):
                    pl = lib.ccl_all_to_all_plan(send, recv, n, dt, sm_count=152)
                    if pl[3]:
                        seen.add(pl[:3] + (pl[4],))
                rng = np.random.default_rng(p)
                for row in (1, 3, 8, 4096):
                    for hi in (2, 40, 3000, 100_000):
                        if row * hi * p * p > 4e9:
                            continue
                        pl = lib.ccl_all_to_allv_plan(send, rng.integers(0, hi, (p, p)), recv, row, dt,
                                                      sm_count=152)
                        if pl[3]:
                            seen.add(pl[:3] + (pl[4],))
    return seen


def test_every_reachable_all_to_all_variant_has_a_gpu_case():
    lib = _lib()
    reach = _reachable(lib)
    covered = {case[-1] for case in av.CASES}
    missing = reach - covered
    assert not missing, f"variants {sorted(missing)} have no GPU parity case"
    # the p <= 16 form with the stage cannot take 16 or 32 KB tiles: blocks
    # of 8 KB on average fill at most 16 x 16 x 8 KB = 2 MB, 13.5 KiB per SM
    # of a 152-SM device, which takes 4 or 8 KB tiles
    for tile in (16384, 32768):
        assert ("small", False, True, tile) not in reach and ("small", True, True, tile) not in reach


def test_row_prefix_width_follows_the_largest_source():
    lib = _lib()
    p = 2
    send, recv = _addresses(p, 0, 2), _addresses(p, 0, 2, base=256)
    wide = np.array([[(1 << 31) + 5, (1 << 31) + 7], [3, 2]])
    assert lib.ccl_all_to_allv_plan(send, wide, recv, 1, "bf16", sm_count=152)[0] == "table64"
    narrow = np.array([[(1 << 31) - 5, (1 << 31) - 7], [3, 2]])
    assert lib.ccl_all_to_allv_plan(send, narrow, recv, 1, "bf16", sm_count=152)[0] == "small"


def test_launch_counts_of_large_p_tables():
    """The 32 KB parameter block holds p x (destinations + 1) <= 7408 row
    prefixes: one launch up to p = 85, two at p = 86, three at p = 128."""
    lib = _lib()
    for p, want in ((85, 1), (86, 2), (128, 3)):
        send, recv = _addresses(p, 0, 2), _addresses(p, 0, 2, base=256)
        pl = lib.ccl_all_to_allv_plan(send, np.ones((p, p), dtype=np.int64), recv, 8, "bf16", sm_count=152)
        assert pl[3] == want


def test_plan_rejects_bad_arguments():
    lib = _lib()
    with pytest.raises(lib.CclError):
        lib.ccl_all_to_all_plan([], [], 10, "f32", sm_count=152)
    with pytest.raises(lib.CclError):
        lib.ccl_all_to_all_plan([0] * 129, [0] * 129, 10, "f32", sm_count=152)
    with pytest.raises(lib.CclError):
        lib.ccl_all_to_allv_plan([1 << 30] * 2, np.full((2, 2), 1 << 60), [1 << 31] * 2, 1, "f32", sm_count=152)
    assert lib.ccl_all_to_all_plan([1 << 30] * 4, [1 << 31] * 4, 0, "f32", sm_count=152)[3] == 0


def test_stage_follows_the_block_size_and_the_grid():
    """The small-block stage runs only when some block edge or destination
    end is off the 16-byte grid and blocks average 8 KB or less; the shift
    only when some block's source and destination phases differ."""
    lib = _lib()
    p = 8
    s, r = _addresses(p, 0, 4), _addresses(p, 0, 4, base=256)
    plan = lambda counts, recv, row: lib.ccl_all_to_allv_plan(s, counts, recv, row, "f32", sm_count=152)
    # blocks of 400 bytes: every edge on the grid, phases equal: neither
    assert plan(np.full((p, p), 100), r, 1)[1:3] == (False, False)
    # blocks of 404 bytes: edges off the grid (stage), and a block's source
    # rows before it differ from its destination's (shift)
    assert plan(np.full((p, p), 101), r, 1)[1:3] == (True, True)
    # blocks of 8,188 bytes on average still stage, of 8,196 not
    assert plan(np.full((p, p), 2047), r, 1)[2] is True
    assert plan(np.full((p, p), 2049), r, 1)[2] is False
    # receive buffers 4 bytes off the grid, 16-byte rows: stage and shift
    assert plan(np.full((p, p), 4), _addresses(p, 1, 4, base=256), 4)[1:3] == (True, True)
    # the plain all-to-all: n a multiple of 4 p keeps every block on the grid
    assert lib.ccl_all_to_all_plan(s, r, 4 * p * 100, "f32", sm_count=152)[1:3] == (False, False)
    assert lib.ccl_all_to_all_plan(s, r, 4 * p * 100 + 1, "f32", sm_count=152)[1:3] == (True, True)


def test_tile_follows_the_bytes_per_sm():
    """4 KB tiles below 5 KiB of destination bytes per SM, 8 KB below 24 KiB,
    16 KB below 64 KiB, else 32 KB."""
    lib = _lib()
    p = 16
    s, r = _addresses(p, 0, 4), _addresses(p, 0, 4, base=256)
    tile = lambda n, sms=152: lib.ccl_all_to_all_plan(s, r, n, "f32", sm_count=sms)[4]
    kib = lambda b: b * 1024 * 152 // (4 * p)  # n per rank for b KiB per SM at 152 SMs
    assert tile(kib(5) - 1) == 4096 and tile(kib(5)) == 8192
    assert tile(kib(24) - 1) == 8192 and tile(kib(24)) == 16384
    assert tile(kib(64) - 1) == 16384 and tile(kib(64)) == 32768
    assert tile(kib(64), sms=304) == 16384  # the same call on twice the SMs
