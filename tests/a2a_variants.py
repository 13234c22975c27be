"""The all-to-all kernel's variants and the GPU cases that reach each one.

``ccl_all_to_all_plan`` / ``ccl_all_to_allv_plan`` name the kernel a call
launches: where its block bounds come from (the 4 KB parameter block at
p <= 16, the chunk rule, or a row-prefix table), whether some block is off
its destination's 16-byte phase (shift), whether straddling units go
through the small-block stage (stage), and the destination tile (4, 8, 16
or 32 KB, by the launch's destination bytes per SM).  Each combination is a separate kernel instantiation (or, for the
unshifted kernel, a different tile loop), so each needs a GPU parity case.
``CASES`` lists them; ``tests/test_a2a_plan.py`` checks on the CPU that
every combination the plan reaches has a case here, and
``tests/test_gpu_a2a_variants.py`` runs them on the GPU, asserting first
that the device's plan picks the expected one.

Buffers sit ``GUARD + offset`` elements into their allocations (256-byte
aligned), so a case's plan depends only on its sizes and offsets.  The
64-bit row-prefix form needs a source of 2^32 rows or more (8 GB and up);
its one case is ``test_all_to_allv_row_prefixes_past_32_bits`` in
``tests/test_gpu_large.py``.
"""
from __future__ import annotations

GUARD = 64  # elements of guard band before each buffer (as gpu_util.GUARD)

# (kind, dtype, p, n per rank (plain) or row elements (v), counts drawn from
# [0, hi) (v), seed, send offset, recv offset (elements),
#  expected (form, shift, stage, tile bytes) on a 152-SM device)
CASES = [
('plain', 'f32', 128, 2048, None, 100, 0, 0, ('plain', False, False, 8192)),
    ('plain', 'f32', 32, 524288, None, 126, 0, 0, ('plain', False, False, 32768)),
    ('plain', 'bf16', 100, 10000, None, 101, 0, 0, ('plain', True, True, 8192)),
    ('plain', 'bf16', 128, 4096, None, 102, 1, 1, ('plain', False, True, 8192)),
    ('plain', 'f32', 100, 10000, None, 103, 1, 1, ('plain', False, True, 16384)),
    ('plain', 'i32', 128, 2048, None, 104, 1, 0, ('plain', True, False, 8192)),
    ('plain', 'i32', 128, 4096, None, 105, 1, 0, ('plain', True, False, 8192)),
    ('plain', 'f32', 17, 65536, None, 106, 0, 0, ('plain', True, False, 16384)),
    ('plain', 'f32', 17, 7, None, 107, 0, 0, ('plain', True, True, 4096)),
    ('plain', 'bf16', 40, 65536, None, 108, 0, 0, ('plain', True, True, 16384)),
    ('plain', 'f32', 40, 65536, None, 109, 0, 0, ('plain', True, True, 32768)),
    ('plain', 'bf16', 2, 1000, None, 110, 0, 0, ('small', True, True, 4096)),
    ('plain', 'f32', 2, 1024, None, 111, 0, 0, ('small', False, False, 4096)),
    ('plain', 'f32', 2, 1048576, None, 112, 0, 0, ('small', False, False, 16384)),
    ('plain', 'f32', 2, 1000, None, 113, 1, 1, ('small', False, True, 4096)),
    ('plain', 'i32', 2, 100003, None, 114, 0, 0, ('small', True, False, 8192)),
    ('plain', 'bf16', 2, 1048576, None, 115, 0, 1, ('small', True, False, 16384)),
    ('plain', 'f32', 2, 7, None, 116, 0, 0, ('small', True, True, 4096)),
    ('v', 'f32', 17, 8, 2, 117, 0, 0, ('table32', False, False, 4096)),
    ('v', 'bf16', 17, 8, 3000, 118, 0, 0, ('table32', False, False, 16384)),
    ('v', 'f32', 17, 8, 2, 119, 1, 1, ('table32', False, True, 4096)),
    ('v', 'f32', 72, 8, 40, 120, 1, 1, ('table32', False, True, 8192)),
    ('v', 'bf16', 17, 4096, 2, 121, 0, 1, ('table32', True, True, 8192)),
    ('v', 'f32', 17, 8, 2, 122, 1, 0, ('table32', True, False, 4096)),
    ('v', 'f32', 17, 1, 100000, 123, 0, 0, ('table32', True, False, 32768)),
    ('v', 'bf16', 17, 1, 2, 124, 0, 0, ('table32', True, True, 4096)),
    ('v', 'f32', 24, 1, 3000, 125, 0, 0, ('table32', True, True, 8192)),
    ('plain', 'f32', 100, 10000, None, 127, 0, 0, ('plain', False, False, 16384)),
    ('plain', 'bf16', 128, 65536, None, 127, 1, 1, ('plain', False, True, 32768)),
    ('plain', 'f32', 24, 131072, None, 127, 0, 0, ('plain', True, False, 32768)),
    ('v', 'bf16', 16, 8, 400, 127, 0, 0, ('small', False, False, 8192)),
    ('v', 'bf16', 8, 4096, 40, 127, 0, 0, ('small', False, False, 32768)),
    ('v', 'bf16', 16, 8, 400, 127, 1, 1, ('small', False, True, 8192)),
    ('v', 'bf16', 2, 8, 2, 127, 1, 0, ('small', True, False, 4096)),
    ('v', 'bf16', 8, 4096, 40, 127, 1, 0, ('small', True, False, 32768)),
    ('v', 'bf16', 16, 1, 3000, 127, 0, 0, ('small', True, True, 8192)),
    ('v', 'bf16', 17, 8, 400, 127, 0, 0, ('table32', False, False, 8192)),
    ('v', 'f32', 40, 8, 400, 127, 0, 0, ('table32', False, False, 32768)),
    ('v', 'bf16', 40, 64, 40, 127, 1, 1, ('table32', False, True, 16384)),
    ('v', 'f32', 40, 8, 400, 127, 1, 1, ('table32', False, True, 32768)),
    ('v', 'bf16', 17, 8, 400, 127, 1, 0, ('table32', True, False, 8192)),
    ('v', 'bf16', 40, 64, 40, 127, 1, 0, ('table32', True, False, 16384)),
    ('v', 'bf16', 40, 64, 40, 127, 0, 1, ('table32', True, True, 16384)),
    ('v', 'f32', 40, 8, 400, 127, 0, 1, ('table32', True, True, 32768)),
]

ELEM_BYTES = {"f32": 4, "bf16": 2, "i32": 4}


def counts_of(case):
    """The p x p row counts of an all-to-allv case."""
    import numpy as np

    kind, _, p, _, hi, seed, _, _, _ = case
    assert kind == "v"
    return np.random.default_rng(seed).integers(0, hi, (p, p))


def case_id(case) -> str:
    kind, dt, p, size, hi, _, so, ro, plan = case
    what = f"n{size}" if kind == "plain" else f"row{size}-hi{hi}"
    return f"{kind}-{dt}-p{p}-{what}-off{so}{ro}-{plan[0]}{'-shift' if plan[1] else ''}{'-stage' if plan[2] else ''}-t{plan[3]}"
