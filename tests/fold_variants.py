"""The fused fold kernel's variants and the GPU cases that reach each one.

``ccl_fold_plan`` names the kernel a sum of p ranks x n elements takes: the
small-p kernel with (ranks per load batch, vectors per thread), (0, 0) for
the general kernel, or (-1, 0) for the kernel of small chunks at p > 16.  Each variant is a separate instantiation per call kind
(all-reduce, reduce-scatter, reduce to the root, DDP bucket), so each
(kind, dtype, variant) needs a GPU parity case at a size that selects it.
``CASES`` lists them; ``tests/test_fold_plan.py`` checks on the CPU that
every variant the plan can pick has a case here, and
``tests/test_gpu_fold_variants.py`` runs them on the GPU, asserting first that
the device's plan picks the expected variant.

The sizes that select the wide variants (many vectors per thread) are the
smallest round ones that still give at least 8 CTAs per SM on a device of up
to 160 SMs, and those that select one vector per thread keep its grid within
one wave (4 CTAs per SM) on a device of 132 SMs, as do the kernel of small
chunks' cases with chunks of 500 - 700 elements; every n leaves p not
dividing n, so chunk edges are ragged.
"""
from __future__ import annotations

KINDS = ("allreduce", "reduce_scatter", "reduce", "bucket")
M = 1 << 20

# (p, n, expected (batch, vectors) of the all-reduce, of the reduce-scatter
# and of the reduce to the root) per dtype: the reduce-scatter and the
# reduce read and write the same bytes and share their plan.
_SUM_CASES = {
    "f32": [(1, 12 * M, (2, 2), (2, 8)), (2, 12 * M + 3, (2, 2), (2, 8)), (3, 6 * M + 1, (4, 2), (4, 2)),
            (4, 6 * M + 2, (4, 1), (4, 2)), (2, 100_003, (2, 1), (2, 2)), (1, 4099, (2, 1), (2, 2)),
            (3, 300_007, (4, 1), (4, 1)), (4, 65_537, (4, 1), (4, 1)), (5, 200_003, (8, 1), (8, 1)),
            (8, 1_000_003, (8, 1), (8, 1)), (9, 100_003, (0, 0), (0, 0)), (16, 50_021, (0, 0), (0, 0)),
            (72, 1_000, (-1, 0), (-1, 0)), (17, 1_999, (-1, 0), (-1, 0)), (72, 14_405, (-1, 0), (-1, 0)),
            (72, 50_413, (-1, 0), (-1, 0))],
    "i32": [(2, 12 * M + 1, (2, 2), (2, 8)), (3, 6 * M + 2, (4, 2), (4, 2)), (4, 6 * M + 1, (4, 1), (4, 2)),
            (2, 100_001, (2, 1), (2, 2)), (4, 65_539, (4, 1), (4, 1)), (7, 200_005, (8, 1), (8, 1)),
            (12, 40_009, (0, 0), (0, 0)), (100, 3_999, (-1, 0), (-1, 0)), (48, 33_605, (-1, 0), (-1, 0))],
    "bf16": [(1, 12 * M + 6, (2, 2), (2, 2)), (2, 12 * M + 1, (2, 2), (2, 2)), (3, 6 * M + 1, (4, 2), (4, 2)),
             (4, 6 * M + 3, (4, 1), (4, 2)), (2, 100_003, (2, 1), (2, 2)), (3, 300_001, (4, 1), (4, 1)),
             (6, 200_003, (8, 1), (8, 1)), (8, 500_009, (8, 1), (8, 1)), (9, 100_003, (0, 0), (0, 0)),
             (16, 50_021, (0, 0), (0, 0)), (72, 1_001, (-1, 0), (-1, 0)), (33, 3_999, (-1, 0), (-1, 0)),
             (128, 32_767, (-1, 0), (-1, 0)), (128, 64_077, (-1, 0), (-1, 0))],
}
_BUCKET_CASES = [(1, 12 * M, (2, 4)), (2, 12 * M + 1, (2, 4)), (3, 6 * M + 2, (4, 2)), (4, 6 * M + 3, (4, 2)),
                 (2, 100_003, (2, 2)), (4, 65_539, (4, 1)), (5, 200_003, (0, 0)), (8, 300_007, (0, 0)),
                 (72, 1_003, (-1, 0)), (72, 43_231, (-1, 0))]

CASES = [(kind, dt, p, n, ar if kind == "allreduce" else rs) for kind in ("allreduce", "reduce_scatter", "reduce")
         for dt, rows in _SUM_CASES.items() for (p, n, ar, rs) in rows]
CASES += [("bucket", "f32", p, n, plan) for (p, n, plan) in _BUCKET_CASES]
# cases sharing inputs run back to back (the GPU test caches one oracle result)
CASES.sort(key=lambda c: (c[0] == "bucket", c[1], c[2], c[3], KINDS.index(c[0])))


def case_id(case) -> str:
    kind, dt, p, n, plan = case
    return f"{kind}-{dt}-p{p}-n{n}-b{plan[0]}u{plan[1]}"
