"""Every instantiation of the fused fold kernels against the oracle.

For each call kind (all-reduce, reduce-scatter, reduce to the root, DDP
bucket), dtype and kernel variant of ``ccl_fold_plan`` -- including the wide
small-p variants (2 or 4 ranks with 4 or 8 vectors per thread) that only
sizes of tens of MiB per rank select -- one case asserts that the device's
plan picks the variant, runs the call and compares every element with the
literal ring oracle ("Networks and Collective Communication" section 5.1),
bit-exact (bf16 outputs: the 1-ulp contract, asserted exact), with guard
bands around every output.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import fold_variants
from a2a_ring_ordered_gb300 import workloads
from gpu_util import Guarded, assert_equal, ccl, to_dev, to_host
from oracle import ring

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


@functools.lru_cache(maxsize=4)
def _inputs(dt, p, n, bucket):
    seed = 1000 + 7 * p + (n % 97)
    if bucket:
        return tuple(workloads.normal(p, n, 1e-3, seed, dtype="f32"))
    if dt == "i32":
        return tuple(workloads.integer_valued(p, n, seed, lo=-2**31, hi=2**31 - 1, dtype="i32"))
    return tuple(workloads.uniform(p, n, seed, dtype=dt))


@functools.lru_cache(maxsize=4)
def _want(dt, p, n, bucket):
    x = list(_inputs(dt, p, n, bucket))
    if bucket:
        return ring.bucket_allreduce_scale_cast(x, float(np.float32(1.0 / p)))[0]
    bufs, _, _ = ring.ring_allreduce(x, dt, "sum")
    return bufs[0]


@pytest.mark.parametrize("case", fold_variants.CASES, ids=fold_variants.case_id)
def test_fold_variant_matches_oracle(lib, case):
    kind, dt, p, n, plan = case
    bucket = kind == "bucket"
    assert lib.ccl_fold_plan(p, n, dt, "sum", kind=kind) == plan, "the device's plan moved"
    x = _inputs(dt, p, n, bucket)
    want = _want(dt, p, n, bucket)
    send = [to_dev(v, dt) for v in x]
    out_dt = "bf16" if bucket else dt
    if kind == "reduce_scatter":
        bounds = ring.chunk_bounds(p, n)
        outs = [Guarded(ln, out_dt) for _, ln in bounds]
        lib.ccl_reduce_scatter(send, [o.view for o in outs])
        expect = [want[off:off + ln] for off, ln in bounds]
    elif kind == "reduce":
        root = p - 1
        outs = [Guarded(n, out_dt)]
        lib.ccl_reduce(send, outs[0].view, root=root)
        expect = [want]
    else:
        outs = [Guarded(n, out_dt) for _ in range(p)]
        if bucket:
            lib.ccl_bucket_allreduce_scale_cast(send, [o.view for o in outs], scale=float(np.float32(1.0 / p)))
        else:
            lib.ccl_allreduce(send, [o.view for o in outs])
        expect = [want] * p
    torch.cuda.synchronize()
    for r, (o, w) in enumerate(zip(outs, expect)):
        assert_equal(to_host(o.view), w, out_dt, f"{fold_variants.case_id(case)} output {r}")
        assert o.guards_intact(), f"{fold_variants.case_id(case)} output {r}: guard band overwritten"
    del send, outs
    torch.cuda.empty_cache()
