"""Every all-to-all kernel variant against the oracle.

For each (form, shift, stage, tile) that ``ccl_all_to_all_plan`` /
``ccl_all_to_allv_plan`` can pick, one case asserts that the device's plan
picks it for these buffers, runs the call and compares every received
element with the oracle's block transpose ("Networks and Collective
Communication" section 4.1; the all-to-allv of section 7.4), bit-exact,
with guard bands around every output.
"""
from __future__ import annotations

import numpy as np
import pytest

import a2a_variants as av
from a2a_ring_ordered_gb300 import workloads
from gpu_util import Guarded, assert_equal, ccl, to_dev, to_host
from oracle import collectives

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _values(dt, m, seed):
    if dt == "i32":
        return workloads.integer_valued(1, m, seed, lo=-2**31, hi=2**31 - 1, dtype="i32")[0]
    return workloads.normal(1, m, 1.0, seed, dtype=dt)[0]


def _placed(v, dt, off):
    """A Guarded buffer holding v, GUARD + off elements into its storage."""
    g = Guarded(len(v), dt, offset=av.GUARD + off)
    if len(v):
        g.view.copy_(to_dev(np.ascontiguousarray(v), dt))
    return g


@pytest.mark.parametrize("case", av.CASES, ids=av.case_id)
def test_all_to_all_variant_matches_oracle(lib, case):
    kind, dt, p, size, _, seed, so, ro, plan = case
    if kind == "plain":
        n = size
        x = [_values(dt, n, seed + r) for r in range(p)]
        want = collectives.all_to_all(x)
        send = [_placed(v, dt, so) for v in x]
        outs = [Guarded(len(want[j]), dt, offset=av.GUARD + ro) for j in range(p)]
        got = lib.ccl_all_to_all_plan([s.view for s in send], [o.view for o in outs], n, dt)
        assert got[:3] + (got[4],) == plan, "the device's plan moved"
        lib.ccl_all_to_all([s.view for s in send], [o.view for o in outs])
    else:
        row = size
        counts = av.counts_of(case)
        x = [_values(dt, int(counts[s].sum()) * row, seed + s) for s in range(p)]
        want = collectives.all_to_allv(x, counts, row)
        send = [_placed(v, dt, so) for v in x]
        outs = [Guarded(int(counts[:, d].sum()) * row, dt, offset=av.GUARD + ro) for d in range(p)]
        got = lib.ccl_all_to_allv_plan([s.view for s in send], counts, [o.view for o in outs], row, dt)
        assert got[:3] + (got[4],) == plan, "the device's plan moved"
        lib.ccl_all_to_allv([s.view for s in send], counts, [o.view for o in outs], row)
    for j in range(p):
        assert_equal(to_host(outs[j].view), want[j], dt, f"{av.case_id(case)} rank {j}")
        assert outs[j].guards_intact(), f"{av.case_id(case)} rank {j}: guard band overwritten"
