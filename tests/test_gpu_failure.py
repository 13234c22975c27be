"""Failure detection without a GPU fault: a device-side wait that runs out.

A one-thread kernel waits on an mbarrier that nothing will ever complete; its
bounded wait gives up, records the device error word and returns (the same
path the bulk-copy fan-out takes).  The host learns of it from
ccl_stream_check, which returns CCL_ERR_TIMEOUT, and the context stays
usable: the next collective still matches the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import ccl, to_dev, to_host
from oracle import ring

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def test_clean_work_checks_ok(lib):
    lib.ccl_stream_check()  # clears anything left from earlier tests
    x = [torch.ones(1000, device="cuda") for _ in range(4)]
    lib.ccl_allreduce(x, [torch.empty_like(t) for t in x])
    lib.ccl_stream_check()
    assert lib.ccl_device_error_flag() == 0


def test_wait_that_runs_out_is_reported_and_the_context_survives(lib):
    lib.ccl_stream_check()
    lib.ccl_selftest_bounded_wait()
    with pytest.raises(lib.CclError) as err:
        lib.ccl_stream_check()
    assert err.value.status == lib.CCL_ERR_TIMEOUT
    assert "bounded device-side wait" in lib.ccl_last_error()
    # the word was cleared by the check, and collectives still work
    assert lib.ccl_device_error_flag() == 0
    p, n = 5, 10_007
    x = workloads.normal(p, n, 1.0, 3)
    recv = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_allreduce([to_dev(v, "f32") for v in x], recv)
    want, _, _ = ring.ring_allreduce(x)
    for r in range(p):
        np.testing.assert_array_equal(to_host(recv[r]), want[r])
    lib.ccl_stream_check()
