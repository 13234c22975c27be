"""bench.py's host logic on CPU: the replica aggregation over ranks (gloo,
world size 2), the reference arm's rank handling, and the clock summary."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each replica timed its own steps; the job takes the slowest
        t = bench.max_over_ranks(1.0 + rank * 0.5, world)
        bench.barrier(world)
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 1.5, 1: 1.5}


def test_reference_arm_other_ranks_exit_without_work():
    class A:
        steps, warmup = 5, 3
    assert bench.run_reference(A(), bench.Bucket(), rank=1, world=2) is None


def test_reference_arm_prints_one_line_on_rank0():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["unit"] == "GB/s" and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] >= 1
    assert out["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_nonzero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_parses_samples():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.source = "test"
    s.samples = [(10.0, ["1900", "2070", "800.5", "Not Active", "Not Active", "Not Active", "Active"]),
                 (10.2, ["1950", "2070", "810.0", "Not Active", "Not Active", "Not Active", "Not Active"]),
                 (99.0, ["300", "2070", "90", "Not Active", "Not Active", "Not Active", "Not Active"])]
    out = s.summary(9.9, 10.3)
    assert out["sm_mhz"] == 1925 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2
    # a region shorter than two periods: bracketed by the samples around it
    short = s.summary(50.0, 50.01)
    assert short["samples"] == 2 and short["sm_mhz"] == (1950 + 300) / 2
    assert "before" in short["note"]


def test_nvml_sample_decodes_clocks_power_and_reasons():
    """The NVML poller (query calls only) against a fake library: SM clock,
    power in W and the clock-event reason bits it reports."""
    import ctypes

    class Fake:
        def nvmlDeviceGetClockInfo(self, h, kind, out):
            ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = 1965 if kind == 1 else 0
            return 0

        def nvmlDeviceGetPowerUsage(self, h, out):
            ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = 812_500
            return 0

        def reasons(self, h, out):
            ctypes.cast(out, ctypes.POINTER(ctypes.c_ulonglong))[0] = 0x4 | 0x40
            return 0

    n = bench._Nvml.__new__(bench._Nvml)
    n.ct, n.lib, n.h, n.max_mhz = ctypes, Fake(), ctypes.c_void_p(), 2070.0
    n.reasons_fn = n.lib.reasons
    smp = n.sample()
    assert smp[:3] == ["1965", "2070.0", "812.50"]
    assert smp[3:] == ["Not Active", "Active", "Not Active", "Active"]  # hw, hw_thermal, sw_thermal, sw_power


def test_warmup_below_three_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--impl", "reference"])


def test_cpu_rank_sample_times_the_same_workload():
    """The CPU-rank ring baseline covers the same bytes as the oracle sample."""
    wl = bench.Bucket()
    wl.x = wl.host_inputs()
    dt, nb, desc, threads = wl.cpu_ranks_sample(0.01)
    dt1, nb1, _ = wl.oracle_sample(0.01)
    assert nb == nb1 and dt > 0 and dt1 > 0
    assert 1 <= threads <= wl.p and f"{threads} threads" in desc


@pytest.mark.parametrize("kind", ["allreduce", "reduce_scatter", "all_gather", "all_to_all"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_oracle_check_leg_accepts_the_oracle_and_catches_one_wrong_element(kind, dt):
    """The bench's sampled check (host logic, CPU tensors): outputs written by
    the oracle pass; one element changed at a chunk edge is caught."""
    import torch

    from a2a_ring_ordered_gb300 import ccl as lib
    from a2a_ring_ordered_gb300 import workloads
    from oracle import collectives, ring

    p, n = 5, 1003
    x = workloads.normal(p, n, 1.0, seed=7, dtype=dt)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if dt == "bf16" else torch.from_numpy(a)
    bounds = ring.chunk_bounds(p, n)
    if kind == "all_gather":
        snd = [x[k][off:off + ln] for k, (off, ln) in enumerate(bounds)]
        rcv = collectives.all_gather(snd)
    elif kind == "all_to_all":
        snd, rcv = x, collectives.all_to_all(x)
    elif kind == "allreduce":
        snd, rcv = x, ring.ring_allreduce(x, dt, "sum")[0]
    else:
        snd, rcv = x, ring.ring_reduce_scatter(x, dt, "sum")[0]
    snd_t = [t(np.ascontiguousarray(v)) for v in snd]
    rcv_t = [t(np.ascontiguousarray(v).copy()) for v in rcv]
    ok = bench.oracle_check_leg(lib, kind, dt, p, n, snd_t, rcv_t, count=64)
    assert ok["checked"] and ok["mismatches"] == 0 and ok["samples"] > 64
    # corrupt one sampled element: a chunk edge of rank 0's output (rank 0's
    # shard start for the reduce-scatter)
    pos = 0 if kind in ("reduce_scatter", "all_to_all") else bounds[1][0]
    v = rcv_t[0].view(torch.int16) if dt == "bf16" else rcv_t[0].view(torch.int32)
    v[pos] ^= 1
    bad = bench.oracle_check_leg(lib, kind, dt, p, n, snd_t, rcv_t, count=64)
    assert not bad["checked"] and bad["mismatches"] == 1
