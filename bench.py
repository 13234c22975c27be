#!/usr/bin/env python3
"""Benchmark of the ring-ordered collectives on one GB300 (p virtual ranks in HBM).

Default workload: the DDP gradient bucket -- p=8 ranks, one 25 MB fp32 bucket
per rank (6,553,600 gradients ~ N(0, 1e-3), seed 1), all-reduced in ring order
with the 1/8 average and the bf16 cast fused in.  One step = one
``ccl_bucket_allreduce_scale_cast`` call, which runs the reduce-scatter fold,
the all-gather and the all-reduce of that bucket in one kernel.

Metric: effective GB/s = the primitive's minimum HBM bytes per step / the
device time of a step (CUDA events on the launching stream), and the fraction
of the measured HBM copy bandwidth.  After the default line's timed region
it also carries ``configs``: the other configurations of the workload set
(the p=4 fp32 collectives, the ZeRO chain, the MoE all-to-allv, the
all-reduce at 8 MiB / 64 MiB / 1 GiB per rank for p = 2, 16, 72), each timed
and checked against the oracle at sampled positions.  Other workloads
(``--workload``) cover the ZeRO chain, MoE dispatch/combine, plain
all-reduce points, the other fold orders and the literal ring engine;
``--sweep`` runs a message-size sweep of one collective.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload bucket|allreduce|reduce_scatter|all_gather|zero|moe|literal]
                    [--p P] [--mib M] [--dtype f32|bf16] [--sweep]

Under torchrun (N > 1) every rank runs the same single-GPU workload on its
own GPU (replicas, no collective on the data path); rank 0 prints one JSON
line with the job total.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (~129 MB)
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def measured_peak_gbs() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(files: list[str]) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str, files: list[str]) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_digest") != source_digest(files):
        return None
    return float(rec["dram_bytes_per_launch"])


class _Nvml:
    """The few NVML queries the clock record needs, through ctypes (query
    only: nothing here sets a clock, a limit or a mode)."""

    SM_CLOCK = 1  # NVML_CLOCK_SM
    # clocks-event reason bits (nvmlClocksEventReason*)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.h)) != 0:
            raise OSError("nvmlDeviceGetHandleByIndex_v2 failed")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        u = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM_CLOCK, ctypes.byref(u)) != 0:
            raise OSError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(u.value)

    def sample(self) -> list[str]:
        ct = self.ct
        mhz, mw, bits = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok_c = self.lib.nvmlDeviceGetClockInfo(self.h, self.SM_CLOCK, ct.byref(mhz)) == 0
        ok_p = self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) == 0
        ok_r = self.reasons_fn(self.h, ct.byref(bits)) == 0
        act = lambda b: ("Active" if (bits.value & b) else "Not Active") if ok_r else "[N/A]"
        return [str(mhz.value) if ok_c else "[N/A]", str(self.max_mhz),
                f"{mw.value / 1000.0:.2f}" if ok_p else "[N/A]",
                act(0x8), act(0x40), act(0x20), act(0x4)]


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons during the timed
    region: NVML polled every 2 ms from a thread (query only), so even a
    timed region of about a millisecond is bracketed by samples; nvidia-smi
    every 200 ms where NVML cannot be loaded."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_index: int):
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.nvml = None
        self._stop = threading.Event()
        try:
            self.nvml = _Nvml(gpu_index)
            self.source = "NVML, every 2 ms"
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            self.nvml = None
        self.source = "nvidia-smi, every 200 ms"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        while not self._stop.is_set():
            self.samples.append((time.time(), self.nvml.sample()))
            self._stop.wait(self.PERIOD_S)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        self._stop.set()
        if self.nvml is not None:
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = f"samples inside the timed region ({self.source})"
        if len(inside) < 2 and self.samples:  # a region shorter than two periods
            before = [ts for ts in self.samples if ts[0] < t0]
            after = [ts for ts in self.samples if ts[0] > t1]
            inside = ([before[-1][1]] if before else []) + inside + ([after[0][1]] if after else [])
            note = (f"samples inside the timed region plus the last one before and the first one "
                    f"after it ({self.source}; the region is shorter than two periods)")
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no clock source (NVML and nvidia-smi unavailable)"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4)
                          if len(s) > 3 + i and s[3 + i].lower().startswith("active")})

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(s[0]) for s in inside) if v is not None]
        mx = [v for v in (num(s[1]) for s in inside) if v is not None]
        pw = [v for v in (num(s[2]) for s in inside) if v is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ---------------------------------------------------------------- workloads
KERNEL_SOURCES = {
    "fold": ["a2a_ring_ordered_gb300/csrc/fold.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh",
             "a2a_ring_ordered_gb300/csrc/realign.cuh"],
    "schedule": ["a2a_ring_ordered_gb300/csrc/schedule_fold.cu",
                 "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
    "hier": ["a2a_ring_ordered_gb300/csrc/hier_fold.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
    "wire": ["a2a_ring_ordered_gb300/csrc/wire_fold.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh",
             "a2a_ring_ordered_gb300/csrc/realign.cuh"],
    "fanout": ["a2a_ring_ordered_gb300/csrc/bulk_fanout.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
    "gather": ["a2a_ring_ordered_gb300/csrc/gather.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh",
               "a2a_ring_ordered_gb300/csrc/realign.cuh"],
    "a2av": ["a2a_ring_ordered_gb300/csrc/a2av.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh",
             "a2a_ring_ordered_gb300/csrc/realign.cuh"],
    "ring_step": ["a2a_ring_ordered_gb300/csrc/ring_step.cu",
                  "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
    "moe": ["a2a_ring_ordered_gb300/csrc/moe.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
    "ulysses": ["a2a_ring_ordered_gb300/csrc/ulysses.cu", "a2a_ring_ordered_gb300/csrc/device_common.cuh"],
}
for _part in ("moe_route", "moe_dispatch", "moe_combine"):
    KERNEL_SOURCES[_part] = KERNEL_SOURCES["moe"]


def host_prefix(tensors, m: int) -> list[np.ndarray]:
    """First m elements of each device rank buffer as numpy (bf16 as uint16 bits)."""
    import torch
    out = []
    for t in tensors:
        h = t[:m].detach().cpu()
        out.append(h.view(torch.int16).numpy().view(np.uint16).copy() if h.dtype == torch.bfloat16
                   else h.numpy().copy())
    return out


def oracle_prefix_sample(tensors, n: int, frac: float, fn, bytes_per_elem_index: float, what: str):
    """Time ``fn`` (an oracle call) on the first frac*n elements of every rank."""
    p = len(tensors)
    m = max(p, int(n * frac))
    xs = host_prefix(tensors, m)
    t0 = time.perf_counter()
    fn(xs)
    dt = time.perf_counter() - t0
    whose = f"each of the {p} ranks" if p > 1 else "the root's buffer"
    return dt, int(m * bytes_per_elem_index), f"{what} on the first {m} of {n} elements of {whose}"


class Workload:
    """One step of a collective on device-resident synthetic inputs."""
    name = ""
    dtype = "f32"
    kernel = "fold"          # dominant kernel (sources for the traffic digest)
    kernel_key = ""          # key in profiles/traffic.json
    # NCCL's conventions (algbw = a rank's message bytes / time, busbw = algbw
    # x the schedule factor: 2(p-1)/p all-reduce, (p-1)/p reduce-scatter and
    # all-gather), for comparison with published collective numbers
    nccl_bytes_per_rank = 0
    nccl_factor = 0.0
    launches_per_step = 1

    def config(self) -> dict:
        raise NotImplementedError

    def bytes_per_step(self) -> int:
        raise NotImplementedError

    def setup(self, lib, torch, device):
        raise NotImplementedError

    def step(self, stream):
        raise NotImplementedError

    def parts(self):
        """(kernel name, algorithmic bytes, callable(stream)) per launch of a step."""
        return [(self.kernel, self.bytes_per_step(), self.step)]

    def e2e_step(self, stream):
        raise NotImplementedError

    def oracle_sample(self, frac: float):
        raise NotImplementedError

    def cpu_ranks_sample(self, frac: float):
        """The same sample on the CPU-rank ring (one host thread per rank):
        (seconds, algorithmic bytes, description, threads)."""
        raise NotImplementedError


def cpu_ranks_prefix_sample(tensors, n: int, frac: float, kind: str, dtype: str, bytes_per_elem_index: float,
                            what: str, scale: float = 1.0, shards: bool = False):
    """Time the CPU-rank ring on the first frac*n elements of every rank (as
    chunk-rule blocks of that prefix when ``shards``)."""
    from oracle import cpu_ranks, ring
    p = len(tensors)
    m = max(p, int(n * frac))
    xs = host_prefix(tensors, m)
    if shards:
        xs = [xs[k][off:off + ln] for k, (off, ln) in enumerate(ring.chunk_bounds(p, m))]
    t0 = time.perf_counter()
    _, _, st, threads = cpu_ranks.ring(kind, xs, dtype, "sum", scale=scale, timeout_s=600.0)
    dt = time.perf_counter() - t0
    if st != cpu_ranks.OK:
        raise RuntimeError(f"CPU-rank ring returned status {st}")
    return dt, int(m * bytes_per_elem_index), (f"{what} on the first {m} of {n} elements of each of the "
                                               f"{p} ranks, {threads} threads"), threads


class Bucket(Workload):
    name = "ddp_bucket_allreduce_scale_cast"
    kernel = "fold"

    def __init__(self, p=8, n=6_553_600, sigma=1e-3, seed=1):
        self.p, self.n, self.sigma, self.seed = p, n, sigma, seed
        self.scale = float(np.float32(1.0 / p))
        self.kernel_key = f"fold_bucket_f32_bf16_p{p}_n{n}"

    def config(self):
        return {"workload": f"DDP bucket all-reduce + 1/p scale + bf16 cast: p={self.p} ranks x "
                            f"{self.n} fp32 (25 MB bucket per rank) -> bf16",
                "p": self.p, "n_per_rank": self.n, "bucket_mb_per_rank": self.n * 4 / 2**20,
                "inputs": f"N(0, sigma={self.sigma}) seed {self.seed}, numpy PCG64",
                "scale": f"1/{self.p}"}

    def bytes_per_step(self):
        return self.p * self.n * 4 + self.p * self.n * 2

    @property
    def nccl_bytes_per_rank(self):
        return self.n * 4

    @property
    def nccl_factor(self):
        return 2.0 * (self.p - 1) / self.p

    def host_inputs(self):
        from a2a_ring_ordered_gb300 import workloads
        return workloads.normal(self.p, self.n, self.sigma, self.seed)

    def setup(self, lib, torch, device):
        self.lib, self.torch = lib, torch
        self.x = self.host_inputs()
        self.send = [torch.from_numpy(v).to(device) for v in self.x]
        self.recv = [torch.empty(self.n, dtype=torch.bfloat16, device=device) for _ in range(self.p)]
        # pinned host copies for the end-to-end path, and a second device buffer
        # set so that consecutive steps can overlap copy-out with copy-in
        self.h_in = [torch.from_numpy(v).pin_memory() for v in self.x]
        self.h_out = [torch.empty(self.n, dtype=torch.bfloat16).pin_memory() for _ in range(self.p)]
        self.sets = [(self.send, self.recv),
                     ([torch.empty_like(t) for t in self.send], [torch.empty_like(t) for t in self.recv])]
        self.s_h2d, self.s_d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
        self.i_e2e = 0
        self.freed = [None, None]  # per set: event after its last kernel and copy-out

    def step(self, stream):
        self.lib.ccl_bucket_allreduce_scale_cast(self.send, self.recv, scale=self.scale, stream=stream)

    def e2e_step(self, stream):
        """Pinned host inputs to pinned host outputs through the public API:
        H2D copies of the p fp32 gradient buffers (copy-in stream), the kernel
        (the caller's stream), D2H copies of the p bf16 results (copy-out
        stream), one cudaMemcpyAsync per buffer.  Consecutive steps alternate
        between two device buffer sets, so step i's copy-out overlaps step
        i+1's copy-in, as successive DDP buckets do."""
        torch = self.torch
        k = self.i_e2e % 2
        self.i_e2e += 1
        send, recv = self.sets[k]
        if self.freed[k] is not None:
            self.s_h2d.wait_event(self.freed[k])
        with torch.cuda.stream(self.s_h2d):
            for d, h in zip(send, self.h_in):
                d.copy_(h, non_blocking=True)
        stream.wait_stream(self.s_h2d)
        self.lib.ccl_bucket_allreduce_scale_cast(send, recv, scale=self.scale, stream=stream)
        self.s_d2h.wait_stream(stream)
        with torch.cuda.stream(self.s_d2h):
            for h, d in zip(self.h_out, recv):
                h.copy_(d, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(self.s_d2h)
        self.freed[k] = ev

    def e2e_begin(self, stream):
        """Order the copy streams after `stream` (after the timed region's start event)."""
        self.s_h2d.wait_stream(stream)
        self.s_d2h.wait_stream(stream)

    def e2e_finish(self, stream):
        """Make `stream` wait for every outstanding copy of the end-to-end path."""
        stream.wait_stream(self.s_h2d)
        stream.wait_stream(self.s_d2h)

    def e2e_zero_copy_step(self, stream):
        """Same data movement with no staging: the kernel reads the gradients
        from pinned host memory and writes the results there directly."""
        self.lib.ccl_bucket_allreduce_scale_cast(self.h_in, self.h_out, scale=self.scale, stream=stream)

    def e2e_bytes(self):
        return self.p * self.n * 4, self.p * self.n * 2

    def oracle_sample(self, frac):
        from oracle import ring
        m = max(self.p, int(self.n * frac))
        xs = [v[:m] for v in self.x]
        t0 = time.perf_counter()
        ring.bucket_allreduce_scale_cast(xs, self.scale)
        dt = time.perf_counter() - t0
        return dt, self.p * m * 6, f"first {m} of {self.n} elements of each of the {self.p} ranks"

    def cpu_ranks_sample(self, frac):
        from oracle import cpu_ranks
        m = max(self.p, int(self.n * frac))
        xs = [v[:m] for v in self.x]
        t0 = time.perf_counter()
        _, _, st, threads = cpu_ranks.ring("bucket", xs, scale=self.scale, timeout_s=600.0)
        dt = time.perf_counter() - t0
        if st != cpu_ranks.OK:
            raise RuntimeError(f"CPU-rank ring returned status {st}")
        return dt, self.p * m * 6, (f"CPU-rank ring bucket on the first {m} of {self.n} elements of each of "
                                    f"the {self.p} ranks, {threads} threads"), threads


class AllReduce(Workload):
    kernel = "fold"

    def __init__(self, p=16, mib=256, dtype="f32", seed=4, op="sum", literal=False, schedule="ring",
                 group=8, wire="fp32"):
        self.p, self.dtype, self.seed, self.op, self.literal = p, dtype, seed, op, literal
        self.wire = wire
        if wire == "bf16" and (dtype != "bf16" or schedule != "ring" or literal):
            raise SystemExit("--wire bf16 needs --dtype bf16 and the fused ring")
        self.schedule = schedule
        self.group = group if schedule == "hierarchical" else None
        if self.group is not None and (group < 1 or p % group):
            raise SystemExit(f"--group {group} must divide --p {p}")
        self.e = 4 if dtype == "f32" else 2
        self.n = mib * (1 << 20) // self.e
        self.mib = mib
        self.name = "ring_allreduce_literal" if literal else "allreduce"
        self.kernel = ("ring_step" if literal else "fold" if schedule == "ring"
                       else "hier" if schedule == "hierarchical" else "schedule")
        tag = "" if schedule == "ring" else f"_{schedule}" + (f"_g{group}" if self.group else "")
        if wire == "bf16":
            self.kernel, tag = "wire", "_bf16wire"
        self.kernel_key = f"{self.kernel}_ar{tag}_{dtype}_p{p}_n{self.n}"
        # literal engine: set-up move + (p-1) reduce-scatter steps + (bf16: rounding
        # move) + (p-1) all-gather steps
        self.launches_per_step = (2 * p - 1 + (1 if dtype == "bf16" else 0)) if literal else 1

    def config(self):
        kind = "literal ring" if self.literal else f"fused {self.schedule.replace('_', ' ')}"
        if self.group is not None:
            kind += f" ({self.p // self.group} groups of {self.group})"
        if self.wire == "bf16":
            kind += " (bf16 partials on the wire)"
        cfg = {"workload": f"{kind} all-reduce: p={self.p} ranks x {self.mib} MiB {self.dtype} per rank",
               "p": self.p, "n_per_rank": self.n, "inputs": f"U(-1,1) seed {self.seed}"}
        if self.group is not None:
            cfg["group"] = self.group
        return cfg

    def bytes_per_step(self):
        return 2 * self.p * self.n * self.e

    @property
    def nccl_bytes_per_rank(self):
        return self.n * self.e

    @property
    def nccl_factor(self):
        return 2.0 * (self.p - 1) / self.p

    def setup(self, lib, torch, device):
        self.lib, self.torch = lib, torch
        gen = torch.Generator(device=device)
        gen.manual_seed(self.seed)
        tdt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        self.send = [(torch.rand(self.n, generator=gen, device=device) * 2 - 1).to(tdt)
                     for _ in range(self.p)]
        self.recv = [torch.empty_like(s) for s in self.send]
        self.ws = None
        if self.literal:
            need = lib.ccl_ring_literal_workspace_bytes(lib.CCL_KIND_ALLREDUCE, self.p, self.n, tdt)
            self.ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

    def oracle_sample(self, frac):
        from oracle import ring, schedules
        if self.wire == "bf16":
            return oracle_prefix_sample(self.send, self.n, frac,
                                        lambda xs: ring.ring_allreduce(xs, self.dtype, self.op, wire="bf16"),
                                        2 * self.p * self.e, "oracle ring all-reduce, bf16 wire")
        if self.schedule == "hierarchical":
            return oracle_prefix_sample(
                self.send, self.n, frac,
                lambda xs: schedules.hierarchical(xs, self.group, self.dtype, self.op),
                2 * self.p * self.e, f"oracle hierarchical all-reduce, groups of {self.group}")
        if self.schedule != "ring":
            return oracle_prefix_sample(
                self.send, self.n, frac,
                lambda xs: schedules.allreduce(self.schedule, xs, self.dtype, self.op),
                2 * self.p * self.e, f"oracle {self.schedule} all-reduce")
        return oracle_prefix_sample(self.send, self.n, frac,
                                    lambda xs: ring.ring_allreduce(xs, self.dtype, self.op),
                                    2 * self.p * self.e, "oracle ring all-reduce")

    def cpu_ranks_sample(self, frac):
        if self.schedule != "ring" or self.wire != "fp32" or self.op != "sum":
            raise NotImplementedError
        return cpu_ranks_prefix_sample(self.send, self.n, frac, "allreduce", self.dtype, 2 * self.p * self.e,
                                       "CPU-rank ring all-reduce")

    def step(self, stream):
        if self.literal:
            self.lib.ccl_ring_allreduce_literal(self.send, self.recv, op=self.op,
                                                workspace=self.ws, stream=stream)
        elif self.wire == "bf16":
            self.lib.ccl_allreduce_bf16_wire(self.send, self.recv, stream=stream)
        elif self.schedule == "hierarchical":
            self.lib.ccl_allreduce_hierarchical(self.send, self.recv, self.group, op=self.op,
                                                stream=stream)
        elif self.schedule != "ring":
            self.lib.ccl_allreduce_schedule(self.send, self.recv, self.schedule, op=self.op,
                                            stream=stream)
        else:
            self.lib.ccl_allreduce(self.send, self.recv, op=self.op, stream=stream)


class ReduceScatter(AllReduce):
    def __init__(self, p=16, mib=192, dtype="bf16", seed=2, wire="fp32"):
        super().__init__(p, mib, dtype, seed, wire=wire)
        self.name = "reduce_scatter"
        self.kernel_key = (f"wire_rs_{dtype}_p{p}_n{self.n}" if wire == "bf16"
                           else f"fold_rs_{dtype}_p{p}_n{self.n}")

    def config(self):
        c = super().config()
        wire = " (bf16 partials on the wire)" if self.wire == "bf16" else ""
        c["workload"] = f"fused reduce-scatter{wire}: p={self.p} ranks x {self.mib} MiB {self.dtype} per rank"
        return c

    def bytes_per_step(self):
        return self.p * self.n * self.e + self.n * self.e

    @property
    def nccl_factor(self):
        return (self.p - 1) / self.p

    def setup(self, lib, torch, device):
        super().setup(lib, torch, device)
        self.shards = [torch.empty(lib.ccl_chunk_bounds(self.p, self.n, k)[1], dtype=self.send[0].dtype,
                                   device=device) for k in range(self.p)]

    def step(self, stream):
        if self.wire == "bf16":
            self.lib.ccl_reduce_scatter_bf16_wire(self.send, self.shards, stream=stream)
        else:
            self.lib.ccl_reduce_scatter(self.send, self.shards, stream=stream)

    def oracle_sample(self, frac):
        from oracle import ring
        return oracle_prefix_sample(self.send, self.n, frac,
                                    lambda xs: ring.ring_reduce_scatter(xs, self.dtype, "sum", self.wire),
                                    (self.p + 1) * self.e, "oracle ring reduce-scatter")

    def cpu_ranks_sample(self, frac):
        if self.wire != "fp32":
            raise NotImplementedError
        return cpu_ranks_prefix_sample(self.send, self.n, frac, "reduce_scatter", self.dtype,
                                       (self.p + 1) * self.e, "CPU-rank ring reduce-scatter")


class AllGather(ReduceScatter):
    kernel = "gather"

    def __init__(self, p=16, mib=192, dtype="bf16", seed=2):
        super().__init__(p, mib, dtype, seed)
        self.name = "all_gather"
        self.kernel = "gather"  # (the base class set "fold")
        self.kernel_key = f"gather_{dtype}_p{p}_n{self.n}"

    def config(self):
        c = super().config()
        c["workload"] = f"all-gather: p={self.p} ranks, {self.mib} MiB {self.dtype} output per rank"
        return c

    def bytes_per_step(self):
        return self.n * self.e + self.p * self.n * self.e

    def step(self, stream):
        self.lib.ccl_all_gather(self.shards, self.recv, stream=stream)

    def oracle_sample(self, frac):
        from oracle import ring

        def gather(xs):
            m = len(xs[0])
            blocks = [xs[k][off:off + ln] for k, (off, ln) in enumerate(ring.chunk_bounds(self.p, m))]
            ring.ring_all_gather(blocks, self.dtype)
        return oracle_prefix_sample(self.send, self.n, frac, gather, (self.p + 1) * self.e,
                                    "oracle ring all-gather")

    def cpu_ranks_sample(self, frac):
        return cpu_ranks_prefix_sample(self.send, self.n, frac, "all_gather", self.dtype, (self.p + 1) * self.e,
                                       "CPU-rank ring all-gather", shards=True)


class Zero(ReduceScatter):
    """ZeRO chain: reduce-scatter of bf16 gradients (fp32 accumulation) then
    all-gather of the shards.  p=16, 192 MiB bf16 per rank, N(0, 1e-2), seed 2."""
    launches_per_step = 2
    nccl_bytes_per_rank = 0  # a chain of two collectives: no single NCCL figure

    def __init__(self, p=16, mib=192):
        super().__init__(p, mib, "bf16", 2)
        self.name = "zero_reduce_scatter_all_gather"
        self.kernel_key = f"fold_rs_bf16_p{p}_n{self.n}"

    def config(self):
        return {"workload": f"ZeRO reduce-scatter (fp32 accumulate) then all-gather: p={self.p} x "
                            f"{self.mib} MiB bf16 per rank", "p": self.p, "n_per_rank": self.n,
                "inputs": "N(0, sigma=1e-2), drawn on the device (torch Philox, seed 2)"}

    def setup(self, lib, torch, device):
        self.lib, self.torch = lib, torch
        gen = torch.Generator(device=device)
        gen.manual_seed(2)
        self.send = [(torch.randn(self.n, generator=gen, device=device) * 1e-2).to(torch.bfloat16)
                     for _ in range(self.p)]
        self.recv = [torch.empty_like(s) for s in self.send]
        self.shards = [torch.empty(lib.ccl_chunk_bounds(self.p, self.n, k)[1], dtype=torch.bfloat16,
                                   device=device) for k in range(self.p)]

    def bytes_per_step(self):
        return (self.p * self.n + self.n) * 2 + (self.n + self.p * self.n) * 2

    def step(self, stream):
        self.lib.ccl_reduce_scatter(self.send, self.shards, stream=stream)
        self.lib.ccl_all_gather(self.shards, self.recv, stream=stream)

    def oracle_sample(self, frac):
        from oracle import ring
        return oracle_prefix_sample(self.send, self.n, frac, ring.zero_rs_then_ag,
                                    2 * (self.p + 1) * 2, "oracle ZeRO RS then AG")

    def cpu_ranks_sample(self, frac):
        from oracle import cpu_ranks
        p = self.p
        m = max(p, int(self.n * frac))
        xs = host_prefix(self.send, m)
        t0 = time.perf_counter()
        shards, _, st, threads = cpu_ranks.ring("reduce_scatter", xs, "bf16", timeout_s=600.0)
        if st == cpu_ranks.OK:
            _, _, st, _ = cpu_ranks.ring("all_gather", shards, "bf16", timeout_s=600.0)
        dt = time.perf_counter() - t0
        if st != cpu_ranks.OK:
            raise RuntimeError(f"CPU-rank ring returned status {st}")
        return dt, m * 2 * (p + 1) * 2, (f"CPU-rank ring ZeRO RS then AG on the first {m} of {self.n} elements "
                                         f"of each of the {p} ranks, {threads} threads"), threads

    def parts(self):
        rs = lambda s: self.lib.ccl_reduce_scatter(self.send, self.shards, stream=s)
        ag = lambda s: self.lib.ccl_all_gather(self.shards, self.recv, stream=s)
        return [("fold", (self.p * self.n + self.n) * 2, rs),
                ("gather", (self.n + self.p * self.n) * 2, ag)]


class Moe(Workload):
    """MoE all-to-allv dispatch then combine: p=8, 16,384 tokens x 4096 bf16 per
    source, Zipf(1.2) destination counts (seed 3)."""
    name = "moe_all_to_allv_dispatch_combine"
    kernel = "a2av"
    launches_per_step = 2

    def __init__(self, p=8, tokens=16384, hidden=4096):
        self.p, self.tokens, self.hidden = p, tokens, hidden
        self.kernel_key = f"a2av_moe_p{p}_t{tokens}_h{hidden}"

    def config(self):
        return {"workload": f"MoE all-to-allv dispatch + combine: p={self.p}, {self.tokens} tokens x "
                            f"{self.hidden} bf16 per rank, Zipf(1.2) counts seed 3",
                "p": self.p, "tokens_per_rank": self.tokens, "hidden": self.hidden}

    def setup(self, lib, torch, device):
        from a2a_ring_ordered_gb300 import workloads
        self.lib, self.torch = lib, torch
        self.counts, rng = workloads.moe_counts(self.p, self.tokens, seed=3)
        x = workloads.moe_tokens(self.counts, self.hidden, rng, dtype="bf16")
        self.send = [torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(device) for v in x]
        rows = self.counts.sum(axis=0)
        self.mid = [torch.empty(int(r) * self.hidden, dtype=torch.bfloat16, device=device) for r in rows]
        self.back = [torch.empty_like(s) for s in self.send]
        self.total_rows = int(self.counts.sum())

    def bytes_per_step(self):
        return 2 * 2 * self.total_rows * self.hidden * 2

    def step(self, stream):
        self.lib.ccl_all_to_allv(self.send, self.counts, self.mid, self.hidden, stream=stream)
        self.lib.ccl_all_to_allv(self.mid, self.counts.T, self.back, self.hidden, stream=stream)

    def oracle_sample(self, frac):
        from oracle import collectives
        if not hasattr(self, "_host_tokens"):
            self._host_tokens = host_prefix(self.send, max(t.numel() for t in self.send))
        t0 = time.perf_counter()
        mid = collectives.all_to_allv(self._host_tokens, self.counts, self.hidden)
        collectives.all_to_allv(mid, self.counts.T, self.hidden)
        dt = time.perf_counter() - t0
        return dt, self.bytes_per_step(), "oracle all-to-allv dispatch + combine, full workload"

    def parts(self):
        half = self.bytes_per_step() // 2
        d = lambda s: self.lib.ccl_all_to_allv(self.send, self.counts, self.mid, self.hidden, stream=s)
        c = lambda s: self.lib.ccl_all_to_allv(self.mid, self.counts.T, self.back, self.hidden, stream=s)
        return [("a2av", half, d), ("a2av", half, c)]


class Ddp(Workload):
    """DDP bucketed gradient all-reduce of a synthetic transformer's gradients:
    p=8 ranks, 24 layers of width 1024 (+ embedding), 25 MiB buckets filled in
    backprop order.  One step = every bucket's fused all-reduce + 1/p + bf16."""
    name = "ddp_bucketed_allreduce"
    kernel = "fold"

    def __init__(self, p=8, layers=24, d=1024, vocab=50257):
        self.p, self.layers, self.d, self.vocab = p, layers, d, vocab
        shapes = [(vocab, d)]
        for _ in range(layers):
            shapes += [(3 * d, d), (3 * d,), (d, d), (d,), (d,), (d,), (4 * d, d), (4 * d,),
                       (d, 4 * d), (d,), (d,), (d,)]
        self.shapes = shapes + [(d,), (d,)]
        self.kernel_key = f"fold_ddp_p{p}_l{layers}_d{d}"

    def config(self):
        return {"workload": f"DDP bucketed all-reduce: p={self.p} ranks, {len(self.shapes)} gradients of a "
                            f"{self.layers}-layer d={self.d} transformer ({self.total} fp32 per rank) in "
                            f"{len(self.gb.bucket_numel)} buckets of <= 25 MiB -> bf16",
                "p": self.p, "params_per_rank": self.total, "buckets": len(self.gb.bucket_numel),
                "inputs": "N(0,1e-3) drawn on the device (torch Philox, seed 1)"}

    def setup(self, lib, torch, device):
        from a2a_ring_ordered_gb300.ddp import GradBuckets, OverlappedReducer
        self.lib, self.torch, self.device = lib, torch, device
        self.gb = GradBuckets(self.shapes, self.p, device)
        self.total = sum(self.gb.bucket_numel)
        gen = torch.Generator(device=device)
        gen.manual_seed(1)
        # the synthetic backward copies these into the gradient buckets
        self.src = [[torch.randn(m, generator=gen, device=device) * 1e-3 for _ in range(self.p)]
                    for m in self.gb.bucket_numel]
        for b in range(self.gb.num_buckets):
            for r in range(self.p):
                self.gb.grads[b][r].copy_(self.src[b][r])
        self.red = OverlappedReducer(self.gb)
        self.producer = torch.cuda.Stream(device)

    def bytes_per_step(self):
        return self.p * self.total * 6

    def step(self, stream):
        for b in range(self.gb.num_buckets):
            self.gb.reduce_bucket(b, stream=stream)

    def parts(self):
        big = max(range(self.gb.num_buckets), key=lambda b: self.gb.bucket_numel[b])
        return [("fold", self.p * self.gb.bucket_numel[big] * 6,
                 lambda s: self.gb.reduce_bucket(big, stream=s))]

    def _backward_and_reduce(self, overlap: bool):
        torch = self.torch
        cur = torch.cuda.current_stream(self.device)
        self.producer.wait_stream(cur)
        self.red.comm.wait_stream(cur)
        self.red.start_step()
        with torch.cuda.stream(self.producer):
            for b in range(self.gb.num_buckets):  # buckets fill in backprop order
                for r in range(self.p):
                    self.gb.grads[b][r].copy_(self.src[b][r])
                if overlap:
                    for q in self.gb.members[b]:
                        self.red.mark_ready(q, self.producer)
        if not overlap:
            self.red.comm.wait_stream(self.producer)
            for b in range(self.gb.num_buckets):
                for q in self.gb.members[b]:
                    self.red.mark_ready(q, self.red.comm)
        self.red.finish(cur)
        cur.wait_stream(self.producer)

    def overlap_report(self, reps=5):
        torch = self.torch
        out = {}
        for mode in ("serial", "overlapped"):
            self._backward_and_reduce(mode == "overlapped")
            torch.cuda.synchronize(self.device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream(self.device)
            e0.record(cur)
            for _ in range(reps):
                self._backward_and_reduce(mode == "overlapped")
            e1.record(cur)
            torch.cuda.synchronize(self.device)
            out[f"step_ms_{mode}"] = round(e0.elapsed_time(e1) / reps, 4)
        out["note"] = ("synthetic backward = one device copy per bucket per rank; on one GPU it "
                       "shares HBM with the all-reduce, so overlap hides launch gaps, not bandwidth")
        return out

    def oracle_sample(self, frac):
        from oracle import ring
        b = 0
        m = max(self.p, int(self.gb.bucket_numel[b] * frac))
        xs = host_prefix(self.gb.grads[b], m)
        t0 = time.perf_counter()
        ring.bucket_allreduce_scale_cast(xs, self.gb.scale)
        dt = time.perf_counter() - t0
        return dt, self.p * m * 6, f"oracle bucket all-reduce on the first {m} elements of bucket 0"


class Rooted(Workload):
    """broadcast / reduce / scatter / gather of p ranks x `mib` MiB, root 0."""
    def __init__(self, kind, p=16, mib=64, dtype="f32"):
        self.kind, self.p, self.mib, self.dtype = kind, p, mib, dtype
        self.e = 4 if dtype == "f32" else 2
        self.n = mib * (1 << 20) // self.e
        self.name = kind
        self.kernel = {"broadcast": "gather", "reduce": "fold", "scatter": "ring_step",
                       "gather": "ring_step"}[kind]
        self.kernel_key = f"{kind}_{dtype}_p{p}_n{self.n}"

    def config(self):
        return {"workload": f"{self.kind}: p={self.p} ranks, {self.mib} MiB {self.dtype} per rank, root 0",
                "p": self.p, "n_per_rank": self.n, "inputs": "U(-1,1) drawn on the device (seed 4)"}

    def bytes_per_step(self):
        n, p, e = self.n, self.p, self.e
        return {"broadcast": n + p * n, "reduce": p * n + n, "scatter": 2 * n, "gather": 2 * n}[self.kind] * e

    def setup(self, lib, torch, device):
        self.lib = lib
        gen = torch.Generator(device=device)
        gen.manual_seed(4)
        tdt = torch.float32 if self.dtype == "f32" else torch.bfloat16
        mk = lambda m: (torch.rand(m, generator=gen, device=device) * 2 - 1).to(tdt)
        sizes = [lib.ccl_chunk_bounds(self.p, self.n, k)[1] for k in range(self.p)]
        if self.kind == "broadcast":
            self.a, self.b = mk(self.n), [torch.empty(self.n, dtype=tdt, device=device) for _ in range(self.p)]
        elif self.kind == "reduce":
            self.a, self.b = [mk(self.n) for _ in range(self.p)], torch.empty(self.n, dtype=tdt, device=device)
        elif self.kind == "scatter":
            self.a, self.b = mk(self.n), [torch.empty(m, dtype=tdt, device=device) for m in sizes]
        else:
            self.a, self.b = [mk(m) for m in sizes], torch.empty(self.n, dtype=tdt, device=device)

    def oracle_sample(self, frac):
        from oracle import collectives
        p, e = self.p, self.e
        if self.kind == "broadcast":
            return oracle_prefix_sample([self.a], self.n, frac, lambda xs: collectives.broadcast(xs * p),
                                        (1 + p) * e, f"oracle broadcast to {p} ranks")
        if self.kind == "scatter":
            return oracle_prefix_sample([self.a], self.n, frac, lambda xs: collectives.scatter(xs[0], p),
                                        2 * e, f"oracle scatter to {p} ranks")
        if self.kind == "reduce":
            return oracle_prefix_sample(self.a, self.n, frac,
                                        lambda xs: collectives.reduce_ring(xs, 0, self.dtype),
                                        (p + 1) * e, "oracle reduce (ring reduce-scatter, gather to the root)")
        return oracle_prefix_sample(self.a, self.n // p, frac, lambda xs: collectives.gather(xs),
                                    2 * p * e, "oracle gather to the root")

    def step(self, stream):
        getattr(self.lib, f"ccl_{self.kind}")(self.a, self.b, stream=stream)


class MoeEp(Workload):
    """MoE expert parallelism with routing: p=8 ranks x 4096 tokens, hidden 7168,
    top-8 of 256 experts (Zipf(1.2) popularity).  One step = route + FP8 (or
    bf16) dispatch + weighted bf16 combine."""
    name = "moe_ep_route_dispatch_combine"
    kernel = "moe"
    launches_per_step = 3

    def __init__(self, p=8, tokens=4096, k=8, experts=256, hidden=7168, fp8=True):
        self.p, self.T, self.k, self.E, self.h, self.fp8 = p, tokens, k, experts, hidden, fp8
        self.kernel_key = f"moe_ep_p{p}_t{tokens}_k{k}_e{experts}_h{hidden}_{'fp8' if fp8 else 'bf16'}"

    def config(self):
        return {"workload": f"MoE EP: p={self.p} ranks x {self.T} tokens, hidden {self.h}, top-{self.k} of "
                            f"{self.E} experts, {'FP8' if self.fp8 else 'bf16'} dispatch, bf16 combine",
                "p": self.p, "tokens_per_rank": self.T, "k": self.k, "experts": self.E, "hidden": self.h,
                "inputs": "tokens N(0,1) drawn on the device; routing Gumbel top-k, Zipf(1.2), seed 3"}

    def setup(self, lib, torch, device):
        from a2a_ring_ordered_gb300 import workloads
        self.lib, self.torch = lib, torch
        p, T, k, E, h = self.p, self.T, self.k, self.E, self.h
        gen = torch.Generator(device=device)
        gen.manual_seed(3)
        self.x = [torch.randn(T, h, generator=gen, device=device).to(torch.bfloat16) for _ in range(p)]
        self.ids = [torch.from_numpy(i).to(device) for i in workloads.moe_topk_routing(p, T, k, E, seed=3)]
        self.w = [torch.from_numpy(w).to(device) for w in workloads.moe_gate_weights(p, T, k, seed=4)]
        self.counts = torch.empty(p * p, dtype=torch.int64, device=device)
        self.slots = [torch.empty(T, k, dtype=torch.int32, device=device) for _ in range(p)]
        lib.ccl_moe_route(self.ids, E, self.counts, self.slots)
        rows = self.counts.cpu().numpy().reshape(p, p).sum(axis=0)
        self.rows = [int(r) for r in rows]
        dt = torch.uint8 if self.fp8 else torch.bfloat16
        self.recv = [torch.empty(r, h, dtype=dt, device=device) for r in self.rows]
        self.scales = [torch.empty(r, h // 128, device=device) for r in self.rows] if self.fp8 else None
        # expert outputs (bf16, dispatch layout) for the combine
        self.y = [torch.randn(r, h, generator=gen, device=device).to(torch.bfloat16) for r in self.rows]
        self.out = [torch.empty(T, h, dtype=torch.bfloat16, device=device) for _ in range(p)]

    def _bytes(self):
        p, T, k, h = self.p, self.T, self.k, self.h
        rows = p * T * k
        route = 2 * rows * 4
        disp = p * T * h * 2 + rows * (h + h // 32 if self.fp8 else 2 * h)
        comb = rows * h * 2 + p * T * h * 2 + rows * 4
        return route, disp, comb

    def bytes_per_step(self):
        return sum(self._bytes())

    def oracle_sample(self, frac):
        """Route, dispatch and combine of the first frac*T tokens of every source."""
        from oracle import moe
        p, T, k, E, h = self.p, self.T, self.k, self.E, self.h
        t1 = max(1, int(T * frac))
        xs = [a.reshape(-1) for a in host_prefix(self.x, t1)]
        ids = [i[:t1].reshape(-1).cpu().numpy() for i in self.ids]
        w = [x[:t1].reshape(-1).cpu().numpy() for x in self.w]
        counts, _, _ = moe.route(ids, p, E)
        rows = counts.sum(axis=0)
        ys = [host_prefix([self.y[d]], int(rows[d]))[0] for d in range(p)]
        t0 = time.perf_counter()
        moe.route(ids, p, E)
        moe.dispatch(xs, ids, p, k, E, h, fp8=self.fp8)
        moe.combine(ys, ids, w, p, k, E, h)
        dt = time.perf_counter() - t0
        nb = int(self.bytes_per_step() * t1 / T)
        return dt, nb, (f"oracle route + {'FP8' if self.fp8 else 'bf16'} dispatch + combine of the first "
                        f"{t1} of {T} tokens of each of the {p} sources")

    def _route(self, s):
        self.lib.ccl_moe_route(self.ids, self.E, self.counts, self.slots, stream=s)

    def _dispatch(self, s):
        self.lib.ccl_moe_dispatch(self.x, self.ids, self.counts, self.slots, self.E, self.recv,
                                  self.scales, None, fp8=self.fp8, stream=s)

    def _combine(self, s):
        self.lib.ccl_moe_combine(self.y, self.ids, self.w, self.counts, self.slots, self.E, self.out,
                                 stream=s)

    def step(self, stream):
        self._route(stream)
        self._dispatch(stream)
        self._combine(stream)

    def parts(self):
        r, d, c = self._bytes()
        return [("moe_route", r, self._route), ("moe_dispatch", d, self._dispatch),
                ("moe_combine", c, self._combine)]


class Ulysses(Workload):
    """Ulysses head <-> sequence all-to-all: p ranks x (S/p tokens, H heads,
    D = 128) bf16, forward then inverse (2 launches)."""
    kernel = "ulysses"
    launches_per_step = 2

    def __init__(self, p=8, seq_per_rank=8192, heads=32, head_dim=128):
        self.p, self.sp, self.H, self.D = p, seq_per_rank, heads, head_dim
        self.n = seq_per_rank * heads * head_dim
        self.name = "ulysses_all_to_all"
        self.kernel_key = f"ulysses_p{p}_s{seq_per_rank}_h{heads}_d{head_dim}"

    def config(self):
        return {"workload": f"Ulysses head<->sequence all-to-all: p={self.p} ranks x {self.sp} tokens x "
                            f"{self.H} heads x {self.D} bf16, forward + inverse",
                "p": self.p, "tokens_per_rank": self.sp, "heads": self.H, "head_dim": self.D,
                "inputs": "N(0,1) drawn on the device (torch Philox, seed 5)"}

    def setup(self, lib, torch, device):
        self.lib = lib
        gen = torch.Generator(device=device)
        gen.manual_seed(5)
        self.x = [torch.randn(self.n, generator=gen, device=device).to(torch.bfloat16) for _ in range(self.p)]
        self.y = [torch.empty_like(t) for t in self.x]
        self.z = [torch.empty_like(t) for t in self.x]

    def bytes_per_step(self):
        return 2 * 2 * self.p * self.n * 2

    def _fwd(self, s):
        self.lib.ccl_all_to_all_heads(self.x, self.y, self.sp, self.H, self.D, stream=s)

    def _inv(self, s):
        self.lib.ccl_all_to_all_heads(self.y, self.z, self.sp, self.H, self.D, inverse=True, stream=s)

    def step(self, stream):
        self._fwd(stream)
        self._inv(stream)

    def parts(self):
        half = self.bytes_per_step() // 2
        return [("ulysses", half, self._fwd), ("ulysses", half, self._inv)]

    def oracle_sample(self, frac):
        """Forward and inverse exchange of the first frac*S/p tokens of every shard."""
        from oracle import collectives
        t1 = max(1, int(self.sp * frac))
        xs = host_prefix(self.x, t1 * self.H * self.D)
        t0 = time.perf_counter()
        y = collectives.ulysses_seq_to_heads(xs, self.H, self.D)
        collectives.ulysses_heads_to_seq(y, self.H, self.D)
        dt = time.perf_counter() - t0
        return dt, int(self.bytes_per_step() * t1 / self.sp), (
            f"oracle forward + inverse exchange of the first {t1} of {self.sp} tokens of each of the {self.p} shards")


def make_workload(a) -> Workload:
    if a.workload == "bucket":
        return Bucket()
    if a.workload == "allreduce":
        return AllReduce(p=a.p or 16, mib=a.mib or 256, dtype=a.dtype, schedule=a.schedule,
                         group=a.group, wire=a.wire)
    if a.workload == "literal":
        return AllReduce(p=a.p or 8, mib=a.mib or 25, dtype=a.dtype, literal=True)
    if a.workload == "reduce_scatter":
        return ReduceScatter(p=a.p or 16, mib=a.mib or 192, dtype=a.dtype if a.dtype != "f32" else "bf16",
                             wire=a.wire)
    if a.workload == "all_gather":
        return AllGather(p=a.p or 16, mib=a.mib or 192, dtype=a.dtype if a.dtype != "f32" else "bf16")
    if a.workload == "zero":
        return Zero()
    if a.workload == "moe":
        return Moe()
    if a.workload == "ddp":
        return Ddp()
    if a.workload == "ulysses":
        return Ulysses(p=a.p or 8)
    if a.workload == "moe_ep":
        return MoeEp(fp8=a.dtype != "bf16")
    if a.workload in ("broadcast", "reduce", "scatter", "gather"):
        return Rooted(a.workload, p=a.p or 16, mib=a.mib or 64, dtype=a.dtype)
    raise SystemExit(f"unknown workload {a.workload}")


# ------------------------------------------------------------- distributed
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (timing only; not on the data path)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------- arms
def cpu_cores_used() -> int:
    return 1  # numpy element-wise arithmetic runs on one thread


def host_description() -> dict:
    """The host the CPU baselines ran on: cores available to this process
    (nproc) and the machine / CPU model."""
    import platform
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu part", "processor name") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"host_cores": cores, "machine": platform.machine(), "cpu": model}


def run_reference(a, wl: Workload, rank: int, world: int) -> dict | None:
    """The oracle, as it stands, on the host cores: each step a bounded sample."""
    if rank != 0:
        return None
    budget_s = 90.0
    if a.steps <= 0:
        a.steps = 20
    # first sample sizes the rest: aim for the whole run within ~budget_s
    wl_host = wl
    if not hasattr(wl_host, "x"):
        wl_host.x = wl_host.host_inputs()
    t_full, _, _ = wl_host.oracle_sample(1.0)
    per_step = budget_s / max(1, a.steps + a.warmup)
    frac = min(1.0, per_step / max(t_full, 1e-9))
    for _ in range(a.warmup):
        wl_host.oracle_sample(frac)
    times, nbytes, desc = [], 0, ""
    for _ in range(a.steps):
        dt, nb, desc = wl_host.oracle_sample(frac)
        times.append(dt)
        nbytes = nb
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    cfg = wl.config()
    cfg["l2"] = "host oracle"
    return {
        "metric": "effective GB/s (primitive minimum bytes / step time) and fraction of HBM roofline",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "impl": "reference", "config": cfg,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores_used(),
                         "kind": "oracle", "sample": desc, **host_description()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def cpu_baseline(wl: Workload) -> dict | None:
    """Time the oracle on the host for ~10-30 s of work (rank 0, N=1 only): the
    full workload when one pass takes under ~1 s, else a prefix sample."""
    try:
        t1, _, _ = wl.oracle_sample(0.01)
    except NotImplementedError:
        return None
    frac = min(1.0, 0.01 * 1.0 / max(t1, 1e-6))  # one sample of about a second
    t_s, nb, desc = wl.oracle_sample(frac)
    reps = max(1, min(200, int(12.0 / max(t_s, 1e-6))))  # about 12 s of host work
    times = [t_s]
    for _ in range(reps - 1):
        dt, nb, desc = wl.oracle_sample(frac)
        times.append(dt)
    t = statistics.median(times)
    out = {"value": round(nb / t / 1e9, 4), "unit": "GB/s", "cores": cpu_cores_used(),
           "kind": "oracle", "sample": f"{desc}; median of {len(times)} runs",
           "seconds_per_sample": round(t, 4), **host_description()}
    # the ring on CPU ranks (one host thread per virtual rank), same workload
    try:
        t1, _, _, _ = wl.cpu_ranks_sample(0.01)
    except NotImplementedError:
        return out
    frac = min(1.0, 0.01 * 1.0 / max(t1, 1e-6))
    times = []
    for _ in range(max(1, min(200, int(12.0 / max(t1 / 0.01 * frac, 1e-6))))):
        dt, nb, desc, threads = wl.cpu_ranks_sample(frac)
        times.append(dt)
    t = statistics.median(times)
    out["cpu_ranks"] = {"value": round(nb / t / 1e9, 4), "unit": "GB/s", "cores": threads,
                        "kind": "oracle_cpu_ranks", "sample": f"{desc}; median of {len(times)} runs",
                        "seconds_per_sample": round(t, 4)}
    return out


def run_ours(a, wl: Workload, rank: int, world: int, local: int) -> dict | None:
    import torch
    from a2a_ring_ordered_gb300 import ccl as lib

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl.setup(lib, torch, device)
    stream = torch.cuda.current_stream(device)

    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(a.warmup):
        wl.step(stream)
    w1.record(stream)
    torch.cuda.synchronize(device)

    def capture(g):
        """A CUDA graph of g steps, replayed once (warm)."""
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            for _ in range(g):
                wl.step(cap)
        stream.wait_stream(cap)
        with torch.cuda.stream(stream):
            gr.replay()
        torch.cuda.synchronize(device)
        return gr

    # The timed steps replay a CUDA graph of G steps (G divides K), so that the
    # host cost of issuing a call never leaves the GPU idle between steps;
    # --eager issues every step from Python instead.
    graph, group = None, 1
    if a.steps <= 0:  # auto: about one second of timed device work, from warm steps
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if a.eager:
            p0.record(stream)
            for _ in range(20):
                wl.step(stream)
            p1.record(stream)
            probe = 20
        else:
            graph, group = capture(64), 64
            p0.record(stream)
            with torch.cuda.stream(stream):
                graph.replay()
                graph.replay()
            p1.record(stream)
            probe = 128
        torch.cuda.synchronize(device)
        ms_probe = p0.elapsed_time(p1) / probe
        a.steps = int(max(64, min(200000, round(1000.0 / max(ms_probe, 1e-3)))))
        a.steps = -(-a.steps // 64) * 64  # a multiple of the graph's 64 steps
        a.steps = int(max_over_ranks(float(a.steps), world, device))
    if not a.eager and graph is None:
        group = max(d for d in range(1, min(a.steps, 64) + 1) if a.steps % d == 0)
        graph = capture(group)
    sampler = ClockSampler(local)
    time.sleep(0.05)
    launches0 = lib.ccl_kernel_launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0 = time.time()
    start.record(stream)
    if graph is None:
        for _ in range(a.steps):
            wl.step(stream)
    else:
        with torch.cuda.stream(stream):
            for _ in range(a.steps // group):
                graph.replay()
    stop.record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    barrier(world, device)
    # kernels launched by the timed steps (a replayed graph launches its
    # captured kernels without calling the library again)
    per_step = (lib.ccl_kernel_launch_count() - launches0) if graph is None else None
    if graph is not None:
        c0 = lib.ccl_kernel_launch_count()
        wl.step(stream)
        torch.cuda.synchronize(device)
        per_step = (lib.ccl_kernel_launch_count() - c0) * a.steps
    launches = per_step
    sampler.stop()
    ms_total = start.elapsed_time(stop)
    ms_total = max_over_ranks(ms_total, world, device)
    ms_step = ms_total / a.steps
    nbytes = wl.bytes_per_step()
    value = world * nbytes / (ms_step * 1e-3) / 1e9

    # end to end through the public API with host buffers
    e2e = None
    if hasattr(wl, "e2e_step") and type(wl).e2e_step is not Workload.e2e_step:
        k = max(3, min(a.steps, 20))
        for _ in range(2):
            wl.e2e_step(stream)
        torch.cuda.synchronize(device)
        barrier(world, device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if hasattr(wl, "e2e_begin"):
            wl.e2e_begin(stream)
        for _ in range(k):
            wl.e2e_step(stream)
        if hasattr(wl, "e2e_finish"):
            wl.e2e_finish(stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier(world, device)
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / k, world, device)
        hb, db = wl.e2e_bytes()
        e2e = {"value": round(world * nbytes / (ms_e2e * 1e-3) / 1e9, 3), "unit": "GB/s",
               "ms_per_step": round(ms_e2e, 4), "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
               "steps": k, "path": "cudaMemcpyAsync H2D (copy-in stream), kernel, cudaMemcpyAsync D2H "
                                   "(copy-out stream); step i's copy-out overlaps step i+1's copy-in"}
        if hasattr(wl, "e2e_zero_copy_step"):
            for _ in range(2):
                wl.e2e_zero_copy_step(stream)
            torch.cuda.synchronize(device)
            e0.record(stream)
            for _ in range(k):
                wl.e2e_zero_copy_step(stream)
            e1.record(stream)
            torch.cuda.synchronize(device)
            ms_st = max_over_ranks(e0.elapsed_time(e1) / k, world, device)
            e2e["zero_copy"] = {"value": round(world * nbytes / (ms_st * 1e-3) / 1e9, 3),
                                "ms_per_step": round(ms_st, 4),
                                "path": "kernel reads and writes pinned host memory directly"}

    # the dominant kernel: time each launch of a step on its own (CUDA events on
    # the launching stream, same back-to-back regime)
    part_stats = []
    for name, pbytes, fn in wl.parts():
        k = max(3, min(a.steps, 200))
        for _ in range(3):
            fn(stream)
        pg = None
        if not a.eager:
            cap = torch.cuda.Stream(device)
            cap.wait_stream(stream)
            pg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pg, stream=cap):
                for _ in range(k):
                    fn(cap)
            stream.wait_stream(cap)
            with torch.cuda.stream(stream):
                pg.replay()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        if pg is None:
            for _ in range(k):
                fn(stream)
        else:
            with torch.cuda.stream(stream):
                pg.replay()
        p1.record(stream)
        torch.cuda.synchronize(device)
        ms = max_over_ranks(p0.elapsed_time(p1) / k, world, device)
        part_stats.append((name, pbytes, ms))
        del pg
    if rank != 0:
        return None
    name, pbytes, pms = max(part_stats, key=lambda t: t[2])
    peak, peak_src = measured_peak_gbs()
    achieved = pbytes / (pms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": ("of measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
                            if peak_src == "measured" else "of fallback 6.8 TB/s"),
            "traffic": committed_traffic(wl.kernel_key, KERNEL_SOURCES[name]),
            "kernel": name, "algorithmic_bytes_per_launch": pbytes,
            "ms_per_launch": round(pms, 5)}
    if len(part_stats) > 1:
        roof["launches"] = [{"kernel": n_, "bytes": b_, "ms": round(m_, 5),
                             "gbs": round(b_ / (m_ * 1e-3) / 1e9, 1)} for n_, b_, m_ in part_stats]
    cfg = wl.config()
    footprint = nbytes
    cfg["l2"] = (f"no flush: each step touches {footprint / 1e6:.0f} MB "
                 f"({footprint / L2_BYTES:.1f}x the 129 MB L2), steps back to back")
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "1 GPU, p virtual ranks in HBM"
    cfg["timing"] = ("eager Python calls" if a.eager else
                     f"CUDA graph of {group} steps replayed {a.steps // group} times")
    nccl = None
    if wl.nccl_bytes_per_rank:
        algbw = wl.nccl_bytes_per_rank / (ms_step * 1e-3) / 1e9
        nccl = {"algbw_gbs": round(algbw, 2), "busbw_gbs": round(algbw * wl.nccl_factor, 2),
                "note": "NCCL conventions, for comparison with network figures only"}
    out = {
        "metric": "effective GB/s (primitive minimum bytes / step time) and fraction of HBM roofline",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if wl.dtype == "f32" else wl.dtype, "data": "synthetic",
        "config": cfg, "roofline": roof, "gpu_launches": launches,
        "clocks": sampler.summary(t0, t1),
    }
    if e2e is not None:
        out["e2e"] = e2e
    if nccl is not None:
        out["nccl_style"] = nccl
    if hasattr(wl, "overlap_report"):
        out["overlap"] = wl.overlap_report()
    if world == 1 and not a.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl)
    if world == 1 and a.workload == "bucket" and not a.no_configs:
        t_cfg = time.time()
        out["configs"] = config_records(lib, torch, device, peak)
        out["configs"]["wall_s"] = round(time.time() - t_cfg, 1)
    return out


# ----------------------------------------------- points and their oracle check
def _bits(t) -> np.ndarray:
    """A device tensor on the host as numpy (bf16 as its uint16 bits)."""
    import torch
    h = t.detach().cpu()
    return h.view(torch.int16).numpy().view(np.uint16) if h.dtype == torch.bfloat16 else h.numpy()


def _sample_positions(n: int, count: int, seed: int, edges=()) -> np.ndarray:
    """count random positions in [0, n) plus the given edge positions and both ends."""
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, n, size=min(count, n)), np.array([0, n - 1]), np.asarray(list(edges), np.int64)]
    idx = np.unique(np.concatenate(idx).astype(np.int64))
    return idx[(idx >= 0) & (idx < n)]


def _chunk_edges(lib, p: int, n: int) -> list[int]:
    out = []
    for k in range(p):
        off, ln = lib.ccl_chunk_bounds(p, n, k)
        out += [off - 1, off, off + ln - 1, off + ln]
    return out


def _mismatches(got: np.ndarray, want: np.ndarray) -> int:
    """Elements whose bits differ (NaN payloads and signed zeros included)."""
    g, w = np.ascontiguousarray(got), np.ascontiguousarray(want)
    if g.dtype.itemsize != w.dtype.itemsize or g.size != w.size:
        return max(g.size, w.size)
    return int((g.view(np.uint8).reshape(g.size, -1) != w.view(np.uint8).reshape(w.size, -1)).any(axis=1).sum())


def _gather_from(snd, src: np.ndarray, pos: np.ndarray, dev) -> np.ndarray:
    """Elements snd[src[i]][pos[i]] on the host."""
    import torch
    out = None
    for s_ in np.unique(src):
        sel = src == s_
        v = _bits(snd[int(s_)][torch.from_numpy(pos[sel]).to(dev)])
        if out is None:
            out = np.empty(src.size, dtype=v.dtype)
        out[sel] = v
    return out


def oracle_check_leg(lib, kind: str, dt: str, p: int, n: int, snd, rcv, count: int = 4096, seed: int = 0) -> dict:
    """The CPU-baseline leg's parity check of a measured point (after its timed
    region): the oracle's per-element forms, on the host, at a bounded sample
    of positions -- random ones plus every chunk edge and both ends -- timed,
    and compared bit for bit with the kernel's output there.  all-reduce /
    reduce-scatter: the ring fold ("Networks and Collective Communication"
    section 5.1); all-gather and all-to-all: the placement of section 4.1."""
    import torch
    from oracle import pointwise
    dev = snd[0].device
    mism, nsamp = 0, 0
    t0 = time.perf_counter()
    ranks = sorted({0, p // 2, p - 1})
    if kind in ("allreduce", "reduce_scatter", "all_gather"):
        idx = _sample_positions(n, count, seed, _chunk_edges(lib, p, n))
        it = torch.from_numpy(idx).to(dev)
        k, pos = pointwise.all_gather_source(p, n, idx)  # chunk of each position
        nsamp = idx.size
        if kind == "all_gather":
            want = _gather_from(snd, k, pos, dev)
        else:
            want = pointwise.allreduce_at_columns([_bits(x[it]) for x in snd], idx, n, dt)
        if kind == "reduce_scatter":  # position off(k) + t is element t of rank k's shard
            mism += _mismatches(_gather_from(rcv, k, pos, dev), want)
        else:
            for r in ranks:
                mism += _mismatches(_bits(rcv[r][it]), want)
    elif kind == "all_to_all":
        for j in ranks:
            m = rcv[j].numel()
            if m == 0:
                continue
            ln = m // p
            edges = [i * ln + d for i in range(p) for d in (-1, 0, ln - 1)]
            idx = _sample_positions(m, count, seed + j, edges)
            src, spos = pointwise.all_to_all_source(p, n, j, idx)
            mism += _mismatches(_bits(rcv[j][torch.from_numpy(idx).to(dev)]), _gather_from(snd, src, spos, dev))
            nsamp += idx.size
    else:
        raise ValueError(kind)
    return {"checked": mism == 0, "samples": int(nsamp), "mismatches": int(mism),
            "oracle_s": round(time.perf_counter() - t0, 3),
            "how": f"oracle.pointwise at random positions plus every chunk edge; output ranks {ranks}"}


def _collective(lib, kind):
    return {"allreduce": lib.ccl_allreduce, "reduce_scatter": lib.ccl_reduce_scatter,
            "all_gather": lib.ccl_all_gather, "all_to_all": lib.ccl_all_to_all}[kind]


def measure_point(lib, torch, device, stream, kind: str, dt: str, p: int, n: int, gen, peak: float,
                  init=None, max_calls: int = 4000, target_us: float = 20000.0):
    """Time one collective call of p ranks x n elements: K calls captured in a
    CUDA graph and replayed under CUDA events on ``stream``, rotating over
    enough buffer sets that the rotated footprint is at least twice the L2
    (where memory allows), every rank buffer on a 256-byte boundary.  Returns
    (record, views of the buffer sets).  ``init(j, inputs)`` may overwrite the
    inputs of set j (the default is U(-1, 1) from ``gen``)."""
    e = 4 if dt == "f32" else 2
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    lens = [lib.ccl_chunk_bounds(p, n, k)[1] for k in range(p)]
    in_sizes = lens if kind == "all_gather" else [n] * p
    out_sizes = (lens if kind == "reduce_scatter" else
                 [p * ln for ln in lens] if kind == "all_to_all" else [n] * p)
    pad = 256 // e
    rnd = lambda m: -(-m // pad) * pad
    n_in, n_out = sum(rnd(m) for m in in_sizes), sum(rnd(m) for m in out_sizes)
    foot = (sum(in_sizes) + sum(out_sizes)) * e  # the primitive's minimum bytes
    sets = int(min(64, max(1, -(-2 * L2_BYTES // foot))))
    arena_in = (torch.rand(sets * n_in, generator=gen, device=device) * 2 - 1).to(tdt)
    arena_out = torch.empty(sets * n_out, dtype=tdt, device=device)

    def split(t, sizes):
        out, off = [], 0
        for m in sizes:
            out.append(t[off:off + m])
            off += rnd(m)
        return out

    views = [(split(arena_in[j * n_in:(j + 1) * n_in], in_sizes),
              split(arena_out[j * n_out:(j + 1) * n_out], out_sizes)) for j in range(sets)]
    if init is not None:
        for j in range(sets):
            init(j, views[j][0])
    call = _collective(lib, kind)
    est_us = max(2.0, foot / (peak * 1e3))
    k = int(min(max_calls, max(2 * sets, target_us / est_us)))
    with torch.cuda.stream(stream):
        for j in range(min(sets, 3)):  # warm-up outside capture
            call(views[j][0], views[j][1], stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(k):
            snd, rcv = views[i % sets]
            call(snd, rcv, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / (reps * k)
    del g
    # the last replay left every set's outputs computed from its own inputs
    gbs = foot / (ms * 1e-3) / 1e9
    rec = {"collective": kind, "dtype": dt, "p": p, "n_per_rank": n, "bytes_per_rank": n * e,
           "us_per_call": round(ms * 1e3, 3), "effective_gbs": round(gbs, 1),
           "frac_of_hbm": round(gbs / peak, 4), "algorithmic_bytes_per_call": foot,
           "buffer_sets": sets, "calls_per_graph": k}
    return rec, views


def run_sweep(a) -> int:
    """Message-size sweep of one collective (``--sweep-collective``, default
    the fused all-reduce): one JSON line per point.

    The message size is a rank's full vector (n elements): all-reduce and
    all-to-all move p*n in and p*n out, reduce-scatter p*n in and n out,
    all-gather n in and p*n out (the primitive's minimum bytes).  Per point,
    K calls are captured in a CUDA graph (small messages are launch-bound, and
    host-side call overhead would otherwise leave the GPU idle between
    kernels) and the graph is replayed under CUDA events on the replay stream
    (``measure_point``).  After the timed region the CPU-baseline leg checks
    the point's output against the oracle at sampled positions
    (``oracle_check_leg``); the line carries ``checked``.
    """
    import torch
    from a2a_ring_ordered_gb300 import ccl as lib

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, peak_src = measured_peak_gbs()
    kind = a.sweep_collective
    dtypes = [a.dtype] if a.sweep_dtype_only else ["f32", "bf16"]
    ps = [a.p] if a.p else [2, 4, 8, 16, 72]
    gen = torch.Generator(device=device)
    gen.manual_seed(4)
    s = torch.cuda.Stream(device)
    for dt in dtypes:
        e = 4 if dt == "f32" else 2
        for p in ps:
            top = 28 if p == 72 else 30  # p=72 up to 256 MiB per rank, else 1 GiB
            lgs = ([int(x) for x in a.sweep_sizes.split(",")] if a.sweep_sizes else
                   range(max(10, a.sweep_lo), min(top, a.sweep_hi) + 1, a.sweep_stride))
            for lg in lgs:
                if lg > top:
                    continue
                nbytes_rank = 1 << lg
                n = nbytes_rank // e
                rec, views = measure_point(lib, torch, device, s, kind, dt, p, n, gen, peak)
                chk = oracle_check_leg(lib, kind, dt, p, n, views[0][0], views[0][1], seed=lg)
                ms = rec["us_per_call"] * 1e-3
                bus = {"allreduce": 2 * (p - 1) / p}.get(kind, (p - 1) / p)
                print(json.dumps({
                    "sweep": kind, "dtype": dt, "p": p, "bytes_per_rank": nbytes_rank,
                    "us_per_call": rec["us_per_call"], "effective_gbs": rec["effective_gbs"],
                    "frac_of_hbm": rec["frac_of_hbm"], "peak": peak, "peak_source": peak_src,
                    "algbw_gbs": round(nbytes_rank / (ms * 1e-3) / 1e9, 2),
                    "busbw_gbs": round(nbytes_rank / (ms * 1e-3) / 1e9 * bus, 2),
                    "buffer_sets": rec["buffer_sets"],
                    "rotated_footprint_mb": round(rec["buffer_sets"] * rec["algorithmic_bytes_per_call"] / 1e6, 1),
                    "calls_per_graph": rec["calls_per_graph"], "checked": chk["checked"],
                    "oracle_check": chk}), flush=True)
                del views
                torch.cuda.empty_cache()
    return 0


def config_records(lib, torch, device, peak: float) -> dict:
    """One record per configuration beside the headline's (run after its timed
    region): the worked-example / p=4 fp32 collectives, the ZeRO chain, the
    MoE all-to-allv and the all-reduce sweep at 8 MiB, 64 MiB and 1 GiB per
    rank for p = 2, 16 and 72.  Each entry: effective GB/s and the fraction
    of the measured copy bandwidth per call (CUDA graph of back-to-back calls,
    ``measure_point``), the kernel's per-launch time, and the CPU-baseline
    leg's oracle check."""
    from a2a_ring_ordered_gb300 import workloads
    out: dict = {}
    s = torch.cuda.Stream(device)
    gen = torch.Generator(device=device)
    kernel = {"allreduce": "fold", "reduce_scatter": "fold", "all_gather": "gather", "all_to_all": "a2av"}

    def point(kind, dt, p, n, init=None, seed=0, count=4096):
        rec, views = measure_point(lib, torch, device, s, kind, dt, p, n, gen, peak, init=init)
        rec["kernel"] = kernel[kind]
        rec["ms_per_launch"] = round(rec["us_per_call"] * 1e-3, 6)
        rec["oracle_check"] = oracle_check_leg(lib, kind, dt, p, n, views[0][0], views[0][1], count=count,
                                               seed=seed)
        rec["checked"] = rec["oracle_check"]["checked"]
        del views
        torch.cuda.empty_cache()
        return rec

    # (1) p=4 fp32, n=1,048,576 per rank ~ N(0,1) from seed 0 (set 0 holds
    # exactly those inputs; the other rotation sets U(-1,1))
    p, n = 4, 1_048_576
    x = workloads.normal(p, n, 1.0, seed=0)
    blocks = [x[k][off:off + ln] for k, (off, ln) in
              ((k, lib.ccl_chunk_bounds(p, n, k)) for k in range(p))]

    def init_full(j, ins):
        if j == 0:
            for r, t in enumerate(ins):
                t.copy_(torch.from_numpy(x[r]))

    def init_blocks(j, ins):
        if j == 0:
            for r, t in enumerate(ins):
                t.copy_(torch.from_numpy(blocks[r]))
    gen.manual_seed(0)
    out["1_p4_f32_n1048576"] = {
        "workload": "p=4 fp32, n=1,048,576 per rank ~ N(0,1) seed 0 (4 MiB per rank)",
        "allreduce": point("allreduce", "f32", p, n, init_full, count=1 << 16),
        "reduce_scatter": point("reduce_scatter", "f32", p, n, init_full, count=1 << 16),
        "all_gather": point("all_gather", "f32", p, n, init_blocks, count=1 << 16),
        "all_to_all": point("all_to_all", "f32", p, n, init_full, count=1 << 16)}

    # (3) ZeRO: p=16 x 100,663,296 bf16 ~ N(0, 1e-2), seed 2: RS then AG
    z = Zero()
    z.setup(lib, torch, device)
    zrec = {"workload": "ZeRO reduce-scatter then all-gather, p=16 x 192 MiB bf16, N(0, 1e-2) seed 2"}
    for name, nb, fn in z.parts():
        zrec[("reduce_scatter" if name == "fold" else "all_gather")] = _time_part(torch, device, s, fn, nb, peak, name)
    chain = zrec["reduce_scatter"]["ms_per_launch"] + zrec["all_gather"]["ms_per_launch"]
    zrec["chain"] = {"ms": round(chain, 5), "effective_gbs": round(z.bytes_per_step() / (chain * 1e-3) / 1e9, 1),
                     "frac_of_hbm": round(z.bytes_per_step() / (chain * 1e-3) / 1e9 / peak, 4)}
    chk_rs = oracle_check_leg(lib, "reduce_scatter", "bf16", z.p, z.n, z.send, z.shards, count=1 << 16, seed=3)
    chk_ar = oracle_check_leg(lib, "allreduce", "bf16", z.p, z.n, z.send, z.recv, count=1 << 16, seed=4)
    zrec["oracle_check"] = {"reduce_scatter": chk_rs, "all_gather_of_shards_equals_allreduce": chk_ar}
    zrec["checked"] = chk_rs["checked"] and chk_ar["checked"]
    out["3_zero_p16_bf16_192MiB"] = zrec
    del z
    torch.cuda.empty_cache()

    # (4) MoE all-to-allv dispatch + combine, p=8, Zipf(1.2) counts, seed 3
    m = Moe()
    m.setup(lib, torch, device)
    mrec = {"workload": "MoE all-to-allv dispatch + combine: p=8, 16,384 tokens x 4096 bf16 per rank, "
                        "Zipf(1.2) counts seed 3"}
    for (name, nb, fn), what in zip(m.parts(), ("dispatch", "combine")):
        mrec[what] = _time_part(torch, device, s, fn, nb, peak, name)
    m.step(s)
    torch.cuda.synchronize(device)
    mrec["oracle_check"] = moe_check_leg(m)
    mrec["checked"] = mrec["oracle_check"]["checked"]
    out["4_moe_p8_zipf"] = mrec
    del m
    torch.cuda.empty_cache()

    # (5) all-reduce at 8 MiB, 64 MiB and 1 GiB per rank (p=72: 256 MiB), U(-1,1) seed 4
    gen.manual_seed(4)
    pts = []
    for dt in ("f32", "bf16"):
        e = 4 if dt == "f32" else 2
        for p in (2, 16, 72):
            for mib in (8, 64, 256 if p == 72 else 1024):
                pts.append(point("allreduce", dt, p, (mib << 20) // e, seed=mib))
    out["5_allreduce_sweep"] = pts
    return out


def _time_part(torch, device, stream, fn, nbytes: int, peak: float, kernel: str, calls: int = 20) -> dict:
    """K back-to-back launches of one part in a CUDA graph, CUDA events."""
    for _ in range(2):
        fn(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / calls
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "ms_per_launch": round(ms, 5), "algorithmic_bytes_per_launch": nbytes,
            "effective_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4)}


def moe_check_leg(m, rows_per_dest: int = 512, seed: int = 3) -> dict:
    """The CPU-baseline leg's check of the MoE exchange: sampled received rows
    of every destination (random rows plus the first and last row of every
    source's block) against the oracle's all-to-allv placement, and the
    combine's rows against the sender's (combine of dispatch = identity)."""
    import torch
    from oracle import pointwise
    t0 = time.perf_counter()
    rng = np.random.default_rng(seed)
    mism, nrows = 0, 0
    h = m.hidden
    dev = m.send[0].device
    for d in range(m.p):
        total = int(m.counts[:, d].sum())
        if total == 0:
            continue
        starts = np.concatenate([[0], np.cumsum(m.counts[:, d])])
        edges = np.concatenate([starts[:-1], starts[1:] - 1])
        rows = np.unique(np.concatenate([rng.integers(0, total, rows_per_dest), edges]))
        rows = rows[(rows >= 0) & (rows < total)]
        src, srow = pointwise.all_to_allv_source(m.counts, d, rows)
        got = _bits(m.mid[d].view(-1, h)[torch.from_numpy(rows).to(dev)])
        want = np.empty_like(got)
        for a_ in np.unique(src):
            sel = src == a_
            want[sel] = _bits(m.send[int(a_)].view(-1, h)[torch.from_numpy(srow[sel]).to(dev)])
        mism += int((got != want).any(axis=1).sum())
        nrows += rows.size
    for s_ in range(m.p):
        total = int(m.counts[s_].sum())
        rows = np.unique(np.concatenate([rng.integers(0, total, rows_per_dest), [0, total - 1]]))
        it = torch.from_numpy(rows).to(dev)
        got, want = _bits(m.back[s_].view(-1, h)[it]), _bits(m.send[s_].view(-1, h)[it])
        mism += int((got != want).any(axis=1).sum())
        nrows += rows.size
    return {"checked": mism == 0, "rows_checked": int(nrows), "mismatching_rows": int(mism),
            "oracle_s": round(time.perf_counter() - t0, 3),
            "how": "oracle.pointwise.all_to_allv_source for sampled received rows; combine rows vs sent rows"}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: enough for ~1 s of device time, so the "
                         "clock record holds hundreds of samples)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bucket",
                    choices=["bucket", "allreduce", "reduce_scatter", "all_gather", "zero", "moe",
                             "literal", "ddp", "broadcast", "reduce", "scatter", "gather", "moe_ep",
                             "ulysses"])
    ap.add_argument("--p", type=int, default=0)
    ap.add_argument("--mib", type=int, default=0)
    ap.add_argument("--dtype", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--schedule", default="ring",
                    choices=["ring", "recursive_doubling", "rabenseifner", "binomial_tree", "naive",
                             "hierarchical"],
                    help="fold order of --workload allreduce")
    ap.add_argument("--wire", default="fp32", choices=["fp32", "bf16"],
                    help="bf16 all-reduce / reduce-scatter: partials travel in fp32 (default) or are "
                         "rounded to bf16 at every hop")
    ap.add_argument("--group", type=int, default=8,
                    help="ranks per group of --schedule hierarchical (groups of consecutive ranks)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration records that follow the default bench line")
    ap.add_argument("--eager", action="store_true",
                    help="issue every timed step from Python instead of replaying a CUDA graph")
    ap.add_argument("--sweep", action="store_true",
                    help="all-reduce message-size sweep (1 KiB..1 GiB per rank), one line per point")
    ap.add_argument("--sweep-stride", type=int, default=1, help="log2 step between sweep sizes")
    ap.add_argument("--sweep-dtype-only", action="store_true", help="sweep only --dtype")
    ap.add_argument("--sweep-lo", type=int, default=10, help="log2 of the smallest per-rank message (bytes)")
    ap.add_argument("--sweep-hi", type=int, default=30, help="log2 of the largest per-rank message (bytes)")
    ap.add_argument("--sweep-sizes", default="",
                    help="comma-separated log2 per-rank message sizes (bytes), in place of --sweep-lo/hi/stride")
    ap.add_argument("--sweep-collective", default="allreduce",
                    choices=["allreduce", "reduce_scatter", "all_gather", "all_to_all"],
                    help="collective of --sweep")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    if a.sweep:
        return run_sweep(a)
    rank, world, local = dist_env()
    wl = make_workload(a)
    if a.impl == "reference":
        # host-only: rank 0 times the oracle, the other ranks exit without work
        if a.workload != "bucket":
            raise SystemExit("the reference arm times the oracle on the default bucket workload")
        out = run_reference(a, wl, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    out = run_ours(a, wl, rank, world, local)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
