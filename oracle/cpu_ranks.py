"""The literal ring on CPU "ranks" -- ctypes shim over ``cpu_ranks.cpp``.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

``cpu_ranks.cpp`` runs the schedule of ``oracle/ring.py`` with one host thread
per virtual rank (at most ``max_threads``; ranks are dealt round-robin to the
threads): each rank keeps its own buffer and an inbox, and the ranks move in
lock step, a barrier after every send and every receive.  It serves two ends:

* a second CPU baseline beside the single-threaded oracle -- the ring as the
  pages' devices run it, on as many host cores as there are ranks;
* host-side fault injection: a rank that stalls (stops taking part from a
  step on) or skips one send; every wait is bounded, so the collective ends
  with TIMEOUT or LOST_MESSAGE instead of hanging.

Its results must equal ``oracle/ring.py`` bit for bit (tests/test_oracle_cpu_ranks.py).
The shared library is compiled on first use with the host C++ compiler into
``oracle/_build/`` (``build()`` does it ahead of time).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

from .ring import chunk_bounds

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpu_ranks.cpp")
LIB = os.path.join(HERE, "_build", "libcpuranks.so")

OK, INVALID, TIMEOUT, LOST_MESSAGE = 0, 1, 4, 5
KINDS = {"allreduce": 0, "reduce_scatter": 1, "all_gather": 2, "bucket": 3}
DTYPES = {"f32": 0, "bf16": 1, "i32": 2}
OPS = {"sum": 0, "max": 1, "min": 2}
FAULTS = {None: 0, "stall": 1, "skip_send": 2}
_NP = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}

_lib = None


def build(force: bool = False) -> str:
    """Compile cpu_ranks.cpp (g++ -O2, no FMA contraction) if missing or stale."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        raise RuntimeError("a C++ compiler (g++) is needed for the CPU-rank oracle")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.run([cxx, "-std=c++17", "-O2", "-ffp-contract=off", "-Wall", "-Wextra", "-fPIC", "-shared",
                    "-pthread", SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        pp = ctypes.POINTER(ctypes.c_void_p)
        L.o3_ring.argtypes = [ctypes.c_int, pp, pp, ctypes.c_int, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                              ctypes.c_float, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_int)]
        L.o3_ring.restype = ctypes.c_int
        _lib = L
    return _lib


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def ring(kind: str, x: list[np.ndarray], dtype: str = "f32", op: str = "sum", scale: float = 1.0,
         max_threads: int | None = None, timeout_s: float = 60.0, fault: str | None = None,
         fault_rank: int = 0, fault_step: int = 0):
    """Run one collective on CPU ranks.

    kind: "allreduce" / "bucket" (x[r] has n elements, output n), "reduce_scatter"
    (output len(k)), "all_gather" (x[k] has len(k) elements, output n).  The
    bucket takes fp32 gradients and returns bf16 bits: the fp32 ring sum times
    ``scale``, rounded once.  Returns (outputs, bytes_sent, status, threads):
    outputs are None unless status is OK.
    """
    p = len(x)
    if kind == "all_gather":
        n = sum(len(v) for v in x)
    else:
        n = len(x[0]) if p else 0
    in_dt = _NP["f32" if kind == "bucket" else dtype]
    xs = [np.ascontiguousarray(v, dtype=in_dt) for v in x]
    bounds = chunk_bounds(p, n)
    out_dt = np.uint16 if kind == "bucket" else _NP[dtype]
    if kind == "reduce_scatter":
        outs = [np.zeros(ln, dtype=out_dt) for _, ln in bounds]
    else:
        outs = [np.zeros(n, dtype=out_dt) for _ in range(p)]
    send = (ctypes.c_void_p * p)(*[v.ctypes.data for v in xs])
    recv = (ctypes.c_void_p * p)(*[o.ctypes.data for o in outs])
    sent = (ctypes.c_uint64 * p)()
    used = ctypes.c_int(0)
    threads = max_threads if max_threads is not None else min(p, host_cores())
    st = _load().o3_ring(KINDS[kind], send, recv, p, n, DTYPES["f32" if kind == "bucket" else dtype],
                         OPS[op], scale, threads, timeout_s, FAULTS[fault], fault_rank, fault_step,
                         sent, ctypes.byref(used))
    return (outs if st == OK else None), list(sent), st, used.value
