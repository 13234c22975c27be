"""Thin Python binding of ``libccl.so`` (include/ccl.h), same names as the C ABI.

Argument marshalling only: each function checks tensor devices, dtypes and
sizes (the C side trusts sizes), packs the per-rank device pointers into
host arrays and calls the library on the current torch stream.  Every
computation runs in the library's CUDA kernels; there is no CPU fallback.
Importing this module fails loudly when the library is missing.

Tensors are the p per-rank buffers of a collective: lists of contiguous CUDA
tensors (torch only provides the device memory and the stream).
"""
from __future__ import annotations

import ctypes
import functools
import os
from typing import Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# CCL_LIBRARY overrides the in-tree library (e.g. a build kept elsewhere)
LIB_PATH = os.environ.get("CCL_LIBRARY") or os.path.join(_PKG, "lib", "libccl.so")

CCL_OK, CCL_ERR_INVALID_ARG, CCL_ERR_UNSUPPORTED, CCL_ERR_CUDA, CCL_ERR_TIMEOUT = 0, 1, 2, 3, 4
CCL_F32, CCL_BF16, CCL_I32 = 0, 1, 2
CCL_SUM, CCL_MAX, CCL_MIN = 0, 1, 2
CCL_KIND_ALLREDUCE, CCL_KIND_REDUCE_SCATTER, CCL_KIND_ALL_GATHER = 0, 1, 2
SCHEDULES = {"ring": 0, "recursive_doubling": 1, "rabenseifner": 2, "binomial_tree": 3, "naive": 4}
CCL_MAX_RANKS = 128

_DTYPES = {torch.float32: CCL_F32, torch.bfloat16: CCL_BF16, torch.int32: CCL_I32}
_OPS = {"sum": CCL_SUM, "max": CCL_MAX, "min": CCL_MIN}


class A2APlan(ctypes.Structure):
    """ccl_a2a_plan_t."""
    _fields_ = [("form", ctypes.c_int), ("shift", ctypes.c_int), ("stage", ctypes.c_int),
                ("launches", ctypes.c_int), ("tile_bytes", ctypes.c_uint)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m a2a_ring_ordered_gb300.build` "
            "(there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
    pp = ctypes.POINTER(ctypes.c_void_p)
    st = ctypes.c_int
    sigs = {
        "ccl_abi_version": (i32, []),
        "ccl_status_string": (ctypes.c_char_p, [st]),
        "ccl_last_error": (ctypes.c_char_p, []),
        "ccl_kernel_launch_count": (u64, []),
        "ccl_chunk_bounds": (st, [i32, sz, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "ccl_fold_plan": (st, [i32, i32, i32, i32, sz, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "ccl_device_error_flag": (st, [ctypes.POINTER(ctypes.c_uint), i32]),
        "ccl_stream_check": (st, [vp]),
        "ccl_selftest_bounded_wait": (st, [vp]),
        "ccl_allreduce": (st, [pp, pp, i32, sz, i32, i32, vp]),
        "ccl_allreduce_schedule": (st, [pp, pp, i32, sz, i32, i32, i32, vp]),
        "ccl_allreduce_hierarchical": (st, [pp, pp, i32, i32, sz, i32, i32, vp]),
        "ccl_allreduce_bf16_wire": (st, [pp, pp, i32, sz, vp]),
        "ccl_all_to_all": (st, [pp, pp, i32, sz, i32, vp]),
        "ccl_reduce_scatter_bf16_wire": (st, [pp, pp, i32, sz, vp]),
        "ccl_reduce_scatter": (st, [pp, pp, i32, sz, i32, i32, vp]),
        "ccl_all_gather": (st, [pp, pp, i32, sz, i32, vp]),
        "ccl_broadcast": (st, [vp, pp, i32, sz, i32, i32, vp]),
        "ccl_reduce": (st, [pp, vp, i32, sz, i32, i32, i32, vp]),
        "ccl_scatter": (st, [vp, pp, i32, sz, i32, i32, vp]),
        "ccl_gather": (st, [pp, vp, i32, sz, i32, i32, vp]),
        "ccl_bucket_allreduce_scale_cast": (st, [pp, pp, i32, sz, ctypes.c_float, vp]),
        "ccl_all_to_allv": (st, [pp, ctypes.POINTER(sz), pp, i32, sz, i32, vp]),
        "ccl_all_to_all_plan": (st, [pp, pp, i32, sz, i32, i32, ctypes.POINTER(A2APlan)]),
        "ccl_all_to_allv_plan": (st, [pp, ctypes.POINTER(sz), pp, i32, sz, i32, i32, ctypes.POINTER(A2APlan)]),
        "ccl_ring_literal_workspace_bytes": (sz, [i32, i32, sz, i32]),
        "ccl_moe_route": (st, [pp, i32, sz, i32, i32, vp, pp, vp]),
        "ccl_all_to_all_heads": (st, [pp, pp, i32, sz, sz, sz, i32, i32, vp]),
        "ccl_moe_dispatch": (st, [pp, pp, vp, pp, i32, sz, i32, i32, sz, i32, pp, ctypes.POINTER(sz),
                                  pp, pp, vp]),
        "ccl_moe_combine": (st, [pp, ctypes.POINTER(sz), pp, pp, vp, pp, i32, sz, i32, i32, sz, pp, vp]),
        "ccl_plan_buckets": (st, [ctypes.POINTER(sz), sz, sz, sz, ctypes.POINTER(ctypes.c_uint32),
                                  ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "ccl_ring_allreduce_literal": (st, [pp, pp, i32, sz, i32, i32, ctypes.POINTER(u64), vp, sz, vp]),
        "ccl_ring_reduce_scatter_literal": (st, [pp, pp, i32, sz, i32, i32, ctypes.POINTER(u64), vp, sz, vp]),
        "ccl_ring_all_gather_literal": (st, [pp, pp, i32, sz, i32, ctypes.POINTER(u64), vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.ccl_abi_version() != 1:
        raise ImportError("libccl.so ABI version mismatch; rebuild it")
    return lib


LIB = _load()


class CclError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = LIB.ccl_last_error().decode()
        super().__init__(f"{what}: {LIB.ccl_status_string(status).decode()}"
                         + (f" -- {detail}" if detail else ""))


def _check(status: int, what: str) -> None:
    if status != CCL_OK:
        raise CclError(status, what)


# ----------------------------------------------------------------- marshalling
def _ptr_array(ptrs: Sequence[int]):
    arr = (ctypes.c_void_p * len(ptrs))()
    for i, v in enumerate(ptrs):
        arr[i] = v
    return arr


def _tensors(ts: Sequence[torch.Tensor], name: str) -> list[torch.Tensor]:
    ts = list(ts)
    if not 1 <= len(ts) <= CCL_MAX_RANKS:
        raise ValueError(f"{name}: need 1..{CCL_MAX_RANKS} rank buffers, got {len(ts)}")
    dev = ts[0].device
    for i, t in enumerate(ts):
        # CUDA tensors, or pinned host tensors: the GPU reads and writes pinned
        # host memory directly (over NVLink-C2C on GB300)
        if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name}[{i}] must be a CUDA tensor or a pinned host tensor")
        if t.is_cuda and dev.type == "cuda" and t.device != dev:
            raise ValueError(f"{name}[{i}] is on {t.device}, expected {dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{i}] must be contiguous")
        if t.dtype != ts[0].dtype:
            raise ValueError(f"{name}[{i}] has dtype {t.dtype}, expected {ts[0].dtype}")
    return ts


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype} (float32, bfloat16, int32)") from None


def _op_code(op: str) -> int:
    try:
        return _OPS[op]
    except KeyError:
        raise ValueError(f"op must be one of {sorted(_OPS)}") from None


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device if device.type == "cuda" else None)
    return int(stream.cuda_stream)


@functools.lru_cache(maxsize=512)
def _chunk_lengths(p: int, n: int) -> tuple[int, ...]:
    """Expected per-rank shard sizes, for size checks: the lengths the
    library's own ``ccl_chunk_bounds`` gives (asked once per (p, n), so the
    binding keeps no copy of the chunk rule and adds no per-call cost)."""
    lens = []
    off, ln = ctypes.c_size_t(), ctypes.c_size_t()
    for c in range(p):
        _check(LIB.ccl_chunk_bounds(p, n, c, ctypes.byref(off), ctypes.byref(ln)), "ccl_chunk_bounds")
        lens.append(ln.value)
    return tuple(lens)


def _numel_check(ts, want, name):
    for i, (t, w) in enumerate(zip(ts, want)):
        if t.numel() != w:
            raise ValueError(f"{name}[{i}] has {t.numel()} elements, expected {w}")


# ------------------------------------------------------------------ utilities
def ccl_abi_version() -> int:
    return LIB.ccl_abi_version()


def ccl_status_string(status: int) -> str:
    return LIB.ccl_status_string(status).decode()


def ccl_last_error() -> str:
    return LIB.ccl_last_error().decode()


def ccl_kernel_launch_count() -> int:
    return LIB.ccl_kernel_launch_count()


def ccl_device_error_flag(clear: bool = False) -> int:
    """The device error word (nonzero once a bounded device-side wait ran out)."""
    flag = ctypes.c_uint(0)
    _check(LIB.ccl_device_error_flag(ctypes.byref(flag), 1 if clear else 0), "ccl_device_error_flag")
    return int(flag.value)


def ccl_stream_check(stream=None) -> None:
    """Synchronize the stream; raise CclError(CCL_ERR_TIMEOUT) if a bounded
    device-side wait ran out since the last check."""
    _check(LIB.ccl_stream_check(_stream(stream, torch.device("cuda", torch.cuda.current_device()))),
           "ccl_stream_check")


def ccl_selftest_bounded_wait(stream=None) -> None:
    """Enqueue a kernel whose bounded wait runs out by construction (self-test
    of the failure path; nothing faults)."""
    _check(LIB.ccl_selftest_bounded_wait(_stream(stream, torch.device("cuda", torch.cuda.current_device()))),
           "ccl_selftest_bounded_wait")


def ccl_chunk_bounds(p: int, n: int, c: int) -> tuple[int, int]:
    """(offset, length) of chunk c of an n-element buffer cut into p chunks."""
    off, ln = ctypes.c_size_t(), ctypes.c_size_t()
    _check(LIB.ccl_chunk_bounds(p, n, c, ctypes.byref(off), ctypes.byref(ln)), "ccl_chunk_bounds")
    return off.value, ln.value


FOLD_KINDS = {"allreduce": 0, "reduce_scatter": 1, "bucket": 2, "reduce": 3}  # ccl_fold_kind_t


def ccl_fold_plan(p: int, n: int, dtype: str = "f32", op: str = "sum", kind: str = "allreduce",
                  aligned: bool = True, sm_count: int = 0) -> tuple[int, int]:
    """(ranks per load batch, vectors per thread) of the fused fold kernel a
    call of the given kind with p ranks x n elements takes; (0, 0) is the
    general kernel.  sm_count <= 0 asks the current device."""
    codes = {"f32": CCL_F32, "bf16": CCL_BF16, "i32": CCL_I32}
    if dtype not in codes:
        raise ValueError(f"dtype must be one of {sorted(codes)}")
    if kind not in FOLD_KINDS:
        raise ValueError(f"kind must be one of {sorted(FOLD_KINDS)}")
    b, v = ctypes.c_int(), ctypes.c_int()
    _check(LIB.ccl_fold_plan(FOLD_KINDS[kind], codes[dtype], _op_code(op), p, n, 1 if aligned else 0,
                             sm_count, ctypes.byref(b), ctypes.byref(v)), "ccl_fold_plan")
    return b.value, v.value


def ccl_plan_buckets(numel, elem_bytes: int = 4, cap_bytes: int = 25 * 1024 * 1024):
    """DDP bucket plan: gradients (element counts, in ready order) -> buckets.

    Returns (bucket_of, offset, bucket_numel): per gradient its bucket and
    element offset in it, and per bucket its element count.
    """
    numel = [int(m) for m in numel]
    count = len(numel)
    arr = (ctypes.c_size_t * max(1, count))(*numel)
    bucket_of = (ctypes.c_uint32 * max(1, count))()
    offset = (ctypes.c_size_t * max(1, count))()
    bucket_numel = (ctypes.c_size_t * max(1, count))()
    nb = ctypes.c_size_t()
    _check(LIB.ccl_plan_buckets(arr, count, elem_bytes, cap_bytes, bucket_of, offset, bucket_numel,
                                ctypes.byref(nb)), "ccl_plan_buckets")
    return list(bucket_of)[:count], list(offset)[:count], list(bucket_numel)[:nb.value]


# ------------------------------------------------------------- fused calls
def ccl_allreduce(send, recv, op: str = "sum", stream=None) -> None:
    """Every recv[r] gets the ring-ordered reduction of send[0..p-1] (in place allowed)."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_allreduce(_ptr_array([t.data_ptr() for t in send]),
                             _ptr_array([t.data_ptr() for t in recv]), p, n,
                             _dtype_code(send[0]), _op_code(op), _stream(stream, send[0].device)),
           "ccl_allreduce")


def ccl_allreduce_schedule(send, recv, schedule: str = "ring", op: str = "sum", stream=None) -> None:
    """All-reduce with the bits another schedule (recursive_doubling,
    rabenseifner, binomial_tree, naive, ring) would give."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    if schedule not in SCHEDULES:
        raise ValueError(f"schedule must be one of {sorted(SCHEDULES)}")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_allreduce_schedule(_ptr_array([t.data_ptr() for t in send]),
                                      _ptr_array([t.data_ptr() for t in recv]), p, n,
                                      _dtype_code(send[0]), _op_code(op), SCHEDULES[schedule],
                                      _stream(stream, send[0].device)),
           "ccl_allreduce_schedule")


def ccl_allreduce_hierarchical(send, recv, group: int, op: str = "sum", stream=None) -> None:
    """All-reduce with the bits of the two-level ring: groups of `group`
    consecutive ranks, a ring inside every group, then a ring over the groups."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_allreduce_hierarchical(_ptr_array([t.data_ptr() for t in send]),
                                          _ptr_array([t.data_ptr() for t in recv]), p, int(group), n,
                                          _dtype_code(send[0]), _op_code(op),
                                          _stream(stream, send[0].device)),
           "ccl_allreduce_hierarchical")


def ccl_allreduce_bf16_wire(send, recv, stream=None) -> None:
    """bf16 ring all-reduce whose partials are rounded to bf16 at every hop."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if send[0].dtype != torch.bfloat16 or len(recv) != p or recv[0].dtype != torch.bfloat16:
        raise ValueError("send and recv must hold p bf16 buffers")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_allreduce_bf16_wire(_ptr_array([t.data_ptr() for t in send]),
                                       _ptr_array([t.data_ptr() for t in recv]), p, n,
                                       _stream(stream, send[0].device)), "ccl_allreduce_bf16_wire")


def ccl_reduce_scatter_bf16_wire(send, recv, stream=None) -> None:
    """bf16 ring reduce-scatter whose partials are rounded to bf16 at every hop."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if send[0].dtype != torch.bfloat16 or len(recv) != p or recv[0].dtype != torch.bfloat16:
        raise ValueError("send and recv must hold p bf16 buffers")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, _chunk_lengths(p, n), "recv")
    _check(LIB.ccl_reduce_scatter_bf16_wire(_ptr_array([t.data_ptr() for t in send]),
                                            _ptr_array([t.data_ptr() for t in recv]), p, n,
                                            _stream(stream, send[0].device)), "ccl_reduce_scatter_bf16_wire")


def ccl_reduce_scatter(send, recv, op: str = "sum", stream=None) -> None:
    """recv[k] (len(k) elements) gets chunk k of the ring-ordered reduction."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, _chunk_lengths(p, n), "recv")
    _check(LIB.ccl_reduce_scatter(_ptr_array([t.data_ptr() for t in send]),
                                  _ptr_array([t.data_ptr() for t in recv]), p, n,
                                  _dtype_code(send[0]), _op_code(op), _stream(stream, send[0].device)),
           "ccl_reduce_scatter")


def ccl_all_gather(send, recv, stream=None) -> None:
    """send[k] is block k (len(k) elements); every recv[r] gets the concatenation."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p = len(send)
    n = sum(t.numel() for t in send)
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, _chunk_lengths(p, n), "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_all_gather(_ptr_array([t.data_ptr() for t in send]),
                              _ptr_array([t.data_ptr() for t in recv]), p, n,
                              _dtype_code(send[0]), _stream(stream, send[0].device)),
           "ccl_all_gather")


def _one(t: torch.Tensor, name: str) -> torch.Tensor:
    return _tensors([t], name)[0]


def ccl_broadcast(send, recv, root: int = 0, stream=None) -> None:
    """Every recv[r] gets a copy of the root's buffer `send`."""
    send, recv = _one(send, "send"), _tensors(recv, "recv")
    p, n = len(recv), send.numel()
    if recv[0].dtype != send.dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_broadcast(send.data_ptr(), _ptr_array([t.data_ptr() for t in recv]), p, n,
                             _dtype_code(send), root, _stream(stream, send.device)), "ccl_broadcast")


def ccl_reduce(send, recv, op: str = "sum", root: int = 0, stream=None) -> None:
    """The root's buffer `recv` gets the ring-ordered reduction of send[0..p-1]."""
    send, recv = _tensors(send, "send"), _one(recv, "recv")
    p, n = len(send), send[0].numel()
    if recv.dtype != send[0].dtype:
        raise ValueError("recv must have the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check([recv], [n], "recv")
    _check(LIB.ccl_reduce(_ptr_array([t.data_ptr() for t in send]), recv.data_ptr(), p, n,
                          _dtype_code(recv), _op_code(op), root, _stream(stream, recv.device)),
           "ccl_reduce")


def ccl_scatter(send, recv, root: int = 0, stream=None) -> None:
    """recv[k] gets chunk k of the root's buffer `send`."""
    send, recv = _one(send, "send"), _tensors(recv, "recv")
    p, n = len(recv), send.numel()
    if recv[0].dtype != send.dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(recv, _chunk_lengths(p, n), "recv")
    _check(LIB.ccl_scatter(send.data_ptr(), _ptr_array([t.data_ptr() for t in recv]), p, n,
                           _dtype_code(send), root, _stream(stream, send.device)), "ccl_scatter")


def ccl_gather(send, recv, root: int = 0, stream=None) -> None:
    """The root's buffer `recv` gets the concatenation of send[0..p-1] (chunk rule)."""
    send, recv = _tensors(send, "send"), _one(recv, "recv")
    p, n = len(send), recv.numel()
    if recv.dtype != send[0].dtype:
        raise ValueError("recv must have the send dtype")
    _numel_check(send, _chunk_lengths(p, n), "send")
    _check(LIB.ccl_gather(_ptr_array([t.data_ptr() for t in send]), recv.data_ptr(), p, n,
                          _dtype_code(recv), root, _stream(stream, recv.device)), "ccl_gather")


def ccl_bucket_allreduce_scale_cast(grads, out_bf16, scale: float | None = None, stream=None) -> None:
    """out_bf16[r] = bf16(ring_sum(grads) * scale); scale defaults to 1/p."""
    grads, out = _tensors(grads, "grads"), _tensors(out_bf16, "out_bf16")
    p, n = len(grads), grads[0].numel()
    if grads[0].dtype != torch.float32 or out[0].dtype != torch.bfloat16 or len(out) != p:
        raise ValueError("grads must be p float32 buffers and out_bf16 p bfloat16 buffers")
    _numel_check(grads, [n] * p, "grads")
    _numel_check(out, [n] * p, "out_bf16")
    s = float(1.0 / p) if scale is None else float(scale)
    _check(LIB.ccl_bucket_allreduce_scale_cast(_ptr_array([t.data_ptr() for t in grads]),
                                               _ptr_array([t.data_ptr() for t in out]), p, n, s,
                                               _stream(stream, grads[0].device)),
           "ccl_bucket_allreduce_scale_cast")


def ccl_all_to_all(send, recv, stream=None) -> None:
    """Block transpose: recv[j] = block j of every send[i] (chunk rule), in
    source order."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [p * ln for ln in _chunk_lengths(p, n)], "recv")
    _check(LIB.ccl_all_to_all(_ptr_array([t.data_ptr() for t in send]), _ptr_array([t.data_ptr() for t in recv]),
                              p, n, _dtype_code(send[0]), _stream(stream, send[0].device)), "ccl_all_to_all")


def ccl_all_to_allv(send, counts, recv, row_elems: int, stream=None) -> None:
    """MoE dispatch/combine: counts[s][d] rows of row_elems go from send[s] to recv[d]."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p = len(send)
    rows = [[int(counts[s][d]) for d in range(p)] for s in range(p)]
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [sum(rows[s]) * row_elems for s in range(p)], "send")
    _numel_check(recv, [sum(rows[s][d] for s in range(p)) * row_elems for d in range(p)], "recv")
    flat = (ctypes.c_size_t * (p * p))(*[rows[s][d] for s in range(p) for d in range(p)])
    _check(LIB.ccl_all_to_allv(_ptr_array([t.data_ptr() for t in send]), flat,
                               _ptr_array([t.data_ptr() for t in recv]), p, row_elems,
                               _dtype_code(send[0]), _stream(stream, send[0].device)),
           "ccl_all_to_allv")


A2A_FORMS = ("small", "plain", "table32", "table64")  # ccl_a2a_form_t


def _addresses(bufs) -> list[int]:
    return [b if isinstance(b, int) else b.data_ptr() for b in bufs]


def _plan_tuple(pl) -> tuple:
    return (A2A_FORMS[pl.form], bool(pl.shift), bool(pl.stage), pl.launches, pl.tile_bytes)


def ccl_all_to_all_plan(send, recv, n: int, dtype: str = "f32", sm_count: int = 0) -> tuple:
    """(form, shift, stage, launches, tile_bytes) of the kernel ccl_all_to_all
    launches for these buffers (tensors, or their addresses as ints: only the
    addresses matter) with n elements per rank; sm_count <= 0 asks the
    current device."""
    codes = {"f32": CCL_F32, "bf16": CCL_BF16, "i32": CCL_I32}
    pl = A2APlan()
    _check(LIB.ccl_all_to_all_plan(_ptr_array(_addresses(send)), _ptr_array(_addresses(recv)), len(send), n,
                                   codes[dtype], sm_count, ctypes.byref(pl)), "ccl_all_to_all_plan")
    return _plan_tuple(pl)


def ccl_all_to_allv_plan(send, counts, recv, row_elems: int, dtype: str = "f32", sm_count: int = 0) -> tuple:
    """(form, shift, stage, launches, tile_bytes) of the kernel ccl_all_to_allv
    launches for these buffers (tensors or addresses) and counts."""
    codes = {"f32": CCL_F32, "bf16": CCL_BF16, "i32": CCL_I32}
    p = len(send)
    flat = (ctypes.c_size_t * (p * p))(*[int(counts[s][d]) for s in range(p) for d in range(p)])
    pl = A2APlan()
    _check(LIB.ccl_all_to_allv_plan(_ptr_array(_addresses(send)), flat, _ptr_array(_addresses(recv)), p,
                                    row_elems, codes[dtype], sm_count, ctypes.byref(pl)), "ccl_all_to_allv_plan")
    return _plan_tuple(pl)


# ------------------------------------------------------- literal ring engine
def ccl_ring_literal_workspace_bytes(kind: int, p: int, n: int, dtype: torch.dtype) -> int:
    return LIB.ccl_ring_literal_workspace_bytes(kind, p, n, _DTYPES[dtype])


def _workspace(kind, p, n, t, workspace):
    need = ccl_ring_literal_workspace_bytes(kind, p, n, t.dtype)
    if need == 0:
        return None, 0
    if workspace is None:  # caller-owned scratch, allocated by torch
        workspace = torch.empty(need, dtype=torch.uint8, device=t.device)
    return workspace, workspace.numel() * workspace.element_size()


def ccl_ring_allreduce_literal(send, recv, op: str = "sum", workspace=None, stream=None) -> list[int]:
    """The 2(p-1)-step ring, one launch per step; returns bytes sent per rank."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    ws, ws_bytes = _workspace(CCL_KIND_ALLREDUCE, p, n, send[0], workspace)
    sent = (ctypes.c_uint64 * p)()
    _check(LIB.ccl_ring_allreduce_literal(_ptr_array([t.data_ptr() for t in send]),
                                          _ptr_array([t.data_ptr() for t in recv]), p, n,
                                          _dtype_code(send[0]), _op_code(op), sent,
                                          None if ws is None else ws.data_ptr(), ws_bytes,
                                          _stream(stream, send[0].device)),
           "ccl_ring_allreduce_literal")
    return list(sent)


def ccl_ring_reduce_scatter_literal(send, recv, op: str = "sum", workspace=None, stream=None) -> list[int]:
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, _chunk_lengths(p, n), "recv")
    ws, ws_bytes = _workspace(CCL_KIND_REDUCE_SCATTER, p, n, send[0], workspace)
    sent = (ctypes.c_uint64 * p)()
    _check(LIB.ccl_ring_reduce_scatter_literal(_ptr_array([t.data_ptr() for t in send]),
                                               _ptr_array([t.data_ptr() for t in recv]), p, n,
                                               _dtype_code(send[0]), _op_code(op), sent,
                                               None if ws is None else ws.data_ptr(), ws_bytes,
                                               _stream(stream, send[0].device)),
           "ccl_ring_reduce_scatter_literal")
    return list(sent)


def ccl_ring_all_gather_literal(send, recv, stream=None) -> list[int]:
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p = len(send)
    n = sum(t.numel() for t in send)
    _numel_check(send, _chunk_lengths(p, n), "send")
    _numel_check(recv, [n] * p, "recv")
    sent = (ctypes.c_uint64 * p)()
    _check(LIB.ccl_ring_all_gather_literal(_ptr_array([t.data_ptr() for t in send]),
                                           _ptr_array([t.data_ptr() for t in recv]), p, n,
                                           _dtype_code(send[0]), sent,
                                           _stream(stream, send[0].device)),
           "ccl_ring_all_gather_literal")
    return list(sent)


# ---------------------------------------------- allocation-free reduce-scatter
def ccl_ring_reduce_scatter_literal_noalloc(send, recv, op: str = "sum", stream=None) -> list[int]:
    """ccl_ring_reduce_scatter_literal without a workspace argument.

    For callers that cannot allocate device memory (for instance code running
    inside an allocator callback, or under a host that owns all device
    memory): the library's built-in static scratch holds the working buffers,
    so p*n must not exceed 8,388,608 elements.  The first call on a device
    looks up the scratch address, so make it before any stream capture; calls
    that overlap on the GPU share the scratch and must be serialised.
    """
    fn = LIB.ccl_ring_reduce_scatter_literal_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
                   ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint64),
                   ctypes.c_void_p]
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p, n = len(send), send[0].numel()
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, _chunk_lengths(p, n), "recv")
    sent = (ctypes.c_uint64 * p)()
    _check(fn(_ptr_array([t.data_ptr() for t in send]), _ptr_array([t.data_ptr() for t in recv]),
              p, n, _dtype_code(send[0]), _op_code(op), sent, _stream(stream, send[0].device)),
           "ccl_ring_reduce_scatter_literal_noalloc")
    return list(sent)


# ------------------------------------------------------------ MoE routing
def _ptrs_or_null(ts):
    return None if ts is None else _ptr_array([t.data_ptr() for t in ts])


def ccl_moe_route(expert_ids, num_experts: int, counts, slots, stream=None) -> None:
    """expert_ids[s]: (tokens, k) int32 CUDA tensors -> counts (p*p int64) and
    slots[s] ((tokens, k) int32; -1 where the id is out of range)."""
    ids = _tensors(expert_ids, "expert_ids")
    p = len(ids)
    tokens, k = (ids[0].shape[0], ids[0].shape[1]) if ids[0].dim() == 2 else (ids[0].numel(), 1)
    if ids[0].dtype != torch.int32 or counts.dtype != torch.int64 or counts.numel() != p * p:
        raise ValueError("expert_ids must be int32 and counts p*p int64")
    slots = _tensors(slots, "slots")
    _numel_check(ids, [tokens * k] * p, "expert_ids")
    _numel_check(slots, [tokens * k] * p, "slots")
    _check(LIB.ccl_moe_route(_ptr_array([t.data_ptr() for t in ids]), p, tokens, k, num_experts,
                             counts.data_ptr(), _ptr_array([t.data_ptr() for t in slots]),
                             _stream(stream, ids[0].device)), "ccl_moe_route")


def ccl_moe_dispatch(x, expert_ids, counts, slots, num_experts: int, recv, recv_scales=None,
                     recv_expert=None, fp8: bool = False, stream=None) -> None:
    """Scatter each token row to the ranks of its k experts (bf16, or FP8 with
    per-128 block scales when fp8=True).  recv[d] sized from counts."""
    x, ids, slots, recv = (_tensors(x, "x"), _tensors(expert_ids, "expert_ids"),
                           _tensors(slots, "slots"), list(recv))
    p = len(x)
    tokens, hidden = x[0].shape
    k = ids[0].numel() // tokens
    rows = (ctypes.c_size_t * p)(*[int(t.shape[0]) if t.numel() else 0 for t in recv])
    _check(LIB.ccl_moe_dispatch(_ptr_array([t.data_ptr() for t in x]),
                                _ptr_array([t.data_ptr() for t in ids]), counts.data_ptr(),
                                _ptr_array([t.data_ptr() for t in slots]), p, tokens, k, num_experts,
                                hidden, 1 if fp8 else 0, _ptr_array([t.data_ptr() for t in recv]), rows,
                                _ptrs_or_null(recv_scales), _ptrs_or_null(recv_expert),
                                _stream(stream, x[0].device)), "ccl_moe_dispatch")


def ccl_moe_combine(y, expert_ids, weights, counts, slots, num_experts: int, out, stream=None) -> None:
    """out[s][t] = bf16(sum_j weights[s][t, j] * y[row of (s, t, j)])."""
    ids, w, slots, out = (_tensors(expert_ids, "expert_ids"), _tensors(weights, "weights"),
                          _tensors(slots, "slots"), _tensors(out, "out"))
    y = list(y)
    p = len(out)
    tokens, hidden = out[0].shape
    k = ids[0].numel() // tokens
    rows = (ctypes.c_size_t * p)(*[int(t.shape[0]) if t.numel() else 0 for t in y])
    _check(LIB.ccl_moe_combine(_ptr_array([t.data_ptr() for t in y]), rows,
                               _ptr_array([t.data_ptr() for t in ids]),
                               _ptr_array([t.data_ptr() for t in w]), counts.data_ptr(),
                               _ptr_array([t.data_ptr() for t in slots]), p, tokens, k, num_experts,
                               hidden, _ptr_array([t.data_ptr() for t in out]),
                               _stream(stream, out[0].device)), "ccl_moe_combine")


# ------------------------------------------------ Ulysses head <-> sequence
def ccl_all_to_all_heads(send, recv, seq_per_rank: int, heads: int, head_dim: int,
                         inverse: bool = False, stream=None) -> None:
    """Forward: send[r] = [seq_per_rank, heads, head_dim] sequence shard ->
    recv[r] = [p*seq_per_rank, heads/p, head_dim] head group; inverse: back."""
    send, recv = _tensors(send, "send"), _tensors(recv, "recv")
    p = len(send)
    n = seq_per_rank * heads * head_dim
    if len(recv) != p or recv[0].dtype != send[0].dtype:
        raise ValueError("recv must hold p buffers of the send dtype")
    _numel_check(send, [n] * p, "send")
    _numel_check(recv, [n] * p, "recv")
    _check(LIB.ccl_all_to_all_heads(_ptr_array([t.data_ptr() for t in send]),
                                    _ptr_array([t.data_ptr() for t in recv]), p, seq_per_rank, heads,
                                    head_dim, _dtype_code(send[0]), 1 if inverse else 0,
                                    _stream(stream, send[0].device)), "ccl_all_to_all_heads")
