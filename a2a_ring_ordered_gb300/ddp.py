"""DDP-style bucketed gradient all-reduce over p virtual ranks on one GPU.

"dist_train", Communication-Computation Overlap: backprop runs from the last
layer to the first; DDP cuts the gradients into buckets of bucket_cap_mb
(25 MB) in the order backprop produces them, and as soon as every gradient of
a bucket is ready it all-reduces that bucket while backprop continues with
earlier layers.

Layout instead of copies: each rank's gradients live in flat fp32 bucket
buffers and every parameter's gradient is a view into its bucket, so the
fused bucket kernel (ring-ordered sum, 1/p average, bf16 cast) runs directly
on the buckets -- there is no copy-in or copy-out pass.  The bf16 results
land in flat output buckets, again with per-parameter views.

All arithmetic runs in libccl's kernels; this module only plans buckets (in
the library), allocates buffers with torch and orders launches with CUDA
events.
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import ccl

DEFAULT_CAP_BYTES = 25 * 1024 * 1024  # bucket_cap_mb = 25


class GradBuckets:
    """Flat fp32 gradient buckets and bf16 output buckets for p virtual ranks.

    shapes       parameter shapes in registration order.
    ready_order  parameter indices in the order backprop produces their
                 gradients; default: the reverse of registration order (the
                 last layer's gradients are ready first).
    """

    def __init__(self, shapes: Sequence[Sequence[int]], p: int, device,
                 cap_bytes: int = DEFAULT_CAP_BYTES, ready_order: Sequence[int] | None = None):
        self.p = p
        self.device = torch.device(device)
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        numel = [int(torch.Size(s).numel()) for s in self.shapes]
        self.ready_order = list(ready_order) if ready_order is not None \
            else list(reversed(range(len(shapes))))
        if sorted(self.ready_order) != list(range(len(shapes))):
            raise ValueError("ready_order must be a permutation of the parameter indices")
        bucket_of, offset, bucket_numel = ccl.ccl_plan_buckets(
            [numel[i] for i in self.ready_order], 4, cap_bytes)
        self.bucket_numel = bucket_numel
        self.where: dict[int, tuple[int, int, int]] = {}
        self.members: list[list[int]] = [[] for _ in bucket_numel]
        for k, param in enumerate(self.ready_order):
            self.where[param] = (bucket_of[k], offset[k], numel[param])
            self.members[bucket_of[k]].append(param)
        self.grads = [[torch.zeros(m, dtype=torch.float32, device=self.device) for _ in range(p)]
                      for m in bucket_numel]
        self.out = [[torch.empty(m, dtype=torch.bfloat16, device=self.device) for _ in range(p)]
                    for m in bucket_numel]
        self.scale = float(torch.tensor(1.0 / p, dtype=torch.float32))

    @property
    def num_buckets(self) -> int:
        return len(self.bucket_numel)

    def grad(self, rank: int, param: int) -> torch.Tensor:
        """Rank `rank`'s fp32 gradient of parameter `param` (a view into its bucket)."""
        b, off, m = self.where[param]
        return self.grads[b][rank][off:off + m].view(self.shapes[param])

    def averaged(self, rank: int, param: int) -> torch.Tensor:
        """Rank `rank`'s bf16 averaged gradient of `param` (a view into its output bucket)."""
        b, off, m = self.where[param]
        return self.out[b][rank][off:off + m].view(self.shapes[param])

    def reduce_bucket(self, b: int, stream=None) -> None:
        """Ring-ordered all-reduce of bucket b over the p ranks, times 1/p, to bf16."""
        ccl.ccl_bucket_allreduce_scale_cast(self.grads[b], self.out[b], scale=self.scale,
                                            stream=stream)


class OverlappedReducer:
    """Fires each bucket's all-reduce on a communication stream as soon as the
    last of its gradients is marked ready on the producer stream."""

    def __init__(self, buckets: GradBuckets, comm_stream: torch.cuda.Stream | None = None):
        self.buckets = buckets
        self.comm = comm_stream or torch.cuda.Stream(buckets.device)
        self.pending: list[int] = []
        self.fired: list[int] = []
        self.start_step()

    def start_step(self) -> None:
        self.pending = [len(m) for m in self.buckets.members]
        self.fired = []

    def mark_ready(self, param: int, producer_stream: torch.cuda.Stream | None = None) -> None:
        """All p ranks' gradients of `param` have been enqueued on the producer stream."""
        b = self.buckets.where[param][0]
        if self.pending[b] <= 0:
            raise RuntimeError(f"parameter {param} marked ready twice in one step")
        self.pending[b] -= 1
        if self.pending[b] == 0:
            producer = producer_stream or torch.cuda.current_stream(self.buckets.device)
            ready = torch.cuda.Event()
            ready.record(producer)
            self.comm.wait_event(ready)
            self.buckets.reduce_bucket(b, stream=self.comm)
            self.fired.append(b)

    def finish(self, stream: torch.cuda.Stream | None = None) -> None:
        """Make `stream` (default: current) wait for every fired bucket."""
        if any(n != 0 for n in self.pending):
            raise RuntimeError("finish() before every gradient was marked ready")
        (stream or torch.cuda.current_stream(self.buckets.device)).wait_stream(self.comm)
