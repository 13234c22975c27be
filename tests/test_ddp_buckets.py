"""DDP bucketing front end: the bucket plan (CPU) and the bucketed,
overlapped reducer against the oracle (GPU)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads

MiB = 1 << 20


@pytest.fixture(scope="module")
def ccl():
    from a2a_ring_ordered_gb300 import build

    build.build()
    from a2a_ring_ordered_gb300 import ccl as mod

    return mod


def plan_by_hand(numel, elem_bytes, cap_bytes):
    """The rule written out: fill while the bucket stays within the cap."""
    cap = cap_bytes // elem_bytes
    buckets, cur = [], []
    for i, m in enumerate(numel):
        if cur and (sum(numel[j] for j in cur) + m > cap):
            buckets.append(cur)
            cur = []
        cur.append(i)
    if cur or not numel:
        buckets.append(cur)
    return buckets if numel else []


def test_plan_25mb_cap_closed_forms(ccl):
    cap = 25 * MiB
    # 8 gradients of exactly a quarter bucket: 4 per bucket, 2 buckets
    q = cap // 4 // 4
    b, off, sizes = ccl.ccl_plan_buckets([q] * 8, 4, cap)
    assert b == [0, 0, 0, 0, 1, 1, 1, 1] and off == [0, q, 2 * q, 3 * q] * 2
    assert sizes == [4 * q, 4 * q]
    # an oversize gradient gets a bucket of its own, and the next one starts fresh
    b, off, sizes = ccl.ccl_plan_buckets([10, 7 * MiB, 5], 4, cap)
    assert b == [0, 1, 2] and sizes == [10, 7 * MiB, 5]
    # the DDP bench bucket: 6,553,600 fp32 = exactly 25 MiB fits one bucket
    b, _, sizes = ccl.ccl_plan_buckets([6_553_600], 4, cap)
    assert b == [0] and sizes == [6_553_600]
    assert ccl.ccl_plan_buckets([], 4, cap) == ([], [], [])


@pytest.mark.parametrize("seed", range(6))
def test_plan_matches_the_rule_by_hand(ccl, seed):
    rng = np.random.default_rng(seed)
    numel = [int(x) for x in rng.choice([0, 1, 3, 1000, 50_000, 300_000, 2_000_000], size=60)]
    cap = int(rng.choice([4 * 1024, 1 * MiB, 4 * MiB]))
    b, off, sizes = ccl.ccl_plan_buckets(numel, 4, cap)
    want = plan_by_hand(numel, 4, cap)
    assert len(sizes) == len(want)
    for k, members in enumerate(want):
        acc = 0
        for i in members:
            assert b[i] == k and off[i] == acc
            acc += numel[i]
        assert sizes[k] == acc
        assert acc * 4 <= cap or len(members) == 1


def test_plan_rejects_bad_arguments(ccl):
    with pytest.raises(ccl.CclError):
        ccl.ccl_plan_buckets([1, 2], 0, 100)
    with pytest.raises(ccl.CclError):
        ccl.ccl_plan_buckets([1, 2], 4, 2)


TRANSFORMER_D = 512


def transformer_shapes(layers=6, d=TRANSFORMER_D, vocab=5003):
    shapes = [(vocab, d)]
    for _ in range(layers):
        shapes += [(3 * d, d), (3 * d,), (d, d), (d,), (d,), (d,), (4 * d, d), (4 * d,),
                   (d, 4 * d), (d,), (d,), (d,)]
    shapes += [(d,), (d,)]
    return shapes


@pytest.mark.gpu
def test_overlapped_bucket_reducer_matches_oracle(ccl):
    from a2a_ring_ordered_gb300.ddp import GradBuckets, OverlappedReducer
    from oracle import ring

    p = 4
    shapes = transformer_shapes()
    cap = 1 * MiB  # small cap: many buckets for this small model
    gb = GradBuckets(shapes, p, "cuda", cap_bytes=cap)
    assert gb.num_buckets > 5
    red = OverlappedReducer(gb)
    producer = torch.cuda.Stream()
    host = {}
    rng = np.random.default_rng(0)
    with torch.cuda.stream(producer):
        for param in gb.ready_order:  # a synthetic backward: last layer first
            m = int(np.prod(shapes[param]))
            for r in range(p):
                g = workloads.normal(1, m, 1e-3, seed=int(rng.integers(1 << 30)))[0]
                host[(r, param)] = g
                gb.grad(r, param).copy_(torch.from_numpy(g).view(shapes[param]), non_blocking=False)
            red.mark_ready(param, producer)
    red.finish()
    torch.cuda.synchronize()
    assert sorted(red.fired) == list(range(gb.num_buckets))
    for b, members in enumerate(gb.members):
        flat = [np.concatenate([host[(r, q)] for q in members]) for r in range(p)]
        want = ring.bucket_allreduce_scale_cast(flat, gb.scale)
        for r in range(p):
            got = gb.out[b][r].cpu().view(torch.int16).numpy().view(np.uint16)
            np.testing.assert_array_equal(got, want[r], err_msg=f"bucket {b} rank {r}")
    # per-parameter views of the averaged gradients
    q = members[0]
    off = 0
    assert gb.averaged(1, q).shape == tuple(shapes[q])
