"""GPU parity: every entry point of libccl against the CPU oracle.

Small and medium cases compare every element with the literal ring oracle;
the full-size workloads compare sampled outputs with the pointwise oracle and
check size-independent properties on the device.  Floating point results are
bit-exact (fp32 ring order; bf16 within the stated 1-ulp contract, asserted
exact); copies and integer sums are bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import (GUARD, Guarded, assert_bf16_close, assert_equal, ccl, sample_indices,
                      to_dev, to_host)
from oracle import collectives, pointwise, ring

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def make_inputs(dtype, p, n, seed):
    if dtype == "i32":
        return workloads.integer_valued(p, n, seed, lo=-2**31, hi=2**31 - 1, dtype="i32")
    return workloads.normal(p, n, 1.0, seed, dtype=dtype)


def guarded_outputs(p, sizes, dtype, offset=GUARD):
    return [Guarded(s, dtype, offset) for s in sizes]


# --------------------------------------------------------- worked example
def test_worked_example_on_gpu(lib, worked_example):
    g = worked_example
    x = workloads.worked_example(4)
    send = [to_dev(v, "f32") for v in x]
    recv = [torch.empty(4, device="cuda") for _ in range(4)]
    lib.ccl_allreduce(send, recv)
    for r in recv:
        assert to_host(r).tolist() == g["allreduce"]
    shards = [torch.empty(1, device="cuda") for _ in range(4)]
    lib.ccl_reduce_scatter(send, shards)
    for k in range(4):
        assert to_host(shards[k]).tolist() == g[f"reduce_scatter {k}"]
    contrib = [to_dev(x[d][d:d + 1].copy(), "f32") for d in range(4)]
    out = [torch.empty(4, device="cuda") for _ in range(4)]
    lib.ccl_all_gather(contrib, out)
    for o in out:
        assert to_host(o).tolist() == g["all_gather"]
    # all-to-all: one element per block, counts all 1
    recv_a2a = [torch.empty(4, device="cuda") for _ in range(4)]
    lib.ccl_all_to_allv(send, np.ones((4, 4), dtype=np.int64), recv_a2a, 1)
    for j in range(4):
        assert to_host(recv_a2a[j]).tolist() == g[f"all_to_all {j}"]


# ------------------------------------------------ p=4 fp32 case, full size
def test_p4_fp32_million_all_primitives(lib):
    p, n = 4, 1 << 20
    x = workloads.normal(p, n, 1.0, seed=0)
    send = [to_dev(v, "f32") for v in x]
    want_ar, _, _ = ring.ring_allreduce(x, "f32", "sum")
    recv = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_allreduce(send, recv)
    for r in range(p):
        assert_equal(to_host(recv[r]), want_ar[r], "f32", f"AR rank {r}")
    want_rs, _ = ring.ring_reduce_scatter(x, "f32", "sum")
    shards = [torch.empty(n // p, device="cuda") for _ in range(p)]
    lib.ccl_reduce_scatter(send, shards)
    for k in range(p):
        assert_equal(to_host(shards[k]), want_rs[k], "f32", f"RS rank {k}")
    out = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_all_gather(shards, out)
    for r in range(p):
        assert_equal(to_host(out[r]), want_ar[r], "f32", f"AG(RS) rank {r}")
    want_a2a = collectives.all_to_all(x)
    counts = np.full((p, p), n // p, dtype=np.int64)
    recv_a2a = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_all_to_allv(send, counts, recv_a2a, 1)
    for r in range(p):
        assert_equal(to_host(recv_a2a[r]), want_a2a[r], "f32", f"A2A rank {r}")


# ------------------------------------------------- dtype x op x shape sweep
SHAPES = [(1, 1000), (2, 4099), (3, 1001), (4, 13), (5, 3), (6, 13), (8, 70001),
          (16, 65543), (72, 10000), (128, 1000)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("p,n", SHAPES)
def test_allreduce_and_reduce_scatter_match_oracle(lib, dtype, op, p, n):
    x = make_inputs(dtype, p, n, seed=p * 1000 + n)
    send = [to_dev(v, dtype) for v in x]
    want, _, _ = ring.ring_allreduce(x, dtype, op)
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_allreduce(send, [o.view for o in outs], op=op)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"AR {dtype} {op} p={p} n={n} rank {r}")
        assert outs[r].guards_intact()
    want_rs, _ = ring.ring_reduce_scatter(x, dtype, op)
    sizes = [ln for _, ln in ring.chunk_bounds(p, n)]
    shards = guarded_outputs(p, sizes, dtype)
    lib.ccl_reduce_scatter(send, [s.view for s in shards], op=op)
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], dtype, f"RS rank {k}")
        assert shards[k].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", SHAPES)
def test_all_gather_matches_oracle(lib, dtype, p, n):
    x = make_inputs(dtype, p, n, seed=7 + p + n)
    bounds = ring.chunk_bounds(p, n)
    blocks = [x[k][off:off + ln].copy() for k, (off, ln) in enumerate(bounds)]
    want, _ = ring.ring_all_gather(blocks, dtype)
    send = [to_dev(b, dtype) for b in blocks]
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_all_gather(send, [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"AG rank {r}")
        assert outs[r].guards_intact()


# vectors per thread of the all-gather (the host picks them by grid size
# and p): mid-size calls take 1 (grids up to 20 CTAs per SM, or p >= 8) or 2,
# larger ones 8, or 1 from p = 8 on when blocks are off the output vectors;
# blocks on the 16-byte grid or off it (p = 72, p = 8, p = 3)
AG_SIZE_CLASSES = [("f32", 2, 2 * 1048576), ("bf16", 8, 8 * 262144 + 8), ("bf16", 72, 72 * 41000 + 5),
                   ("f32", 2, 4 * 1048576), ("bf16", 3, 3 * 4194304 + 1), ("f32", 2, 16 * 1048576 + 4),
                   ("f32", 3, 3 * 3400000 + 1), ("f32", 8, 8 * 2097152 + 3), ("bf16", 16, 16 * 1048576 + 16)]


@pytest.mark.parametrize("dtype,p,n", AG_SIZE_CLASSES)
def test_all_gather_size_classes_match_oracle(lib, dtype, p, n):
    """Every element of every output against the literal ring all-gather,
    at sizes that select 1, 2 and 8 vectors per thread, aligned and
    realigned blocks, guard bands."""
    test_all_gather_matches_oracle(lib, dtype, p, n)


# the reduce-scatter with 9..32 ranks and chunks of at least 128 KiB loads 8
# ranks per batch (the general kernel otherwise 16): chunks off the vector
# grid (p = 9, 32) and on it (p = 16), every op, and the boundaries of the
# rule (p = 8 and 33 keep their kernels)
RS_BATCH8 = [(dt, op, 9, 9 * 40000 + 5) for dt in ("f32", "bf16", "i32") for op in ("sum", "max", "min")]
RS_BATCH8 += [(dt, "sum", p, n) for dt in ("f32", "bf16", "i32")
              for p, n in ((16, 16 * 65536), (32, 32 * 40000 + 17), (33, 33 * 40000 + 1))]


@pytest.mark.parametrize("dtype,op,p,n", RS_BATCH8)
def test_reduce_scatter_eight_rank_batches_match_oracle(lib, dtype, op, p, n):
    """Every element of every shard against the literal ring reduce-scatter,
    guard bands around each shard."""
    x = make_inputs(dtype, p, n, seed=p * 31 + n % 1000)
    want, _ = ring.ring_reduce_scatter(x, dtype, op)
    send = [to_dev(v, dtype) for v in x]
    shards = guarded_outputs(p, [ln for _, ln in ring.chunk_bounds(p, n)], dtype)
    lib.ccl_reduce_scatter(send, [s.view for s in shards], op=op)
    for k in range(p):
        assert_equal(to_host(shards[k].view), want[k], dtype, f"RS {dtype} {op} p={p} n={n} rank {k}")
        assert shards[k].guards_intact()


@pytest.mark.parametrize("dtype,op,p,n", RS_BATCH8)
def test_reduce_eight_rank_batches_match_oracle(lib, dtype, op, p, n):
    """The reduce to the root takes the same 8-rank batches: the root's
    buffer against the literal ring all-reduce's bits, guard bands."""
    x = make_inputs(dtype, p, n, seed=p * 37 + n % 1000)
    want, _, _ = ring.ring_allreduce(x, dtype, op)
    root = p - 2
    out = Guarded(n, dtype)
    lib.ccl_reduce([to_dev(v, dtype) for v in x], out.view, op=op, root=root)
    assert_equal(to_host(out.view), want[root], dtype, f"reduce {dtype} {op} p={p} n={n}")
    assert out.guards_intact()


# -------------------------------------------- alignment and in-place forms
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p,n", [(4, 1027), (8, 4096), (3, 50001)])
def test_unaligned_buffers_take_the_elementwise_path(lib, dtype, p, n):
    x = make_inputs(dtype, p, n, seed=3)
    ins = [Guarded(n, dtype, offset=GUARD + 1) for _ in range(p)]  # 4 or 2 bytes off 16
    for g, v in zip(ins, x):
        g.view.copy_(to_dev(v, dtype))
    want, _, _ = ring.ring_allreduce(x, dtype, "sum")
    outs = guarded_outputs(p, [n] * p, dtype, offset=GUARD + (1 if p % 2 else 0))
    lib.ccl_allreduce([g.view for g in ins], [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"unaligned AR rank {r}")
        assert outs[r].guards_intact()
    want_rs, _ = ring.ring_reduce_scatter(x, dtype, "sum")
    shards = guarded_outputs(p, [ln for _, ln in ring.chunk_bounds(p, n)], dtype, offset=GUARD + 1)
    lib.ccl_reduce_scatter([g.view for g in ins], [s.view for s in shards])
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], dtype, f"unaligned RS rank {k}")
        assert shards[k].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(4, 1 << 16), (5, 12345), (16, 1000)])
def test_in_place_forms(lib, dtype, p, n):
    x = make_inputs(dtype, p, n, seed=11)
    want, _, _ = ring.ring_allreduce(x, dtype, "sum")
    bufs = [to_dev(v, dtype) for v in x]
    lib.ccl_allreduce(bufs, bufs)
    for r in range(p):
        assert_equal(to_host(bufs[r]), want[r], dtype, f"in-place AR rank {r}")
    # reduce-scatter in place: rank k's shard is chunk k of its own input
    bufs = [to_dev(v, dtype) for v in x]
    bounds = ring.chunk_bounds(p, n)
    shards = [bufs[k][off:off + ln] for k, (off, ln) in enumerate(bounds)]
    want_rs, _ = ring.ring_reduce_scatter(x, dtype, "sum")
    lib.ccl_reduce_scatter(bufs, shards)
    for k in range(p):
        assert_equal(to_host(shards[k]), want_rs[k], dtype, f"in-place RS rank {k}")
    # all-gather in place: block k already sits at off(k) of rank k's output
    outs = [torch.zeros(n, dtype=bufs[0].dtype, device="cuda") for _ in range(p)]
    blocks = []
    for k, (off, ln) in enumerate(bounds):
        outs[k][off:off + ln].copy_(to_dev(want_rs[k], dtype))
        blocks.append(outs[k][off:off + ln])
    lib.ccl_all_gather(blocks, outs)
    for r in range(p):
        assert_equal(to_host(outs[r]), want[r], dtype, f"in-place AG rank {r}")


def test_zero_length_and_single_rank(lib):
    z = [torch.empty(0, device="cuda") for _ in range(3)]
    lib.ccl_allreduce(z, z)
    x = workloads.normal(1, 777, 1.0, seed=1)
    send = [to_dev(x[0], "f32")]
    recv = [torch.empty(777, device="cuda")]
    lib.ccl_allreduce(send, recv)
    assert_equal(to_host(recv[0]), x[0], "f32", "p=1")


def test_launch_counter_counts_one_fused_launch(lib):
    p, n = 4, 4096
    send = [torch.randn(n, device="cuda") for _ in range(p)]
    recv = [torch.empty(n, device="cuda") for _ in range(p)]
    before = lib.ccl_kernel_launch_count()
    lib.ccl_allreduce(send, recv)
    torch.cuda.synchronize()
    assert lib.ccl_kernel_launch_count() == before + 1


def test_fold_order_discriminator_on_gpu(lib):
    """Per chunk: x_{c+1} = 2^24, x_{c+2} = x_{c+3} = 1, x_c = -2^24; only the
    ring order (start at c+1, walk forward) yields 0."""
    p, n = 8, 8 * 1024
    bounds = ring.chunk_bounds(p, n)
    x = [np.zeros(n, dtype=np.float32) for _ in range(p)]
    for c, (off, ln) in enumerate(bounds):
        sl = slice(off, off + ln)
        x[(c + 1) % p][sl] = 2.0**24
        x[(c + 2) % p][sl] = 1.0
        x[(c + 3) % p][sl] = 1.0
        x[c][sl] = -(2.0**24)
    send = [to_dev(v, "f32") for v in x]
    recv = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_allreduce(send, recv)
    for r in range(p):
        assert (to_host(recv[r]) == 0).all()


# ------------------------------------------------------------- DDP bucket
def test_ddp_bucket_full_size(lib):
    """25 MB fp32 bucket per rank, p=8, N(0, 1e-3), scale 1/8 -> bf16."""
    p, n = 8, 6_553_600
    g = workloads.normal(p, n, 1e-3, seed=1)
    want = ring.bucket_allreduce_scale_cast(g, 1.0 / 8)
    send = [to_dev(v, "f32") for v in g]
    outs = guarded_outputs(p, [n] * p, "bf16")
    lib.ccl_bucket_allreduce_scale_cast(send, [o.view for o in outs], scale=1.0 / 8)
    for r in range(p):
        assert_bf16_close(to_host(outs[r].view), want[r], f"bucket rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("p,n,scale", [(3, 1001, 1 / 3), (8, 13, 0.125), (16, 70001, 1 / 16),
                                       (7, 4099, 1 / 7), (72, 5000, 1 / 72)])
def test_ddp_bucket_shapes(lib, p, n, scale):
    g = workloads.normal(p, n, 1e-3, seed=p)
    want = ring.bucket_allreduce_scale_cast(g, float(np.float32(scale)))
    send = [to_dev(v, "f32") for v in g]
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    lib.ccl_bucket_allreduce_scale_cast(send, outs, scale=float(np.float32(scale)))
    for r in range(p):
        assert_bf16_close(to_host(outs[r]), want[r], f"bucket p={p} rank {r}")


# ------------------------------------------------------- ZeRO, full size
def test_zero_rs_then_ag_full_size(lib):
    """p=16, 192 MiB bf16 per rank, N(0, 1e-2): RS (fp32 accumulation) then AG.
    Sampled outputs against the pointwise oracle; AG(RS) == AR on the device."""
    p, n = 16, 100_663_296
    idx = sample_indices(n, p, 1 << 20, seed=2)
    rng = np.random.default_rng(2)
    send, cols = [], []
    for _ in range(p):  # same stream as workloads.normal(p, n, 1e-2, 2, "bf16")
        v = rng.standard_normal(n, dtype=np.float32)
        v *= np.float32(1e-2)
        b = workloads.to_bf16_bits(v)
        cols.append(b[idx])
        send.append(to_dev(b, "bf16"))
        del v, b
    want = pointwise.allreduce_at_columns(cols, idx, n, "bf16")
    bounds = ring.chunk_bounds(p, n)
    shards = [torch.empty(ln, dtype=torch.bfloat16, device="cuda") for _, ln in bounds]
    lib.ccl_reduce_scatter(send, shards)
    gathered = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    lib.ccl_all_gather(shards, gathered)
    torch.cuda.synchronize()
    idx_t = torch.from_numpy(idx).cuda()
    for r in (0, 7, 15):
        assert_bf16_close(to_host(gathered[r][idx_t]), want, f"ZeRO AG(RS) rank {r}")
    # shard k at sampled positions of chunk k
    chunk = pointwise.chunk_of(p, n, idx)
    for k in (0, 5, 15):
        sel = chunk == k
        local = torch.from_numpy(idx[sel] - bounds[k][0]).cuda()
        assert_bf16_close(to_host(shards[k][local]), want[sel], f"ZeRO shard {k}")
    # properties at full size, on the device: every rank identical; AG(RS) == AR
    for r in range(1, p):
        assert torch.equal(gathered[r].view(torch.int16), gathered[0].view(torch.int16))
    ar = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lib.ccl_allreduce(send, ar + gathered[2:])  # gathered[0] still holds AG(RS)
    assert torch.equal(ar[0].view(torch.int16), gathered[0].view(torch.int16))
    assert torch.equal(gathered[2].view(torch.int16), gathered[0].view(torch.int16))


# ------------------------------------------------------------ all-to-allv
def test_moe_dispatch_combine_full_size(lib):
    """p=8, 16,384 tokens of 4096 bf16 per rank, Zipf(1.2) counts, seed 3."""
    hidden = 4096
    counts, rng = workloads.moe_counts(p=8, tokens_per_rank=16384, seed=3)
    tokens = workloads.moe_tokens(counts, hidden, rng, dtype="bf16")
    want = collectives.all_to_allv(tokens, counts, hidden)
    send = [to_dev(t, "bf16") for t in tokens]
    recv_rows = counts.sum(axis=0)
    recv = [torch.empty(int(r) * hidden, dtype=torch.bfloat16, device="cuda") for r in recv_rows]
    lib.ccl_all_to_allv(send, counts, recv, hidden)
    for d in range(8):
        assert_equal(to_host(recv[d]), want[d], "bf16", f"dispatch rank {d}")
    back = [torch.empty_like(s) for s in send]
    lib.ccl_all_to_allv(recv, counts.T, back, hidden)
    for s in range(8):
        assert torch.equal(back[s].view(torch.int16), send[s].view(torch.int16)), f"combine {s}"


@pytest.mark.parametrize("row_elems,dtype", [(7, "bf16"), (1, "bf16"), (3, "f32"), (13, "bf16"),
                                             (8, "bf16"), (33, "f32")])
@pytest.mark.parametrize("p", [2, 5, 8])
def test_all_to_allv_ragged_rows(lib, row_elems, dtype, p):
    """Rows whose byte size is not a multiple of 16: source and destination
    blocks differ in 16-byte phase, which takes the shuffle realignment path."""
    rng = np.random.default_rng(row_elems * 10 + p)
    counts = rng.integers(0, 300, size=(p, p))
    counts[p - 1, :] = 0
    counts[0, 1 % p] = 5000
    send_np = [make_inputs(dtype, 1, int(counts[s].sum()) * row_elems, seed=s)[0] for s in range(p)]
    want = collectives.all_to_allv(send_np, counts, row_elems)
    send = [to_dev(v, dtype) for v in send_np]
    outs = [Guarded(int(counts[:, d].sum()) * row_elems, dtype, offset=GUARD + d % 3)
            for d in range(p)]
    lib.ccl_all_to_allv(send, counts, [o.view for o in outs], row_elems)
    for d in range(p):
        assert_equal(to_host(outs[d].view), want[d], dtype, f"a2av rank {d}")
        assert outs[d].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(1, 9), (2, 4099), (3, 1001), (5, 3), (8, 70001), (16, 1 << 20),
                                 (72, 10000)])
def test_all_to_all_equal_blocks(lib, dtype, p, n):
    """The plain block transpose, ragged chunk-rule blocks included (n not a
    multiple of p, and n < p where some blocks are empty)."""
    x = make_inputs(dtype, p, n, seed=p * 7 + n)
    want = collectives.all_to_all(x)
    outs = [Guarded(len(want[j]), dtype, offset=GUARD + j % 3) for j in range(p)]
    lib.ccl_all_to_all([to_dev(v, dtype) for v in x], [o.view for o in outs])
    for j in range(p):
        assert_equal(to_host(outs[j].view), want[j], dtype, f"A2A {dtype} p={p} n={n} rank {j}")
        assert outs[j].guards_intact()
    if n % p == 0:  # the transpose is its own inverse when all blocks are equal
        back = [torch.empty_like(o.view) for o in outs]
        lib.ccl_all_to_all([o.view for o in outs], back)
        for j in range(p):
            assert_equal(to_host(back[j]), x[j], dtype, f"A2A twice rank {j}")


def a2av_launches(p: int) -> int:
    """Launches of an all-to-allv: the row-prefix table of p sources x
    (destinations + 1) columns travels in the parameter block, 16 x 17
    entries in the 4 KB form, 7408 in the 32 KB form (uint32 entries)."""
    if p <= 16:
        return 1
    per = 7408 // p - 1
    return -(-p // per)


@pytest.mark.parametrize("p,row,hi", [(16, 64, 40), (48, 3, 6), (85, 1, 3), (86, 2, 3), (128, 8, 2)])
def test_all_to_allv_many_blocks(lib, p, row, hi):
    """Many blocks: p=16 (256 blocks, the 4 KB parameter block), p=48 with
    3-element rows (about 1900 blocks, phase-shifted, one launch), p=85 with
    one-element rows (the largest p whose table fits one launch), p=86 (two
    launches), p=128 (about 8200 blocks of 0-1 rows, three launches)."""
    rng = np.random.default_rng(5 + p)
    counts = rng.integers(0 if p > 16 else 1, hi, size=(p, p))
    x = [workloads.normal(1, max(int(counts[s].sum()), 1) * row, 1.0, seed=s, dtype="bf16")[0][: int(counts[s].sum()) * row]
         for s in range(p)]
    want = collectives.all_to_allv(x, counts, row)
    recv = [torch.empty(int(counts[:, d].sum()) * row, dtype=torch.bfloat16, device="cuda")
            for d in range(p)]
    blocks = int((counts > 0).sum())
    n0 = lib.ccl_kernel_launch_count()
    lib.ccl_all_to_allv([to_dev(v, "bf16") for v in x], counts, recv, row)
    assert blocks > 0
    assert lib.ccl_kernel_launch_count() - n0 == a2av_launches(p)
    for d in range(p):
        assert_equal(to_host(recv[d]), want[d], "bf16", f"rank {d}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p,n", [(72, 256), (72, 512), (128, 1000), (72, 72 * 301 + 5), (100, 37)])
def test_all_to_all_small_blocks_one_launch(lib, dtype, p, n):
    """The plain all-to-all is one launch for any p (its blocks follow the
    chunk rule, nothing travels in a table): 1 KiB and 2 KiB per rank at
    p = 72 (blocks of 3-4 and 7-8 elements, no block holding a whole 16-byte
    unit), p = 128, p = 100 with n < p (empty blocks), and mid-size blocks
    off the 16-byte grid; every element against the oracle, guard bands."""
    x = make_inputs(dtype, p, n, seed=p + n)
    want = collectives.all_to_all(x)
    outs = [Guarded(len(want[j]), dtype, offset=GUARD + j % 5) for j in range(p)]
    send = [to_dev(v, dtype) for v in x]
    n0 = lib.ccl_kernel_launch_count()
    lib.ccl_all_to_all(send, [o.view for o in outs])
    assert lib.ccl_kernel_launch_count() - n0 == 1
    for j in range(p):
        assert_equal(to_host(outs[j].view), want[j], dtype, f"A2A {dtype} p={p} n={n} rank {j}")
        assert outs[j].guards_intact()


@pytest.mark.parametrize("row_elems,dtype", [(1, "bf16"), (1, "f32"), (3, "bf16"), (5, "f32")])
def test_all_to_allv_tiny_rows_straddle_units(lib, row_elems, dtype):
    """Rows far smaller than a 16-byte unit with many empty blocks: every
    destination unit holds elements of several blocks and is assembled
    element by element; p = 24, counts 0-3 rows."""
    p = 24
    rng = np.random.default_rng(row_elems * 31 + len(dtype))
    counts = rng.integers(0, 4, size=(p, p))
    counts[rng.random((p, p)) < 0.3] = 0
    send_np = [make_inputs(dtype, 1, max(1, int(counts[s].sum()) * row_elems), seed=s)[0][: int(counts[s].sum()) * row_elems]
               for s in range(p)]
    want = collectives.all_to_allv(send_np, counts, row_elems)
    send = [to_dev(np.ascontiguousarray(v), dtype) for v in send_np]
    outs = [Guarded(int(counts[:, d].sum()) * row_elems, dtype, offset=GUARD + d % 7) for d in range(p)]
    n0 = lib.ccl_kernel_launch_count()
    lib.ccl_all_to_allv(send, counts, [o.view for o in outs], row_elems)
    assert lib.ccl_kernel_launch_count() - n0 == 1
    for d in range(p):
        assert_equal(to_host(outs[d].view), want[d], dtype, f"a2av rank {d}")
        assert outs[d].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "i32", "bf16"])
@pytest.mark.parametrize("scale", [0, 1, 9000])
def test_all_to_allv_block_edges_off_grid_same_phase(lib, dtype, scale):
    """Block edges off the 16-byte grid while every block's source and
    destination share the 16-byte phase (so no realignment is needed):
    p = 2, one-element rows, counts chosen so that block (1, 1) starts
    6 or 4 bytes into a unit on both sides and destination 0 ends off the
    grid.  The units holding those edges go through the small-block stage;
    scale 9000 spreads each destination over a hundred tiles or more."""
    u = 16 // (2 if dtype == "bf16" else 4)  # elements per 16-byte unit
    a, b, c, d = (scale, 2 * scale + 1, 3 * scale + 2, scale + 3)
    if dtype == "bf16":
        counts = np.array([[8 + u * a, 3 + u * b], [3 + u * c, 5 + u * d]])
    else:
        counts = np.array([[4 + u * a, 1 + u * b], [1 + u * c, 3 + u * d]])
    p = 2
    send_np = [make_inputs(dtype, 1, int(counts[s].sum()), seed=40 + s)[0] for s in range(p)]
    want = collectives.all_to_allv(send_np, counts, 1)
    send = [to_dev(v, dtype) for v in send_np]
    outs = [Guarded(int(counts[:, j].sum()), dtype) for j in range(p)]
    n0 = lib.ccl_kernel_launch_count()
    lib.ccl_all_to_allv(send, counts, [o.view for o in outs], 1)
    assert lib.ccl_kernel_launch_count() - n0 == 1
    for j in range(p):
        assert_equal(to_host(outs[j].view), want[j], dtype, f"a2av {dtype} scale {scale} rank {j}")
        assert outs[j].guards_intact()


# ------------------------------------------- bulk-copy fan-out (TMA bulk)
# with CCL_FORCE_VARIANT=tma, all-gather / broadcast calls with blocks >= 1 MiB,
# p | n and aligned device buffers run on the bulk-copy engine: whole tiles, a
# partial last tile when a block is not a whole number of tiles, 1 to 24 ranks


@pytest.fixture
def tma(monkeypatch):
    monkeypatch.setenv("CCL_FORCE_VARIANT", "tma")
    yield



@pytest.mark.parametrize("dtype,p,block", [("bf16", 16, 1 << 20), ("f32", 2, (1 << 18) + 12),
                                           ("f32", 24, 1 << 18), ("bf16", 1, 1 << 21), ("f32", 5, 300_004)])
def test_bulk_fanout_all_gather(lib, tma, dtype, p, block):
    n = p * block
    shards_np = make_inputs(dtype, p, block, seed=p + block)  # rank k's block
    want, _ = ring.ring_all_gather(shards_np, dtype)
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_device_error_flag(clear=True)
    lib.ccl_all_gather([to_dev(v, dtype) for v in shards_np], [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"fan-out all-gather rank {r}")
        assert outs[r].guards_intact()
    assert lib.ccl_device_error_flag() == 0


def test_bulk_fanout_all_gather_in_place(lib, tma):
    p, block = 8, 1 << 18  # 1 MiB fp32 blocks
    n = p * block
    x = make_inputs("f32", p, n, seed=3)
    want, _ = ring.ring_all_gather([x[k][k * block:(k + 1) * block].copy() for k in range(p)], "f32")
    bufs = [to_dev(v, "f32") for v in x]  # block k already sits at off(k) of rank k's buffer
    lib.ccl_all_gather([bufs[k][k * block:(k + 1) * block] for k in range(p)], bufs)
    for r in range(p):
        assert_equal(to_host(bufs[r]), want[r], "f32", f"in-place all-gather rank {r}")


@pytest.mark.parametrize("dtype,p,n,root", [("f32", 16, (1 << 24) + 4, 0), ("bf16", 3, 1 << 20, 2)])
def test_bulk_fanout_broadcast(lib, tma, dtype, p, n, root):
    data = make_inputs(dtype, 1, n, seed=p + root)[0]  # the root's buffer
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_broadcast(to_dev(data, dtype), [o.view for o in outs], root=root)
    want = [data] * p
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"fan-out broadcast rank {r}")
        assert outs[r].guards_intact()
    # in place: the root's buffer is its own output
    bufs = [torch.empty(n, dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device="cuda")
            for _ in range(p)]
    bufs[root].copy_(to_dev(data, dtype))
    lib.ccl_broadcast(bufs[root], bufs, root=root)
    for r in range(p):
        assert_equal(to_host(bufs[r]), want[r], dtype, f"in-place broadcast rank {r}")
    assert lib.ccl_device_error_flag() == 0


# -------------------------------------------------------- literal engine
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", [(1, 100), (2, 4099), (4, 1 << 16), (5, 13), (8, 70001), (16, 1000)])
def test_literal_engine_matches_oracle_and_counts_bytes(lib, dtype, p, n):
    x = make_inputs(dtype, p, n, seed=p + n)
    send = [to_dev(v, dtype) for v in x]
    want, rs_bytes, ag_bytes = ring.ring_allreduce(x, dtype, "sum")
    recv = [torch.empty(n, dtype=send[0].dtype, device="cuda") for _ in range(p)]
    sent = lib.ccl_ring_allreduce_literal(send, recv)
    for r in range(p):
        assert_equal(to_host(recv[r]), want[r], dtype, f"literal AR rank {r}")
    assert sent == [a + b for a, b in zip(rs_bytes, ag_bytes)]
    # the fused kernel gives the same bits
    fused = [torch.empty_like(t) for t in recv]
    lib.ccl_allreduce(send, fused)
    for r in range(p):
        assert torch.equal(fused[r].view(torch.int16 if dtype == "bf16" else torch.int32),
                           recv[r].view(torch.int16 if dtype == "bf16" else torch.int32))
    want_rs, rs_only = ring.ring_reduce_scatter(x, dtype, "sum")
    shards = [torch.empty(ln, dtype=send[0].dtype, device="cuda") for _, ln in ring.chunk_bounds(p, n)]
    sent_rs = lib.ccl_ring_reduce_scatter_literal(send, shards)
    for k in range(p):
        assert_equal(to_host(shards[k]), want_rs[k], dtype, f"literal RS rank {k}")
    assert sent_rs == rs_only
    gathered = [torch.empty(n, dtype=send[0].dtype, device="cuda") for _ in range(p)]
    sent_ag = lib.ccl_ring_all_gather_literal(shards, gathered)
    _, ag_only = ring.ring_all_gather(want_rs, dtype)
    for r in range(p):
        assert_equal(to_host(gathered[r]), want[r], dtype, f"literal AG rank {r}")
    assert sent_ag == ag_only


@pytest.mark.parametrize("op", ["max", "min"])
def test_literal_engine_max_min_in_place(lib, op):
    p, n = 6, 10007
    x = workloads.normal(p, n, 1.0, seed=4)
    want, _, _ = ring.ring_allreduce(x, "f32", op)
    bufs = [to_dev(v, "f32") for v in x]
    lib.ccl_ring_allreduce_literal(bufs, bufs, op=op)
    for r in range(p):
        assert_equal(to_host(bufs[r]), want[r], "f32", f"literal {op} rank {r}")


# ------------------------------------------------- message-size sweep
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p", [2, 4, 8, 16])
def test_sweep_sizes_small_full_compare(lib, dtype, p):
    """1 KiB .. 4 MiB per rank (powers of two), U(-1, 1), every element."""
    e = 4 if dtype == "f32" else 2
    for kib in [1 << k for k in range(0, 13)]:
        n = kib * 1024 // e
        x = workloads.uniform(p, n, seed=4, dtype=dtype)
        want, _, _ = ring.ring_allreduce(x, dtype, "sum")
        send = [to_dev(v, dtype) for v in x]
        recv = [torch.empty_like(s) for s in send]
        lib.ccl_allreduce(send, recv)
        for r in (0, p - 1):
            assert_equal(to_host(recv[r]), want[r], dtype, f"sweep {kib} KiB p={p} rank {r}")


@pytest.mark.parametrize("dtype,p,mib", [("f32", 16, 1024), ("bf16", 16, 1024), ("f32", 72, 256),
                                         ("bf16", 72, 256), ("f32", 2, 1024)])
def test_sweep_largest_sizes_sampled(lib, dtype, p, mib):
    """The sweep's largest messages: sampled elements against the pointwise
    oracle; all ranks identical on the device.  At these sizes the U(-1, 1)
    inputs are drawn on the device by torch's seeded generator (drawing up to
    16 GiB on the host would take minutes); the oracle reads the values at the
    sampled positions."""
    e = 4 if dtype == "f32" else 2
    n = mib * (1 << 20) // e
    idx = sample_indices(n, p, 1 << 20, seed=p)  # >= 1 M sampled elements (plus every chunk edge)
    idx_t = torch.from_numpy(idx).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4)
    send, cols = [], []
    for _ in range(p):
        v = torch.rand(n, generator=gen, device="cuda", dtype=torch.float32) * 2.0 - 1.0
        v = v.to(torch.bfloat16) if dtype == "bf16" else v
        cols.append(to_host(v[idx_t]))
        send.append(v)
    recv = [torch.empty_like(s) for s in send]
    lib.ccl_allreduce(send, recv)
    want = pointwise.allreduce_at_columns(cols, idx, n, dtype)
    for r in (0, p // 2, p - 1):
        assert_equal(to_host(recv[r][idx_t]), want, dtype, f"sweep {mib} MiB p={p} rank {r}")
    view = torch.int16 if dtype == "bf16" else torch.int32
    for r in range(1, p):
        assert torch.equal(recv[r].view(view), recv[0].view(view))


# ------------------------------------ chunks off the 16-byte grid, many warps
UNALIGNED_BIG = [(72, 72 * 20011 + 29), (3, 3 * 400009 + 2), (7, 7 * 100003 + 5)]


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", UNALIGNED_BIG)
def test_unaligned_chunks_span_many_warps(lib, dtype, p, n):
    """Chunk offsets off the 16-byte grid, chunks spanning many warps and
    grid-stride passes: the reduce-scatter's realigned shard stores and the
    all-gather's realigned block loads.  Sampled indices (every chunk edge
    included) against the oracle; AG(RS) == AR and RS == AR's chunks on every
    element; guard bands intact."""
    x = make_inputs(dtype, p, n, seed=p + n)
    idx = sample_indices(n, p, 1 << 16, seed=p)
    want = pointwise.allreduce_at_columns([v[idx] for v in x], idx, n, dtype)
    send = [to_dev(v, dtype) for v in x]
    del x
    ar = [torch.empty_like(t) for t in send]
    lib.ccl_allreduce(send, ar)
    assert_equal(to_host(ar[0][torch.from_numpy(idx).cuda()]), want, dtype, "AR")
    bounds = ring.chunk_bounds(p, n)
    shards = [Guarded(ln, dtype) for _, ln in bounds]
    lib.ccl_reduce_scatter(send, [g.view for g in shards])
    for k, (off, ln) in enumerate(bounds):
        sel = (idx >= off) & (idx < off + ln)
        got = to_host(shards[k].view[torch.from_numpy(idx[sel] - off).cuda()])
        assert_equal(got, want[sel], dtype, f"RS rank {k}")
        assert torch.equal(_bits(shards[k].view), _bits(ar[0][off:off + ln])), f"RS == AR chunk {k}"
        assert shards[k].guards_intact()
    out = [Guarded(n, dtype, offset=GUARD + (4 if dtype != "bf16" else 8) * (r % 2)) for r in range(p)]
    lib.ccl_all_gather([g.view for g in shards], [o.view for o in out])
    for r in range(p):
        assert torch.equal(_bits(out[r].view), _bits(ar[0])), f"AG(RS) rank {r}"
        assert out[r].guards_intact()


@pytest.mark.parametrize("p,n", [(72, 72 * 20011 + 29), (3, 3 * 400009 + 2), (9, 9 * 50021 + 4)])
def test_bf16_wire_reduce_scatter_unaligned_shards(lib, p, n):
    x = make_inputs("bf16", p, n, seed=p * 3 + n)
    idx = sample_indices(n, p, 1 << 16, seed=p + 1)
    want = pointwise.allreduce_at_columns([v[idx] for v in x], idx, n, "bf16", wire="bf16")
    send = [to_dev(v, "bf16") for v in x]
    bounds = ring.chunk_bounds(p, n)
    shards = [Guarded(ln, "bf16") for _, ln in bounds]
    lib.ccl_reduce_scatter_bf16_wire(send, [g.view for g in shards])
    for k, (off, ln) in enumerate(bounds):
        sel = (idx >= off) & (idx < off + ln)
        got = to_host(shards[k].view[torch.from_numpy(idx[sel] - off).cuda()])
        assert_equal(got, want[sel], "bf16", f"wire RS rank {k}")
        assert shards[k].guards_intact()


# ------------------------------------------------ other all-reduce schedules
SCHED_CASES = [(s, p, n) for s in ("recursive_doubling", "rabenseifner") for p, n in
               [(2, 4099), (4, 1000), (8, 70001), (16, 65536), (128, 1000)]] + \
              [(s, p, n) for s in ("binomial_tree", "naive") for p, n in
               [(1, 10), (2, 4099), (3, 1001), (5, 13), (7, 70001), (16, 65536), (72, 1000)]]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("schedule,p,n", SCHED_CASES)
def test_allreduce_schedules_match_their_oracles(lib, dtype, schedule, p, n):
    from oracle import schedules

    x = make_inputs(dtype, p, n, seed=p + 31 * n)
    want, _ = schedules.allreduce(schedule, x, dtype)
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_allreduce_schedule([to_dev(v, dtype) for v in x], [o.view for o in outs], schedule)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"{schedule} p={p} rank {r}")
        assert outs[r].guards_intact()


def test_schedule_discriminators_on_gpu(lib):
    """Hand-derived per-schedule values (see tests/test_oracle_schedules.py)."""
    cases = {"recursive_doubling": 1.0, "binomial_tree": 1.0, "rabenseifner": 2.0, "naive": 1.0,
             "ring": None}
    vals = [2.0**24, 1.0, -(2.0**24), 1.0]
    n = 4096 + 3
    send = [torch.full((n,), v, device="cuda") for v in vals]
    for s, want in cases.items():
        recv = [torch.empty(n, device="cuda") for _ in range(4)]
        lib.ccl_allreduce_schedule(send, recv, s)
        if want is not None:
            assert (to_host(recv[0]) == want).all(), s


def test_schedule_argument_errors(lib):
    x = [torch.ones(8, device="cuda") for _ in range(6)]
    with pytest.raises(lib.CclError):
        lib.ccl_allreduce_schedule(x, [torch.empty_like(t) for t in x], "recursive_doubling")
    with pytest.raises(lib.CclError):
        lib.ccl_allreduce_schedule(x, [torch.empty_like(t) for t in x], "naive", op="max")


# ------------------------------------------------ bf16 on the wire
WIRE_CASES = [(1, 10), (2, 4099), (3, 1001), (4, 70001), (8, 65536 + 3), (16, 1000), (72, 1000), (5, 4)]


@pytest.mark.parametrize("p,n", WIRE_CASES)
def test_bf16_wire_matches_oracle(lib, p, n):
    x = make_inputs("bf16", p, n, seed=p * 13 + n)
    send = [to_dev(v, "bf16") for v in x]
    want, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    outs = guarded_outputs(p, [n] * p, "bf16")
    lib.ccl_allreduce_bf16_wire(send, [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], "bf16", f"bf16-wire AR rank {r}")
        assert outs[r].guards_intact()
    want_rs, _ = ring.ring_reduce_scatter(x, "bf16", wire="bf16")
    shards = guarded_outputs(p, [ln for _, ln in ring.chunk_bounds(p, n)], "bf16", offset=GUARD + 1)
    lib.ccl_reduce_scatter_bf16_wire(send, [g.view for g in shards])
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], "bf16", f"bf16-wire RS rank {k}")
        assert shards[k].guards_intact()


def test_bf16_wire_unaligned_and_in_place(lib):
    p, n = 6, 10007
    x = make_inputs("bf16", p, n, seed=21)
    want, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    ins = [Guarded(n, "bf16", offset=GUARD + 1) for _ in range(p)]
    for g, v in zip(ins, x):
        g.view.copy_(to_dev(v, "bf16"))
    lib.ccl_allreduce_bf16_wire([g.view for g in ins], [g.view for g in ins])
    for r in range(p):
        assert_equal(to_host(ins[r].view), want[r], "bf16", f"in place rank {r}")
        assert ins[r].guards_intact()


def test_bf16_wire_hand_case_on_gpu(lib):
    """The tie case of tests/test_oracle_bf16_wire.py on 3 x 4096 elements."""
    n = 3 * 4096
    send = [torch.full((n,), v, dtype=torch.bfloat16, device="cuda") for v in (2.0**-8, 1.0, 2.0**-8)]
    recv = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    lib.ccl_allreduce_bf16_wire(send, recv)
    want = np.repeat(np.array([1.0, 1.0 + 2.0**-7, 1.0], dtype=np.float32), 4096)
    for r in range(3):
        np.testing.assert_array_equal(recv[r].float().cpu().numpy(), want)
    fp32 = [torch.empty_like(t) for t in recv]
    lib.ccl_allreduce(send, fp32)
    assert (fp32[0].float() == 1.0 + 2.0**-7).all()


def test_bf16_wire_full_size_sampled(lib):
    """The ZeRO reduce-scatter size (p=16, 192 MiB bf16 per rank), sampled."""
    p, n = 16, 192 * (1 << 20) // 2
    idx = sample_indices(n, p, 1 << 17, seed=77)
    idx_t = torch.from_numpy(idx).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2)
    send = [(torch.randn(n, generator=gen, device="cuda") * 1e-2).to(torch.bfloat16) for _ in range(p)]
    cols = [to_host(v[idx_t]) for v in send]
    recv = [torch.empty_like(v) for v in send]
    lib.ccl_allreduce_bf16_wire(send, recv)
    want = pointwise.allreduce_at_columns(cols, idx, n, "bf16", wire="bf16")
    for r in (0, 7, 15):
        assert_equal(to_host(recv[r][idx_t]), want, "bf16", f"bf16-wire 192 MiB rank {r}")


def test_bf16_wire_rejects_other_dtypes(lib):
    x = [torch.ones(8, device="cuda") for _ in range(2)]
    with pytest.raises(ValueError):
        lib.ccl_allreduce_bf16_wire(x, [torch.empty_like(t) for t in x])


# ------------------------------------------- hierarchical / 2-D two-level ring
# (p, group, n): 2 nodes x 8, 4 x 2, 3 x 3 with sub-chunks that start off the
# 16-byte grid, one group (the flat ring), groups of one, tiny n (empty
# sub-chunks), 9 x 8 = 72 ranks
HIER_CASES = [(16, 8, 65536 + 7), (8, 2, 70001), (9, 3, 1001), (6, 6, 4099), (6, 1, 4099),
              (4, 2, 3), (72, 8, 1000), (2, 1, 4096 * 4 + 5)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,group,n", HIER_CASES)
def test_hierarchical_allreduce_matches_oracle(lib, dtype, p, group, n):
    from oracle import schedules

    x = make_inputs(dtype, p, n, seed=p + 7 * n + group)
    want, _ = schedules.hierarchical(x, group, dtype)
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_allreduce_hierarchical([to_dev(v, dtype) for v in x], [o.view for o in outs], group)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"hierarchical p={p} a={group} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_hierarchical_unaligned_and_in_place(lib, dtype):
    from oracle import schedules

    p, group, n = 8, 4, 10007
    x = make_inputs(dtype, p, n, seed=11)
    want, _ = schedules.hierarchical(x, group, dtype)
    ins = [Guarded(n, dtype, offset=GUARD + 1) for _ in range(p)]  # off the 16-byte grid
    for g, v in zip(ins, x):
        g.view.copy_(to_dev(v, dtype))
    lib.ccl_allreduce_hierarchical([g.view for g in ins], [g.view for g in ins], group)  # in place
    for r in range(p):
        assert_equal(to_host(ins[r].view), want[r], dtype, f"in place rank {r}")
        assert ins[r].guards_intact()


def test_hierarchical_hand_cases_on_gpu(lib):
    """The hand-derived fold orders of tests/test_oracle_schedules.py, on
    vectors long enough for the 16-byte path."""
    cases = [(3, [-(2.0**24), 2.0**24, 1.0, 0.0, 0.0, 0.0]), (2, [-(2.0**24), 0.0, 2.0**24, 0.0, 1.0, 0.0])]
    n = 6 * 1024
    for group, vals in cases:
        send = [torch.full((n,), v, device="cuda") for v in vals]
        recv = [torch.empty(n, device="cuda") for _ in range(6)]
        lib.ccl_allreduce_hierarchical(send, recv, group)
        from oracle import schedules
        want, _ = schedules.hierarchical([to_host(t) for t in send], group)
        for r in range(6):
            np.testing.assert_array_equal(to_host(recv[r]), want[r])
        assert set(np.unique(to_host(recv[0])).tolist()) == {0.0, 1.0}


@pytest.mark.parametrize("p,group,mib", [(16, 8, 256), (72, 8, 128)])
def test_hierarchical_full_size_sampled(lib, p, group, mib):
    """The bench's hierarchical configurations (fp32, U(-1, 1) drawn on the
    device with torch's seeded generator): sampled elements against the
    pointwise two-level fold; all ranks identical on the device."""
    from oracle import pointwise

    n = mib * (1 << 20) // 4
    b = p // group
    edges = []
    for off, ln in ring.chunk_bounds(group, n):  # every sub-chunk's first and last element
        for o2, l2 in ring.chunk_bounds(b, ln):
            edges += [off + o2, off + o2 + max(l2 - 1, 0)]
    idx = np.unique(np.concatenate([sample_indices(n, p, 1 << 17, seed=p + group),
                                    np.array(edges, dtype=np.int64)]))
    idx_t = torch.from_numpy(idx).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4)
    send = [torch.rand(n, generator=gen, device="cuda") * 2.0 - 1.0 for _ in range(p)]
    cols = [to_host(v[idx_t]) for v in send]
    recv = [torch.empty_like(v) for v in send]
    lib.ccl_allreduce_hierarchical(send, recv, group)
    want = pointwise.hierarchical_at_columns(cols, idx, n, group, "f32")
    for r in (0, group, p - 1):
        assert_equal(to_host(recv[r][idx_t]), want, "f32", f"hierarchical {mib} MiB p={p} rank {r}")
    for r in range(1, p):
        assert torch.equal(recv[r].view(torch.int32), recv[0].view(torch.int32))


def test_hierarchical_argument_errors(lib):
    x = [torch.ones(8, device="cuda") for _ in range(6)]
    for bad in (0, 4, 7):
        with pytest.raises(lib.CclError):
            lib.ccl_allreduce_hierarchical(x, [torch.empty_like(t) for t in x], bad)
    with pytest.raises(lib.CclError):
        lib.ccl_allreduce_hierarchical(x, [torch.empty_like(t) for t in x], 3, op="max")


# ---------------------------------------- broadcast / reduce / scatter / gather
ROOTED = [(1, 10), (3, 1001), (4, 4), (8, 70001), (16, 65543), (72, 1000)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("p,n", ROOTED)
def test_rooted_primitives_match_oracle(lib, dtype, p, n):
    x = make_inputs(dtype, p, n, seed=3 * p + n)
    root = p // 2
    send = [to_dev(v, dtype) for v in x]
    # broadcast
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_broadcast(send[root], [o.view for o in outs], root=root)
    for r, o in enumerate(outs):
        assert_equal(to_host(o.view), collectives.broadcast(x, root)[r], dtype, f"bcast {r}")
        assert o.guards_intact()
    # reduce: the root gets the ring all-reduce's bits
    red = Guarded(n, dtype)
    lib.ccl_reduce(send, red.view, root=root)
    assert_equal(to_host(red.view), collectives.reduce_ring(x, root, dtype)[root], dtype, "reduce")
    assert red.guards_intact()
    # scatter of the root's buffer, then gather back to the root
    parts = guarded_outputs(p, [ln for _, ln in ring.chunk_bounds(p, n)], dtype, offset=GUARD + 1)
    lib.ccl_scatter(send[root], [q.view for q in parts], root=root)
    want_parts = collectives.scatter(x[root], p)
    for k, q in enumerate(parts):
        assert_equal(to_host(q.view), want_parts[k], dtype, f"scatter {k}")
        assert q.guards_intact()
    back = Guarded(n, dtype)
    lib.ccl_gather([q.view for q in parts], back.view, root=root)
    assert_equal(to_host(back.view), x[root], dtype, "gather(scatter)")
    assert back.guards_intact()


@pytest.mark.parametrize("p,n", [(4, 1 << 20), (8, 6_553_600), (16, 1000)])
def test_identities_on_gpu(lib, p, n):
    """Section 4.2 on the device: broadcast = scatter + all-gather, and
    all-reduce = reduce + broadcast, bit for bit."""
    x = make_inputs("f32", p, n, seed=p)
    send = [to_dev(v, "f32") for v in x]
    root = 1
    parts = [torch.empty(ln, device="cuda") for _, ln in ring.chunk_bounds(p, n)]
    lib.ccl_scatter(send[root], parts, root=root)
    via_ag = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_all_gather(parts, via_ag)
    direct = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_broadcast(send[root], direct, root=root)
    for a_, b_ in zip(via_ag, direct):
        assert torch.equal(a_.view(torch.int32), b_.view(torch.int32))
    red = torch.empty(n, device="cuda")
    lib.ccl_reduce(send, red, root=root)
    bc = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_broadcast(red, bc, root=root)
    ar = [torch.empty(n, device="cuda") for _ in range(p)]
    lib.ccl_allreduce(send, ar)
    for a_, b_ in zip(ar, bc):
        assert torch.equal(a_.view(torch.int32), b_.view(torch.int32))


# vectors per thread of the broadcast (the host picks them by grid size):
# 2 for small calls, 1 once that grid fills a wave, 8 for large ones
BCAST_SIZE_CLASSES = [("bf16", 16, 100_003), ("f32", 8, 2 * 1048576 + 3), ("bf16", 4, 4 * 1048576 + 1),
                      ("f32", 4, 6 * 1048576 + 5)]


@pytest.mark.parametrize("dtype,p,n", BCAST_SIZE_CLASSES)
def test_broadcast_size_classes_match_oracle(lib, dtype, p, n):
    """Every element of every output against the root's buffer, at sizes
    that select 2, 1 and 8 vectors per thread, guard bands."""
    x = make_inputs(dtype, p, n, seed=11 * p + n % 1000)
    root = p - 1
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_broadcast(to_dev(x[root], dtype), [o.view for o in outs], root=root)
    want = collectives.broadcast(x, root)
    for r, o in enumerate(outs):
        assert_equal(to_host(o.view), want[r], dtype, f"bcast {dtype} p={p} n={n} rank {r}")
        assert o.guards_intact()


def test_rooted_in_place_forms(lib):
    p, n = 5, 12345
    x = make_inputs("f32", p, n, seed=9)
    send = [to_dev(v, "f32") for v in x]
    root = 2
    outs = [torch.empty(n, device="cuda") for _ in range(p)]
    outs[root] = send[root]
    lib.ccl_broadcast(send[root], outs, root=root)
    for o in outs:
        assert_equal(to_host(o), x[root], "f32", "in-place bcast")
    want = collectives.reduce_ring(x, root)[root]
    lib.ccl_reduce(send, send[root], root=root)
    assert_equal(to_host(send[root]), want, "f32", "in-place reduce")


def test_bucket_reads_and_writes_pinned_host_memory(lib):
    """Inputs and outputs in pinned host memory: the kernel moves the data over
    the host link itself; the bits equal the oracle's."""
    p, n = 8, 1_000_003
    g = workloads.normal(p, n, 1e-3, seed=21)
    want = ring.bucket_allreduce_scale_cast(g, 0.125)
    h_in = [torch.from_numpy(v).pin_memory() for v in g]
    h_out = [torch.empty(n, dtype=torch.bfloat16).pin_memory() for _ in range(p)]
    lib.ccl_bucket_allreduce_scale_cast(h_in, h_out, scale=0.125)
    torch.cuda.synchronize()
    for r in range(p):
        np.testing.assert_array_equal(h_out[r].view(torch.int16).numpy().view(np.uint16), want[r])


# ------------------------------------------------ Ulysses head <-> sequence
def test_ulysses_full_size(lib):
    """The bench's Ulysses configuration (p=8, 8192 tokens x 32 heads x 128
    bf16 per rank), every element, forward and inverse."""
    p, sp, H, D = 8, 8192, 32, 128
    n = sp * H * D
    x = workloads.normal(p, n, 1.0, 17, dtype="bf16")
    want = collectives.ulysses_seq_to_heads(x, H, D)
    send = [to_dev(v, "bf16") for v in x]
    recv = [torch.empty_like(t) for t in send]
    lib.ccl_all_to_all_heads(send, recv, sp, H, D)
    for r in range(p):
        assert_equal(to_host(recv[r]), want[r], "bf16", f"heads rank {r}")
    back = [torch.empty_like(t) for t in send]
    lib.ccl_all_to_all_heads(recv, back, sp, H, D, inverse=True)
    for r in range(p):
        assert torch.equal(back[r], send[r])


# rows of 8 KB and over (x covers 256 vectors), rows under 256 vectors (2-D
# blocks), 30 vectors a row (a part-idle warp), unaligned segments (scalar
# path), ragged row blocks (sp = 33, 50, 1001)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("p,sp,H,D", [(1, 5, 4, 8), (2, 64, 8, 64), (4, 33, 16, 128), (8, 128, 32, 128),
                                      (4, 7, 4, 3), (2, 50, 6, 20), (8, 1001, 32, 128)])
def test_ulysses_all_to_all_matches_oracle(lib, dtype, p, sp, H, D):
    n = sp * H * D
    x = make_inputs(dtype, p, n, seed=p * 7 + sp)
    want = collectives.ulysses_seq_to_heads(x, H, D)
    outs = guarded_outputs(p, [n] * p, dtype)
    lib.ccl_all_to_all_heads([to_dev(v, dtype) for v in x], [o.view for o in outs], sp, H, D)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"heads rank {r}")
        assert outs[r].guards_intact()
    back = [torch.empty(n, dtype=outs[0].view.dtype, device="cuda") for _ in range(p)]
    lib.ccl_all_to_all_heads([o.view for o in outs], back, sp, H, D, inverse=True)
    for r in range(p):
        assert_equal(to_host(back[r]), x[r], dtype, f"inverse rank {r}")
