"""Seeded random parity cases across the primitives: sizes, rank counts,
dtypes, ops, alignments (buffers shifted off the 16-byte grid) and in-place
forms drawn at random, every result compared with the oracle element by
element, every output's guard bands checked."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import GUARD, Guarded, assert_equal, ccl, to_dev, to_host
from oracle import collectives, ring, schedules

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _draw(seed):
    rng = np.random.default_rng(seed)
    p = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 33]))
    n = int(rng.choice([1, 3, p, 17 * p + 5, 4096 + 7, int(rng.integers(1, 200_000))]))
    dtype = str(rng.choice(["f32", "bf16", "i32"]))
    shift = int(rng.integers(0, 2))  # 1: every buffer one element off the 16-byte grid
    return rng, p, n, dtype, shift


def _inputs(dtype, p, n, seed):
    if dtype == "i32":
        return workloads.integer_valued(p, n, seed, lo=-2**31, hi=2**31 - 1, dtype="i32")
    return workloads.normal(p, n, 1.0, seed, dtype=dtype)


def _placed(values, dtype, shift):
    bufs = [Guarded(len(v), dtype, offset=GUARD + shift) for v in values]
    for b, v in zip(bufs, values):
        if len(v):
            b.view.copy_(to_dev(v, dtype))
    return bufs


@pytest.mark.parametrize("seed", range(CASES))
def test_random_allreduce_family(lib, seed):
    rng, p, n, dtype, shift = _draw(seed)
    x = _inputs(dtype, p, n, seed)
    op = str(rng.choice(["sum", "max", "min"]))
    send = _placed(x, dtype, shift)
    in_place = bool(rng.integers(0, 2))
    outs = send if in_place else [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    want, _, _ = ring.ring_allreduce(x, dtype, op)
    lib.ccl_allreduce([b.view for b in send], [o.view for o in outs], op=op)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"AR seed {seed} p={p} n={n} {op} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_reduce_scatter_and_all_gather(lib, seed):
    rng, p, n, dtype, shift = _draw(100 + seed)
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, shift)
    lens = [ln for _, ln in ring.chunk_bounds(p, n)]
    shards = [Guarded(ln, dtype, offset=GUARD + int(rng.integers(0, 2))) for ln in lens]
    want_rs, _ = ring.ring_reduce_scatter(x, dtype, "sum")
    lib.ccl_reduce_scatter([b.view for b in send], [s.view for s in shards])
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], dtype, f"RS seed {seed} p={p} n={n} rank {k}")
        assert shards[k].guards_intact()
    full = [Guarded(n, dtype, offset=GUARD + shift) for _ in range(p)]
    lib.ccl_all_gather([s.view for s in shards], [f.view for f in full])
    want_ag, _ = ring.ring_all_gather(want_rs, dtype)
    for r in range(p):
        assert_equal(to_host(full[r].view), want_ag[r], dtype, f"AG seed {seed} p={p} n={n} rank {r}")
        assert full[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_other_fold_orders(lib, seed):
    rng, p, n, dtype, shift = _draw(200 + seed)
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, shift)
    outs = [Guarded(n, dtype, offset=GUARD + shift) for _ in range(p)]
    choices = ["binomial_tree", "naive", "hierarchical"]
    if p & (p - 1) == 0:
        choices += ["recursive_doubling", "rabenseifner"]
    sched = str(rng.choice(choices))
    if sched == "hierarchical":
        group = int(rng.choice([g for g in range(1, p + 1) if p % g == 0]))
        want, _ = schedules.hierarchical(x, group, dtype)
        lib.ccl_allreduce_hierarchical([b.view for b in send], [o.view for o in outs], group)
    else:
        want, _ = schedules.allreduce(sched, x, dtype)
        lib.ccl_allreduce_schedule([b.view for b in send], [o.view for o in outs], sched)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"{sched} seed {seed} p={p} n={n} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_bf16_wire(lib, seed):
    rng, p, n, _, shift = _draw(300 + seed)
    x = _inputs("bf16", p, n, seed)
    send = _placed(x, "bf16", shift)
    outs = [Guarded(n, "bf16", offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    want, _, _ = ring.ring_allreduce(x, "bf16", wire="bf16")
    lib.ccl_allreduce_bf16_wire([b.view for b in send], [o.view for o in outs])
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], "bf16", f"bf16 wire seed {seed} p={p} n={n} rank {r}")
        assert outs[r].guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_rooted(lib, seed):
    rng, p, n, dtype, shift = _draw(400 + seed)
    x = _inputs(dtype, p, n, seed)
    root = int(rng.integers(0, p))
    send = _placed(x, dtype, shift)
    # broadcast
    outs = [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    lib.ccl_broadcast(send[root].view, [o.view for o in outs], root=root)
    for r, w in enumerate(collectives.broadcast(x, root)):
        assert_equal(to_host(outs[r].view), w, dtype, f"broadcast seed {seed} rank {r}")
        assert outs[r].guards_intact()
    # reduce (the ring's bits on the root)
    red = Guarded(n, dtype, offset=GUARD + shift)
    lib.ccl_reduce([b.view for b in send], red.view, root=root)
    want_root = collectives.reduce_ring(x, root, dtype)[root]
    assert_equal(to_host(red.view), want_root, dtype, f"reduce seed {seed} p={p} n={n}")
    assert red.guards_intact()
    # scatter then gather back
    parts = [Guarded(ln, dtype, offset=GUARD + int(rng.integers(0, 2))) for _, ln in ring.chunk_bounds(p, n)]
    lib.ccl_scatter(send[root].view, [g.view for g in parts], root=root)
    for k, w in enumerate(collectives.scatter(x[root], p)):
        assert_equal(to_host(parts[k].view), w, dtype, f"scatter seed {seed} rank {k}")
        assert parts[k].guards_intact()
    back = Guarded(n, dtype, offset=GUARD + shift)
    lib.ccl_gather([g.view for g in parts], back.view, root=root)
    assert_equal(to_host(back.view), x[root], dtype, f"gather seed {seed}")
    assert back.guards_intact()


@pytest.mark.parametrize("seed", range(CASES))
def test_random_all_to_allv(lib, seed):
    rng = np.random.default_rng(500 + seed)
    p = int(rng.choice([1, 2, 3, 5, 8, 13]))
    row = int(rng.choice([1, 2, 3, 7, 8, 64, 129]))
    dtype = str(rng.choice(["f32", "bf16", "i32"]))
    counts = rng.integers(0, int(rng.choice([2, 9, 300])), size=(p, p))
    send_np = [_inputs(dtype, 1, max(int(counts[s].sum()) * row, 1), seed + s)[0][: int(counts[s].sum()) * row]
               for s in range(p)]
    want = collectives.all_to_allv(send_np, counts, row)
    send = _placed(send_np, dtype, int(rng.integers(0, 2)))
    outs = [Guarded(int(counts[:, d].sum()) * row, dtype, offset=GUARD + int(rng.integers(0, 3))) for d in range(p)]
    lib.ccl_all_to_allv([b.view for b in send], counts, [o.view for o in outs], row)
    for d in range(p):
        assert_equal(to_host(outs[d].view), want[d], dtype, f"a2av seed {seed} p={p} row={row} rank {d}")
        assert outs[d].guards_intact()
    # combine with the transposed counts returns every source's rows
    back = [torch.empty_like(b.view) for b in send]
    lib.ccl_all_to_allv([o.view for o in outs], counts.T.copy(), back, row)
    for s in range(p):
        assert_equal(to_host(back[s]), send_np[s], dtype, f"a2av combine seed {seed} rank {s}")


@pytest.mark.parametrize("seed", range(CASES))
def test_random_moe_route_dispatch_combine(lib, seed):
    from oracle import moe
    rng = np.random.default_rng(600 + seed)
    p = int(rng.choice([1, 2, 3, 4, 8, 16]))
    epr = int(rng.choice([1, 2, 4]))
    E = p * epr
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 5, 33, 300, 1000]))
    h = 128 * int(rng.choice([1, 2, 3, 8]))
    fp8 = bool(rng.integers(0, 2))
    ids = workloads.moe_topk_routing(p, T, k, E, seed=seed)
    if T > 2:
        ids[0][1, 0] = -1  # routes nowhere
    toks = workloads.normal(p, T * h, 1.0, seed + 1, dtype="bf16")
    d_ids = [torch.from_numpy(i).cuda() for i in ids]
    counts = torch.empty(p * p, dtype=torch.int64, device="cuda")
    slots = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(p)]
    lib.ccl_moe_route(d_ids, E, counts, slots)
    flat = [i.reshape(-1) for i in ids]
    want_c, want_s, _ = moe.route(flat, p, E)
    np.testing.assert_array_equal(counts.cpu().numpy().reshape(p, p), want_c)
    for s in range(p):
        np.testing.assert_array_equal(slots[s].cpu().numpy().reshape(-1), want_s[s])
    rows = want_c.sum(axis=0)
    if fp8:
        recv = [torch.empty(int(m), h, dtype=torch.uint8, device="cuda") for m in rows]
        scales = [torch.empty(int(m), h // 128, device="cuda") for m in rows]
    else:
        recv = [torch.empty(int(m), h, dtype=torch.bfloat16, device="cuda") for m in rows]
        scales = None
    rexp = [torch.empty(int(m), dtype=torch.int32, device="cuda") for m in rows]
    lib.ccl_moe_dispatch([to_dev(t, "bf16").view(T, h) for t in toks], d_ids, counts, slots, E, recv, scales,
                         rexp, fp8=fp8)
    w_rows, w_scales, w_exp, _, _ = moe.dispatch(toks, flat, p, k, E, h, fp8=fp8)
    for d in range(p):
        got = recv[d].cpu()
        got = got.numpy() if fp8 else got.view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, w_rows[d], err_msg=f"dispatch seed {seed} rank {d}")
        np.testing.assert_array_equal(rexp[d].cpu().numpy(), w_exp[d])
        if fp8:
            np.testing.assert_array_equal(scales[d].cpu().numpy(), w_scales[d])
    y = [workloads.normal(1, max(int(m) * h, 1), 1.0, seed + 10 + d, dtype="bf16")[0][: int(m) * h].reshape(int(m), h)
         for d, m in enumerate(rows)]
    gw = workloads.moe_gate_weights(p, T, k, seed=seed + 2)
    out = [torch.empty(T, h, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    lib.ccl_moe_combine([to_dev(v.reshape(-1), "bf16").view(-1, h) for v in y], d_ids,
                        [torch.from_numpy(w).cuda() for w in gw], counts, slots, E, out)
    want_out = moe.combine(y, flat, gw, p, k, E, h)
    for s in range(p):
        np.testing.assert_array_equal(out[s].cpu().view(torch.int16).numpy().view(np.uint16).reshape(-1),
                                      want_out[s], err_msg=f"combine seed {seed} rank {s}")


@pytest.mark.parametrize("seed", range(CASES))
def test_random_ulysses(lib, seed):
    rng = np.random.default_rng(700 + seed)
    p = int(rng.choice([1, 2, 4, 8]))
    H = p * int(rng.choice([1, 2, 3]))
    D = int(rng.choice([1, 3, 8, 64, 128]))
    sp = int(rng.choice([1, 7, 64, 129]))
    dtype = str(rng.choice(["f32", "bf16"]))
    n = sp * H * D
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, int(rng.integers(0, 2)))
    outs = [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    lib.ccl_all_to_all_heads([b.view for b in send], [o.view for o in outs], sp, H, D)
    want = collectives.ulysses_seq_to_heads(x, H, D)
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"Ulysses seed {seed} p={p} H={H} D={D} sp={sp}")
        assert outs[r].guards_intact()
    back = [Guarded(n, dtype, offset=GUARD) for _ in range(p)]
    lib.ccl_all_to_all_heads([o.view for o in outs], [b.view for b in back], sp, H, D, inverse=True)
    for r in range(p):
        assert_equal(to_host(back[r].view), x[r], dtype, f"Ulysses inverse seed {seed} rank {r}")


@pytest.mark.parametrize("seed", range(CASES))
def test_random_literal_engine(lib, seed):
    """The 2(p-1)-step engine: bits and per-rank byte counters against the
    literal simulation, for all-reduce, reduce-scatter and all-gather."""
    rng, p, n, dtype, shift = _draw(800 + seed)
    op = str(rng.choice(["sum", "max", "min"]))
    x = _inputs(dtype, p, n, seed)
    send = _placed(x, dtype, shift)
    outs = [Guarded(n, dtype, offset=GUARD + int(rng.integers(0, 2))) for _ in range(p)]
    sent = lib.ccl_ring_allreduce_literal([b.view for b in send], [o.view for o in outs], op=op)
    want, rs_b, ag_b = ring.ring_allreduce(x, dtype, op)
    assert list(sent) == [a + b for a, b in zip(rs_b, ag_b)]
    for r in range(p):
        assert_equal(to_host(outs[r].view), want[r], dtype, f"literal AR seed {seed} p={p} n={n} {op} rank {r}")
        assert outs[r].guards_intact()
    shards = [Guarded(ln, dtype, offset=GUARD + shift) for _, ln in ring.chunk_bounds(p, n)]
    sent_rs = lib.ccl_ring_reduce_scatter_literal([b.view for b in send], [s.view for s in shards], op=op)
    want_rs, rs_only = ring.ring_reduce_scatter(x, dtype, op)
    assert list(sent_rs) == list(rs_only)
    for k in range(p):
        assert_equal(to_host(shards[k].view), want_rs[k], dtype, f"literal RS seed {seed} rank {k}")
        assert shards[k].guards_intact()
    full = [Guarded(n, dtype, offset=GUARD) for _ in range(p)]
    sent_ag = lib.ccl_ring_all_gather_literal([s.view for s in shards], [f.view for f in full])
    want_ag, ag_only = ring.ring_all_gather(want_rs, dtype)
    assert list(sent_ag) == list(ag_only)
    for r in range(p):
        assert_equal(to_host(full[r].view), want_ag[r], dtype, f"literal AG seed {seed} rank {r}")
        assert full[r].guards_intact()
