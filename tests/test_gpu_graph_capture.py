"""Every entry point can be captured into a CUDA graph and replayed: the
calls only enqueue kernels on the given stream (the bench times replayed
graphs, and training loops capture their collectives).  Each replay's
results are compared with the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import assert_equal, ccl, to_dev, to_host
from oracle import collectives, moe, ring, schedules

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _capture(fn):
    """Warm up once, capture fn on a side stream, return the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    torch.cuda.synchronize()
    return g


def test_reductions_and_copies_replay(lib):
    p, n = 6, 70_001
    x = workloads.normal(p, n, 1.0, 41)
    xb = workloads.normal(p, n, 1.0, 42, dtype="bf16")
    send = [to_dev(v, "f32") for v in x]
    sendb = [to_dev(v, "bf16") for v in xb]
    ar = [torch.empty(n, device="cuda") for _ in range(p)]
    lens = [ln for _, ln in ring.chunk_bounds(p, n)]
    rs = [torch.empty(ln, dtype=torch.bfloat16, device="cuda") for ln in lens]
    ag = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    hier = [torch.empty(n, device="cuda") for _ in range(p)]
    naive = [torch.empty(n, device="cuda") for _ in range(p)]
    wire = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    bc = [torch.empty(n, device="cuda") for _ in range(p)]

    def step(s):
        lib.ccl_allreduce(send, ar, stream=s)
        lib.ccl_reduce_scatter(sendb, rs, stream=s)
        lib.ccl_all_gather(rs, ag, stream=s)
        lib.ccl_allreduce_hierarchical(send, hier, 3, stream=s)
        lib.ccl_allreduce_schedule(send, naive, "naive", stream=s)
        lib.ccl_allreduce_bf16_wire(sendb, wire, stream=s)
        lib.ccl_broadcast(send[2], bc, root=2, stream=s)

    g = _capture(step)
    for t in ar + hier + naive + bc:
        t.zero_()
    for t in ag + wire:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    want_ar, _, _ = ring.ring_allreduce(x)
    want_rs, _ = ring.ring_reduce_scatter(xb, "bf16")
    want_ag, _ = ring.ring_all_gather(want_rs, "bf16")
    want_h, _ = schedules.hierarchical(x, 3)
    want_n, _ = schedules.naive(x)
    want_w, _, _ = ring.ring_allreduce(xb, "bf16", wire="bf16")
    for r in range(p):
        assert_equal(to_host(ar[r]), want_ar[r], "f32", f"AR rank {r}")
        assert_equal(to_host(ag[r]), want_ag[r], "bf16", f"AG rank {r}")
        assert_equal(to_host(hier[r]), want_h[r], "f32", f"hierarchical rank {r}")
        assert_equal(to_host(naive[r]), want_n[r], "f32", f"naive rank {r}")
        assert_equal(to_host(wire[r]), want_w[r], "bf16", f"bf16 wire rank {r}")
        assert_equal(to_host(bc[r]), x[2], "f32", f"broadcast rank {r}")
    for k in range(p):
        assert_equal(to_host(rs[k]), want_rs[k], "bf16", f"RS rank {k}")


def test_all_to_allv_moe_and_ulysses_replay(lib):
    p, row = 5, 7
    rng = np.random.default_rng(43)
    counts = rng.integers(0, 40, size=(p, p))
    xa = [workloads.normal(1, int(counts[s].sum()) * row, 1.0, 50 + s, dtype="bf16")[0] for s in range(p)]
    sa = [to_dev(v, "bf16") for v in xa]
    ra = [torch.empty(int(counts[:, d].sum()) * row, dtype=torch.bfloat16, device="cuda") for d in range(p)]

    P, T, k, E, h = 4, 100, 4, 16, 256
    ids = workloads.moe_topk_routing(P, T, k, E, seed=44)
    toks = workloads.normal(P, T * h, 1.0, 45, dtype="bf16")
    d_ids = [torch.from_numpy(i).cuda() for i in ids]
    d_x = [to_dev(t, "bf16").view(T, h) for t in toks]
    counts_m = torch.empty(P * P, dtype=torch.int64, device="cuda")
    slots = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(P)]
    lib.ccl_moe_route(d_ids, E, counts_m, slots)  # sizes the receive buffers once
    rows = counts_m.cpu().numpy().reshape(P, P).sum(axis=0)
    q = [torch.empty(int(m), h, dtype=torch.uint8, device="cuda") for m in rows]
    sc = [torch.empty(int(m), h // 128, device="cuda") for m in rows]

    sp, H, D = 16, 8, 64
    xu = workloads.normal(4, sp * H * D, 1.0, 46, dtype="bf16")
    su = [to_dev(v, "bf16") for v in xu]
    ru = [torch.empty_like(t) for t in su]
    rt = [torch.empty_like(t) for t in su]

    def step(s):
        lib.ccl_all_to_allv(sa, counts, ra, row, stream=s)
        lib.ccl_moe_route(d_ids, E, counts_m, slots, stream=s)
        lib.ccl_moe_dispatch(d_x, d_ids, counts_m, slots, E, q, sc, fp8=True, stream=s)
        lib.ccl_all_to_all_heads(su, ru, sp, H, D, stream=s)
        lib.ccl_all_to_all(su, rt, stream=s)

    g = _capture(step)
    for t in ra + q + sc + ru + rt:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for d, w in enumerate(collectives.all_to_allv(xa, counts, row)):
        assert_equal(to_host(ra[d]), w, "bf16", f"a2av rank {d}")
    w_q, w_sc, _, _, _ = moe.dispatch(toks, [i.reshape(-1) for i in ids], P, k, E, h, fp8=True)
    for d in range(P):
        np.testing.assert_array_equal(q[d].cpu().numpy(), w_q[d])
        np.testing.assert_array_equal(sc[d].cpu().numpy(), w_sc[d])
    for r, w in enumerate(collectives.ulysses_seq_to_heads(xu, H, D)):
        assert_equal(to_host(ru[r]), w, "bf16", f"Ulysses rank {r}")
    for r, w in enumerate(collectives.all_to_all(xu)):
        assert_equal(to_host(rt[r]), w, "bf16", f"all-to-all rank {r}")
