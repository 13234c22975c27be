"""GPU parity of the MoE routing, dispatch (bf16 / FP8) and combine kernels."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from gpu_util import ccl, to_dev, to_host
from oracle import moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _run(lib, p, T, k, E, h, fp8, seed=0, bad_id=False):
    ids = workloads.moe_topk_routing(p, T, k, E, seed=seed)
    if bad_id:
        ids[p - 1][T // 2, 0] = E + 5
    toks = workloads.normal(p, T * h, 1.0, seed, dtype="bf16")
    d_ids = [torch.from_numpy(i).cuda() for i in ids]
    d_x = [to_dev(t, "bf16").view(T, h) for t in toks]
    counts = torch.empty(p * p, dtype=torch.int64, device="cuda")
    slots = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(p)]
    lib.ccl_moe_route(d_ids, E, counts, slots)
    c = counts.cpu().numpy().reshape(p, p)
    rows = c.sum(axis=0)
    if fp8:
        recv = [torch.empty(int(m), h, dtype=torch.uint8, device="cuda") for m in rows]
        scales = [torch.empty(int(m), h // 128, dtype=torch.float32, device="cuda") for m in rows]
    else:
        recv = [torch.empty(int(m), h, dtype=torch.bfloat16, device="cuda") for m in rows]
        scales = None
    rexp = [torch.full((int(m),), -7, dtype=torch.int32, device="cuda") for m in rows]
    lib.ccl_moe_dispatch(d_x, d_ids, counts, slots, E, recv, scales, rexp, fp8=fp8)
    torch.cuda.synchronize()
    return ids, toks, d_ids, counts, c, slots, recv, scales, rexp


# items = T * k: one 4096-item tile and under; 8 tiles (a cluster of 8 CTAs per
# source, one tile each); 35,000 (9 tiles: two-tile segments, the last CTAs
# empty, a ragged last tile); 200,000 (seven-tile segments); none at all
@pytest.mark.parametrize("p,T,k,E", [(1, 10, 1, 4), (2, 300, 2, 8), (4, 1000, 4, 16), (8, 777, 8, 64),
                                     (16, 200, 3, 32), (64, 50, 2, 128), (8, 4096, 8, 256),
                                     (5, 7000, 5, 10), (2, 100000, 2, 8), (4, 0, 2, 8)])
def test_route_matches_oracle(lib, p, T, k, E):
    ids = workloads.moe_topk_routing(p, T, k, E, seed=p)
    if T:
        ids[0][0, 0] = -1  # routes nowhere
    want_c, want_s, _ = moe.route([i.reshape(-1) for i in ids], p, E)
    counts = torch.empty(p * p, dtype=torch.int64, device="cuda")
    slots = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(p)]
    lib.ccl_moe_route([torch.from_numpy(i).cuda() for i in ids], E, counts, slots)
    np.testing.assert_array_equal(counts.cpu().numpy().reshape(p, p), want_c)
    for s in range(p):
        np.testing.assert_array_equal(slots[s].cpu().numpy().reshape(-1), want_s[s])


# h = 7168 (the DeepSeek-V3 hidden size): 8 tokens per CTA for dispatch, 2 for
# combine; T = 37 leaves a short last CTA
@pytest.mark.parametrize("p,T,k,E,h", [(2, 100, 2, 8, 128), (4, 500, 4, 16, 256), (8, 1024, 8, 64, 4096),
                                       (8, 37, 8, 256, 7168)])
def test_dispatch_bf16_matches_oracle(lib, p, T, k, E, h):
    ids, toks, *_, recv, _, rexp = _run(lib, p, T, k, E, h, fp8=False, seed=1, bad_id=True)
    want, _, want_e, _, _ = moe.dispatch(toks, [i.reshape(-1) for i in ids], p, k, E, h)
    for d in range(p):
        np.testing.assert_array_equal(to_host(recv[d]).reshape(-1, h), want[d], err_msg=f"rank {d}")
        np.testing.assert_array_equal(rexp[d].cpu().numpy(), want_e[d])


@pytest.mark.parametrize("p,T,k,E,h", [(2, 100, 2, 8, 128), (8, 512, 8, 64, 4096), (8, 37, 8, 256, 7168)])
def test_dispatch_fp8_matches_oracle(lib, p, T, k, E, h):
    ids, toks, *_, recv, scales, _ = _run(lib, p, T, k, E, h, fp8=True, seed=2)
    want, want_sc, _, _, _ = moe.dispatch(toks, [i.reshape(-1) for i in ids], p, k, E, h, fp8=True)
    for d in range(p):
        np.testing.assert_array_equal(recv[d].cpu().numpy(), want[d], err_msg=f"codes rank {d}")
        np.testing.assert_array_equal(scales[d].cpu().numpy(), want_sc[d], err_msg=f"scales rank {d}")


@pytest.mark.parametrize("p,T,k,E,h", [(2, 100, 2, 8, 128), (4, 300, 3, 16, 256), (8, 512, 8, 64, 4096),
                                       (8, 37, 8, 256, 7168), (3, 5, 16, 48, 384)])
def test_combine_matches_oracle_and_inverts_dispatch(lib, p, T, k, E, h):
    ids, toks, d_ids, counts, c, slots, recv, _, _ = _run(lib, p, T, k, E, h, fp8=False, seed=3)
    w = workloads.moe_gate_weights(p, T, k, seed=5)
    # expert outputs: a fresh bf16 array in dispatch layout
    ys = [workloads.normal(1, int(r.shape[0]) * h, 1.0, 10 + d, dtype="bf16")[0] for d, r in enumerate(recv)]
    d_y = [to_dev(y, "bf16").view(-1, h) for y in ys]
    out = [torch.empty(T, h, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    lib.ccl_moe_combine(d_y, d_ids, [torch.from_numpy(x).cuda() for x in w], counts, slots, E, out)
    want = moe.combine([y.reshape(-1, h) for y in ys], [i.reshape(-1) for i in ids],
                       [x.reshape(-1) for x in w], p, k, E, h)
    for s in range(p):
        np.testing.assert_array_equal(to_host(out[s]).reshape(-1), want[s], err_msg=f"combine {s}")
    if k & (k - 1) == 0:  # weights 1/k: combine(dispatch(x)) == x
        ones = [torch.full((T, k), 1.0 / k, device="cuda") for _ in range(p)]
        lib.ccl_moe_combine(recv, d_ids, ones, counts, slots, E, out)
        for s in range(p):
            np.testing.assert_array_equal(to_host(out[s]).reshape(-1), toks[s], err_msg=f"identity {s}")


def test_dispatch_never_writes_past_a_short_buffer(lib):
    """A receive buffer smaller than its count: rows past the capacity are
    dropped, the guard band after the buffer stays intact."""
    p, T, k, E, h = 2, 64, 2, 4, 128
    ids = workloads.moe_topk_routing(p, T, k, E, seed=9)
    d_ids = [torch.from_numpy(i).cuda() for i in ids]
    x = [to_dev(t, "bf16").view(T, h) for t in workloads.normal(p, T * h, 1.0, 9, dtype="bf16")]
    counts = torch.empty(p * p, dtype=torch.int64, device="cuda")
    slots = [torch.empty(T, k, dtype=torch.int32, device="cuda") for _ in range(p)]
    lib.ccl_moe_route(d_ids, E, counts, slots)
    rows = counts.cpu().numpy().reshape(p, p).sum(axis=0)
    store = [torch.full((int(m) + 16, h), 3.0, dtype=torch.bfloat16, device="cuda") for m in rows]
    short = [st[: int(m) - 5] for st, m in zip(store, rows)]
    lib.ccl_moe_dispatch(x, d_ids, counts, slots, E, short)
    torch.cuda.synchronize()
    for st, m in zip(store, rows):
        assert (st[int(m) - 5:].float() == 3.0).all()
