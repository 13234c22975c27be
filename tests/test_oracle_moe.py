"""Pins for the MoE routing / dispatch / combine oracle and its e4m3 encoder."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from a2a_ring_ordered_gb300 import workloads
from oracle import moe
from oracle.bf16 import bf16_to_f32


def _torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    vals = [0.0, -0.0, 2.0**-9, 1.5 * 2.0**-9, 2.5 * 2.0**-9, 2.0**-6, 448.0, 460.0, 464.0,
            1.0625, 1.1875, 3.0, -7.5, 2.0**-10, 0.75 * 2.0**-6]
    # every code, its neighbours' midpoints (ties) and random values up to 464
    codes = np.arange(256, dtype=np.uint8)
    dec = moe.e4m3_to_f32(codes)
    fin = np.sort(np.unique(dec[np.isfinite(dec)]))
    mids = ((fin[1:].astype(np.float64) + fin[:-1]) / 2).astype(np.float32)
    x = np.concatenate([np.array(vals, np.float32), fin, mids, -mids,
                        rng.uniform(-464, 464, 100_000).astype(np.float32),
                        rng.uniform(-0.05, 0.05, 100_000).astype(np.float32)])
    np.testing.assert_array_equal(moe.f32_to_e4m3(x), _torch_e4m3(x))


def test_e4m3_decode_matches_torch_and_round_trips():
    codes = np.arange(256, dtype=np.uint8)
    t = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    d = moe.e4m3_to_f32(codes)
    np.testing.assert_array_equal(np.isnan(d), np.isnan(t))
    ok = ~np.isnan(d)
    np.testing.assert_array_equal(d[ok], t[ok])
    np.testing.assert_array_equal(moe.f32_to_e4m3(d[ok]) & 0x7F, codes[ok] & 0x7F)


def test_e4m3_saturates_instead_of_nan():
    """Beyond 464 torch's cast gives NaN; the satfinite conversion clamps."""
    assert moe.f32_to_e4m3(np.array([500.0, -1e30, np.inf], np.float32)).tolist() == [0x7E, 0xFE, 0x7E]
    assert moe.f32_to_e4m3(np.array([np.nan], np.float32))[0] == 0x7F


def _routing(p, T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = []
    for _ in range(p):
        w = rng.gumbel(size=(T, E)) + np.log((np.arange(E) + 1.0) ** -1.2)
        ids.append(np.argsort(-w, axis=1)[:, :k].astype(np.int32).reshape(-1))  # k distinct experts
    return ids


def test_route_slots_are_stable_ranks():
    p, T, k, E = 4, 50, 3, 16
    ids = _routing(p, T, k, E, 1)
    ids[2][7] = 99  # out of range: routes nowhere
    counts, slots, dests = moe.route(ids, p, E)
    for s in range(p):
        for d in range(p):
            sel = np.flatnonzero(dests[s] == d)
            np.testing.assert_array_equal(slots[s][sel], np.arange(sel.size))
            assert counts[s][d] == sel.size
    assert slots[2][7] == -1 and counts[2].sum() == T * k - 1


def test_dispatch_places_every_row_by_brute_force():
    p, T, k, E, h = 3, 20, 2, 6, 128
    ids = _routing(p, T, k, E, 2)
    toks = [workloads.to_bf16_bits(np.repeat(np.arange(T, dtype=np.float32) + 100 * s, h)) for s in range(p)]
    recv, _, rexp, counts, _ = moe.dispatch(toks, ids, p, k, E, h)
    for d in range(p):
        expect = []
        for s in range(p):
            for t in range(T):
                for j in range(k):
                    if ids[s][t * k + j] // (E // p) == d:
                        expect.append((100 * s + t, ids[s][t * k + j]))
        assert len(expect) == recv[d].shape[0]
        for r, (val, e) in enumerate(expect):
            assert (bf16_to_f32(recv[d][r]) == val).all() and rexp[d][r] == e


@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_combine_of_dispatch_is_identity(k):
    """combine(dispatch(x)) with weights 1/k returns x exactly (bf16 values,
    power-of-two k: every partial sum is exact)."""
    p, T, E, h = 4, 64, 32, 256
    ids = _routing(p, T, k, E, k)
    toks = workloads.normal(p, T * h, 1.0, k, dtype="bf16")
    recv, _, _, _, _ = moe.dispatch(toks, ids, p, k, E, h)
    w = [np.full(T * k, 1.0 / k, np.float32) for _ in range(p)]
    back = moe.combine(recv, ids, w, p, k, E, h)
    for a, b in zip(toks, back):
        np.testing.assert_array_equal(a, b)


def test_combine_weighted_sum_integer_exact():
    p, T, k, E, h = 2, 16, 2, 4, 128
    ids = _routing(p, T, k, E, 5)
    vals = [np.random.default_rng(s).integers(-50, 50, size=(T * k,)) for s in range(p)]
    # expert outputs: each dispatched row replaced by an integer; weights 0.5 and 2
    recv, _, _, counts, slots = moe.dispatch(
        [workloads.to_bf16_bits(np.zeros(T * h, np.float32)) for _ in range(p)], ids, p, k, E, h)
    base = np.vstack([np.zeros((1, p), np.int64), np.cumsum(counts, 0)[:-1]])
    for s in range(p):
        for i in range(T * k):
            d = ids[s][i] // (E // p)
            recv[d][base[s][d] + slots[s][i]] = workloads.to_bf16_bits(np.full(h, vals[s][i], np.float32))
    w = [np.tile(np.array([0.5, 2.0], np.float32), T) for _ in range(p)]
    out = moe.combine(recv, ids, w, p, k, E, h)
    for s in range(p):
        want = 0.5 * vals[s][0::2] + 2.0 * vals[s][1::2]
        got = bf16_to_f32(out[s]).reshape(T, h)
        np.testing.assert_array_equal(got, np.repeat(want[:, None], h, axis=1).astype(np.float32))


def test_fp8_rows_within_half_ulp():
    """Dequantised codes are within half an e4m3 ulp of the input.

    With s the block's scale, v = fl(x / s) = (x / s)(1 + d1), c the e4m3 code
    of v and d = fl(c * s) = c s (1 + d2) (|d1|, |d2| <= u = 2^-24):
    d - x = (c - v) s + x d1 + c s d2.  A normal code is within half an ulp
    of v, |c - v| <= 2^-4 |v|, so |d - x| <= |x| 2^-4 [(1 + u) + 16u +
    17u(1 + u)] <= |x| 2^-4 (1 + 34u).  A subnormal code is within 2^-10 of
    v and |x| < 2^-6 s (1 + u), so |d - x| <= 2^-10 s (1 + 33u).  Saturation
    at 448 moves v by at most 3u * 448.  The check runs in float64 so that
    its own arithmetic adds no rounding."""
    p, T, k, E, h = 2, 32, 2, 4, 256
    slack = 34 * 2.0**-24
    ids = _routing(p, T, k, E, 6)
    toks = workloads.normal(p, T * h, 3.0, 6, dtype="bf16")
    recv, scales, _, counts, slots = moe.dispatch(toks, ids, p, k, E, h, fp8=True)
    base = np.vstack([np.zeros((1, p), np.int64), np.cumsum(counts, 0)[:-1]])
    for s in range(p):
        x = bf16_to_f32(toks[s]).reshape(T, h).astype(np.float64)
        for i in range(T * k):
            d = ids[s][i] // (E // p)
            pos = base[s][d] + slots[s][i]
            sc = scales[d][pos].astype(np.float64)[:, None]
            deq = (moe.e4m3_to_f32(recv[d][pos]).reshape(-1, 128) * scales[d][pos][:, None]).astype(np.float64)
            xb = x[i // k].reshape(-1, 128)
            err = np.abs(deq - xb)
            bound = np.maximum(np.abs(xb) * 2.0**-4, sc * 2.0**-10) * (1 + slack)
            assert (err <= bound).all()
            amax = np.abs(xb).max(axis=1).astype(np.float32)
            np.testing.assert_array_equal(scales[d][pos], (amax / np.float32(448)).astype(np.float32))


def test_fp8_codes_are_the_e4m3_of_x_over_scale():
    """The block's codes are torch's e4m3 cast of torch's fp32 quotient x / s
    (both correctly rounded; |x / s| stays at or below 448 (1 + 2u), which
    rounds to 448, so torch's cast never reaches its NaN range); an all-zero
    block has scale 1 and zero codes; the largest magnitude maps to +-448."""
    rng = np.random.default_rng(11)
    rows = (rng.standard_normal((64, 512)) * rng.uniform(1e-3, 50.0, (64, 1))).astype(np.float32)
    rows[3] = 0.0
    rows[5, :128] = 0.0
    rows[7, 200] = -1e4  # one large outlier in block 1
    codes, scales = moe.quantize_rows_fp8(rows)
    xb = torch.from_numpy(rows.reshape(64, 4, 128))
    sc = torch.from_numpy(scales)[:, :, None]
    want = (xb / sc).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(64, 512)
    np.testing.assert_array_equal(codes, want)
    assert (scales[3] == 1.0).all() and (codes[3] == 0).all() and scales[5, 0] == 1.0
    blocks = np.abs(rows.reshape(64, 4, 128))
    at_max = blocks == blocks.max(axis=2, keepdims=True)
    nz = blocks.max(axis=2, keepdims=True) > 0
    assert ((codes.reshape(64, 4, 128) & 0x7F)[at_max & nz] == 0x7E).all()
