"""Buffers past 32-bit indexing: more than 2^31 elements per rank and block
offsets past 2^32 bytes.  The kernels index in 64 bits; these cases would
catch a 32-bit index or byte offset anywhere on the path.  Inputs are drawn on
the device by torch's seeded generator; sampled outputs are checked against
the oracle (the pointwise ring fold, the chunk rule), and AG(RS) == AR is
checked on every element."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import assert_equal, ccl, sample_indices, to_host
from oracle import pointwise, ring

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ccl()


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_allreduce_reduce_scatter_all_gather_past_2_31_elements(lib):
    p, n = 3, (1 << 31) + (1 << 20) + 7  # 4.3 GB of bf16 per rank; ragged chunk edges
    idx = sample_indices(n, p, 1 << 18, seed=31)
    idx_t = torch.from_numpy(idx).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(31)
    send, cols = [], []
    for _ in range(p):
        v = (torch.rand(n, generator=gen, device="cuda", dtype=torch.float32) * 2.0 - 1.0).to(torch.bfloat16)
        cols.append(to_host(v[idx_t]))
        send.append(v)
    want = pointwise.allreduce_at_columns(cols, idx, n, "bf16")

    recv = [torch.empty_like(s) for s in send]
    lib.ccl_allreduce(send, recv)
    for r in range(p):
        assert_equal(to_host(recv[r][idx_t]), want, "bf16", f"AR rank {r}")

    bounds = ring.chunk_bounds(p, n)
    shards = [torch.empty(ln, dtype=torch.bfloat16, device="cuda") for _, ln in bounds]
    lib.ccl_reduce_scatter(send, shards)
    for k, (off, ln) in enumerate(bounds):
        sel = (idx >= off) & (idx < off + ln)
        local = torch.from_numpy(idx[sel] - off).cuda()
        assert_equal(to_host(shards[k][local]), want[sel], "bf16", f"RS rank {k}")
    del send
    _free()

    out = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    lib.ccl_all_gather(shards, out)
    for r in range(p):  # AG(RS) == AR, every element
        assert torch.equal(out[r].view(torch.int16), recv[0].view(torch.int16)), f"AG(RS) rank {r}"
    del recv, shards, out
    _free()


def test_all_to_all_past_4_gib_offsets(lib):
    p, n = 2, (1 << 31) + 12_345  # fp32: 8.6 GB per rank, rank 1's block starts past 2^32 bytes
    gen = torch.Generator(device="cuda")
    gen.manual_seed(32)
    send = [torch.rand(n, generator=gen, device="cuda", dtype=torch.float32) for _ in range(p)]
    bounds = ring.chunk_bounds(p, n)
    recv = [torch.empty(p * ln, device="cuda") for _, ln in bounds]
    lib.ccl_all_to_all(send, recv)
    rng = np.random.default_rng(33)
    for j, (off, ln) in enumerate(bounds):
        # recv[j] = block j of send[0], then block j of send[1] (chunk rule)
        pos = np.unique(np.concatenate([rng.integers(0, p * ln, size=1 << 16),
                                        [0, ln - 1, ln, p * ln - 1]]))
        src_rank, src_idx = pos // ln, off + pos % ln
        want = np.empty(pos.size, dtype=np.float32)
        for s in range(p):
            sel = src_rank == s
            want[sel] = to_host(send[s][torch.from_numpy(src_idx[sel]).cuda()])
        assert_equal(to_host(recv[j][torch.from_numpy(pos).cuda()]), want, "f32", f"A2A rank {j}")
    del send, recv
    _free()


def test_all_to_allv_row_prefixes_past_32_bits(lib):
    """A source with more than 2^32 rows: the row-prefix table takes 64-bit
    entries.  p = 2, one-element bf16 rows, source 0 sends 2^31 + 5 rows to
    destination 0 and 2^31 + 7 to destination 1 (8.6 GB), source 1 three and
    two rows.  Sampled received rows (every block edge included) against the
    oracle's placement (oracle.pointwise.all_to_allv_source), and every
    block equal to its source slice on the device."""
    from oracle import pointwise
    p = 2
    counts = np.array([[(1 << 31) + 5, (1 << 31) + 7], [3, 2]], dtype=np.int64)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(34)
    send = [(torch.rand(int(counts[s].sum()), generator=gen, device="cuda") * 2 - 1).to(torch.bfloat16)
            for s in range(p)]
    recv = [torch.empty(int(counts[:, d].sum()), dtype=torch.bfloat16, device="cuda") for d in range(p)]
    lib.ccl_all_to_allv(send, counts, recv, 1)
    rng = np.random.default_rng(35)
    for d in range(p):
        total = int(counts[:, d].sum())
        starts = np.concatenate([[0], np.cumsum(counts[:, d])])
        rows = np.unique(np.concatenate([rng.integers(0, total, size=1 << 16), starts[:-1], starts[1:] - 1]))
        rows = rows[rows < total]
        src, srow = pointwise.all_to_allv_source(counts, d, rows)
        want = np.empty(rows.size, dtype=np.uint16)
        for s in range(p):
            sel = src == s
            want[sel] = to_host(send[s][torch.from_numpy(srow[sel]).cuda()])
        assert_equal(to_host(recv[d][torch.from_numpy(rows).cuda()]), want, "bf16", f"a2av rank {d}")
    # whole blocks on the device
    a, b = int(counts[0, 0]), int(counts[0, 1])
    assert torch.equal(recv[0][:a].view(torch.int16), send[0][:a].view(torch.int16))
    assert torch.equal(recv[0][a:].view(torch.int16), send[1][:3].view(torch.int16))
    assert torch.equal(recv[1][:b].view(torch.int16), send[0][a:].view(torch.int16))
    assert torch.equal(recv[1][b:].view(torch.int16), send[1][3:].view(torch.int16))
    del send, recv
    _free()
