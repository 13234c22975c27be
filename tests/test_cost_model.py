"""The alpha-beta cost model against the figures the pages print."""
from __future__ import annotations

import math

import pytest

from a2a_ring_ordered_gb300 import cost_model as cm
from conftest import read_golden

G = {k: v for k, v in read_golden("alpha_beta_pages.txt").items()}
NV = (2e-6, 450e9)  # NVLink alpha, beta used throughout the lecture


def near(key, got):
    want, tol = G[key]
    assert abs(got - want) <= tol + 1e-12, f"{key}: model {got} vs page {want} (+-{tol})"


def test_exercise1_half_bandwidth_point():
    a, b = 5e-6, 50e9
    near("ex1_half_bandwidth_bytes", cm.half_bandwidth_point(a, b))
    near("ex1_time_25KB_us", cm.p2p_time(25e3, a, b) * 1e6)
    near("ex1_bw_25KB_GBs", cm.effective_bandwidth(25e3, a, b) / 1e9)
    near("ex1_time_2_5MB_us", cm.p2p_time(2.5e6, a, b) * 1e6)
    near("ex1_bw_2_5MB_GBs", cm.effective_bandwidth(2.5e6, a, b) / 1e9)


def test_ring_vs_tree_crossover_680KiB():
    a, b, p = 0.822e-6, 450e9, 8
    n = cm.crossover(lambda m: cm.ring_allreduce(p, m, a, b),
                     lambda m: 2 * math.log2(p) * (a + m / b))  # unsegmented tree
    near("ch67_ring_tree_crossover_KiB", n / 1024)


@pytest.mark.parametrize("p,key", [(8, "ex3_rd_ring_crossover_p8_MB"), (16, "ex3_rd_ring_crossover_p16_MB")])
def test_recursive_doubling_vs_ring_crossover(p, key):
    n = cm.crossover(lambda m: cm.recursive_doubling_allreduce(p, m, *NV),
                     lambda m: cm.ring_allreduce(p, m, *NV))
    near(key, n / 1e6)


def test_exercise4_ring_all_gather():
    n = 1024 * 16384 * 2
    near("ex4_ag_bandwidth_us", cm.ring_all_gather(8, n, 0.0, 450e9) * 1e6)
    near("ex4_ag_with_latency_us", cm.ring_all_gather(8, n, *NV) * 1e6)


def test_exercise6_hierarchical():
    h = cm.hierarchical_allreduce(4, 8, 512e6, 0.0, 450e9, 0.0, 50e9)
    near("ex6_intra_rs_ms", h["intra_reduce_scatter"] * 1e3)
    near("ex6_inter_ar_ms", h["inter_allreduce"] * 1e3)
    near("ex6_total_ms", h["total"] * 1e3)
    near("ex6_flat_ring_ms", cm.ring_allreduce(32, 512e6, 0.0, 50e9) * 1e3)


def test_exercise7_tensor_parallel_decode():
    n = 16 * 4096 * 2
    assert n == 131072
    near("ex7_ring_us", cm.ring_allreduce(4, n, *NV) * 1e6)
    near("ex7_rd_us", cm.recursive_doubling_allreduce(4, n, *NV) * 1e6)
    near("ex7_ring_x64_ms", 64 * cm.ring_allreduce(4, n, *NV) * 1e3)
    near("ex7_rd_x64_ms", 64 * cm.recursive_doubling_allreduce(4, n, *NV) * 1e3)


def test_exercise9_pipelined_chain_broadcast():
    a, b = 1e-6, 45e9
    near("ex9_optimal_chunks", cm.optimal_chain_chunks(8, 8e6, a, b))
    near("ex9_optimal_time_us", cm.optimal_chain_broadcast(8, 8e6, a, b) * 1e6)
    near("ex9_time_k32_us", cm.chain_broadcast(8, 8e6, 32, a, b) * 1e6)
    # the closed-form optimum is the minimum over integer k
    best = min(cm.chain_broadcast(8, 8e6, k, a, b) for k in range(1, 200))
    assert cm.optimal_chain_broadcast(8, 8e6, a, b) <= best + 1e-12


def test_section42_broadcast_algorithms():
    near("s42_binomial_32KB_us", cm.binomial_broadcast(8, 32 * 1024, *NV) * 1e6)
    near("s42_binomial_8MB_us", cm.binomial_broadcast(8, 8 * 2**20, *NV) * 1e6)
    # the page's qualitative result: scatter + all-gather loses at 32 KB, wins at 8 MB
    assert cm.scatter_allgather_broadcast(8, 32 * 1024, *NV) > cm.binomial_broadcast(8, 32 * 1024, *NV)
    assert cm.scatter_allgather_broadcast(8, 8 * 2**20, *NV) < cm.binomial_broadcast(8, 8 * 2**20, *NV)


def test_sections53_54_latency_terms():
    near("s53_ring_latency_us", cm.ring_allreduce(8, 0.0, *NV) * 1e6)
    a, b = 5e-6, 50e9
    assert cm.ring_allreduce(512, 64e3, a, b) * 1e3 > G["s54_ring_64KB_p512_ms_at_least"][0]
    near("s54_rd_64KB_p512_us", cm.recursive_doubling_allreduce(512, 64e3, a, b) * 1e6)


def test_section56_effective_alpha():
    """busbw = 150 GB/s at 58 MB on 8 GPUs -> solve the ring model for alpha."""
    p, n, b = 8, 58e6, 450e9
    t = n / (150e9 * p / (2 * (p - 1)))  # busbw = algbw * 2(p-1)/p, algbw = n / t
    alpha = (t - 2 * (p - 1) * n / (p * b)) / (2 * (p - 1))
    near("s56_effective_alpha_us", alpha * 1e6)
    assert abs(cm.bus_bandwidth(n / cm.ring_allreduce(p, n, alpha, b), p) - 150e9) < 1e3


def test_bandwidth_terms_match_the_byte_lower_bounds():
    """Ring and Rabenseifner move 2(p-1)/p n per device (section 4.3): their
    alpha-free times equal that over beta; recursive doubling moves log2 p n."""
    for p in (2, 4, 8, 16):
        n, b = 1e9, 1e11
        assert math.isclose(cm.ring_allreduce(p, n, 0.0, b), 2 * (p - 1) / p * n / b)
        assert math.isclose(cm.rabenseifner_allreduce(p, n, 0.0, b), 2 * (p - 1) / p * n / b)
        assert math.isclose(cm.recursive_doubling_allreduce(p, n, 0.0, b), math.log2(p) * n / b)


def test_cheapest_allreduce_follows_message_size():
    assert cm.cheapest_allreduce(8, 1e3, *NV)[0] in ("naive", "recursive_doubling")
    assert cm.cheapest_allreduce(8, 1e9, *NV)[0] in ("ring", "rabenseifner")
    assert cm.cheapest_allreduce(6, 1e9, *NV)[0] == "ring"  # no power-of-two algorithms at p=6
