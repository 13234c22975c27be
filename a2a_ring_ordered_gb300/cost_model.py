"""alpha-beta (Hockney) cost model of the collective algorithms.

"Networks and Collective Communication" section 2.1 and "dist_train",
Communication Cost Model: sending n bytes costs T = alpha + n / beta, with
alpha the start-up latency and beta the link bandwidth (bytes per second);
the half-bandwidth point n_1/2 = alpha * beta separates latency-dominated
from bandwidth-dominated messages.  Section 5 of the former gives each
all-reduce algorithm's time; section 5.5 and Exercise 9 the pipelined chain
broadcast; section 6.3 and Exercise 6 the hierarchical all-reduce.

These are models of networks, used to choose a schedule by message size the
way collective libraries do; the single-GPU kernels of this package are bound
by HBM, not by these terms.  All sizes are in bytes, times in seconds.
"""
from __future__ import annotations

import math

__all__ = [
    "p2p_time", "half_bandwidth_point", "effective_bandwidth",
    "ring_allreduce", "recursive_doubling_allreduce", "rabenseifner_allreduce",
    "binary_tree_allreduce", "naive_allreduce", "in_network_allreduce",
    "ring_all_gather", "binomial_broadcast", "scatter_allgather_broadcast",
    "chain_broadcast", "optimal_chain_chunks", "optimal_chain_broadcast",
    "hierarchical_allreduce", "crossover", "bus_bandwidth", "ALLREDUCE_MODELS",
    "cheapest_allreduce",
]


def p2p_time(n: float, alpha: float, beta: float) -> float:
    """One message of n bytes: alpha + n / beta."""
    return alpha + n / beta


def half_bandwidth_point(alpha: float, beta: float) -> float:
    """n_1/2 = alpha * beta: the size at which latency and transfer time are equal."""
    return alpha * beta


def effective_bandwidth(n: float, alpha: float, beta: float) -> float:
    """Bytes per second actually obtained for one n-byte message."""
    return n / p2p_time(n, alpha, beta)


def ring_allreduce(p: int, n: float, alpha: float, beta: float) -> float:
    """2(p-1) steps of n/p bytes each: 2(p-1)(alpha + n/(p beta))."""
    return 2 * (p - 1) * (alpha + n / (p * beta))


def recursive_doubling_allreduce(p: int, n: float, alpha: float, beta: float) -> float:
    """log2 p steps, each exchanging the whole vector: log2 p (alpha + n/beta)."""
    return math.log2(p) * (alpha + n / beta)


def rabenseifner_allreduce(p: int, n: float, alpha: float, beta: float) -> float:
    """Recursive-halving reduce-scatter + doubling all-gather:
    2 log2 p alpha + 2 (p-1)/p n / beta."""
    return 2 * math.log2(p) * alpha + 2 * (p - 1) / p * n / beta


def binary_tree_allreduce(p: int, n: float, alpha: float, beta: float) -> float:
    """Binomial-tree reduce then broadcast: 2 ceil(log2 p) (alpha + n/beta)."""
    return 2 * math.ceil(math.log2(p)) * (alpha + n / beta)


def naive_allreduce(p: int, n: float, alpha: float, beta: float) -> float:
    """Everyone to the root and back: 2 (alpha + (p-1) n / beta)."""
    return 2 * (alpha + (p - 1) * n / beta)


def in_network_allreduce(n: float, alpha: float, beta: float) -> float:
    """Switch-side reduction with up/down pipelining: about alpha + n/beta."""
    return alpha + n / beta


def ring_all_gather(p: int, n: float, alpha: float, beta: float) -> float:
    """Ring all-gather of an n-byte result: (p-1)(alpha + n/(p beta))."""
    return (p - 1) * (alpha + n / (p * beta))


def binomial_broadcast(p: int, n: float, alpha: float, beta: float) -> float:
    """ceil(log2 p) rounds, each forwarding the whole message."""
    return math.ceil(math.log2(p)) * (alpha + n / beta)


def scatter_allgather_broadcast(p: int, n: float, alpha: float, beta: float) -> float:
    """Van de Geijn: binomial scatter (log2 p rounds, (p-1)/p n bytes) then ring
    all-gather ((p-1) rounds of n/p)."""
    return (math.ceil(math.log2(p)) * alpha + (p - 1) / p * n / beta
            + ring_all_gather(p, n, alpha, beta))


def chain_broadcast(p: int, n: float, k: int, alpha: float, beta: float) -> float:
    """Pipelined chain over p devices in k chunks: (p - 2 + k)(alpha + n/(k beta))."""
    return (p - 2 + k) * (alpha + n / (k * beta))


def optimal_chain_chunks(p: int, n: float, alpha: float, beta: float) -> float:
    """k* = sqrt((p-2) n / (alpha beta)) minimises chain_broadcast over k."""
    return math.sqrt((p - 2) * n / (alpha * beta))


def optimal_chain_broadcast(p: int, n: float, alpha: float, beta: float) -> float:
    """T* = (sqrt((p-2) alpha) + sqrt(n/beta))^2, the minimum over real k."""
    return (math.sqrt((p - 2) * alpha) + math.sqrt(n / beta)) ** 2


def hierarchical_allreduce(nodes: int, per_node: int, n: float, alpha_intra: float,
                           beta_intra: float, alpha_inter: float, beta_inter: float) -> dict:
    """Intra-node reduce-scatter, per_node concurrent inter-node ring
    all-reduces of n/per_node bytes each, intra-node all-gather; bandwidth and
    latency terms of each phase (section 6.3)."""
    g = per_node
    rs = (g - 1) * alpha_intra + (g - 1) / g * n / beta_intra
    inter = ring_allreduce(nodes, n / g, alpha_inter, beta_inter)
    ag = rs
    return {"intra_reduce_scatter": rs, "inter_allreduce": inter, "intra_all_gather": ag,
            "total": rs + inter + ag}


def crossover(f, g, lo: float = 1.0, hi: float = 1e12) -> float:
    """Message size where two models cost the same (bisection on f - g, which
    must change sign between lo and hi)."""
    d_lo = f(lo) - g(lo)
    d_hi = f(hi) - g(hi)
    if d_lo == 0:
        return lo
    if (d_lo > 0) == (d_hi > 0):
        raise ValueError("the models do not cross in [lo, hi]")
    for _ in range(200):
        mid = math.sqrt(lo * hi) if lo > 0 else 0.5 * (lo + hi)
        d = f(mid) - g(mid)
        if (d > 0) == (d_lo > 0):
            lo, d_lo = mid, d
        else:
            hi = mid
    return 0.5 * (lo + hi)


def bus_bandwidth(algbw: float, p: int) -> float:
    """NCCL's bus bandwidth of an all-reduce: algbw * 2(p-1)/p."""
    return algbw * 2 * (p - 1) / p


ALLREDUCE_MODELS = {
    "ring": ring_allreduce,
    "recursive_doubling": recursive_doubling_allreduce,
    "rabenseifner": rabenseifner_allreduce,
    "binary_tree": binary_tree_allreduce,
    "naive": naive_allreduce,
}


def cheapest_allreduce(p: int, n: float, alpha: float, beta: float) -> tuple[str, float]:
    """The all-reduce algorithm the model predicts fastest for (p, n); the
    power-of-two algorithms are considered only when p is a power of two."""
    best = None
    for name, fn in ALLREDUCE_MODELS.items():
        if name in ("recursive_doubling", "rabenseifner") and p & (p - 1):
            continue
        t = fn(p, n, alpha, beta)
        if best is None or t < best[1]:
            best = (name, t)
    return best
