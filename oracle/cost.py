"""Cost models of a collective: the α-β model and the round model.

* α-β model (primer ch. 4, "Collective communication: algorithms, cost and the
  library that runs them", §4.3; Scaling ML Systems, "Collective
  communication", ring/tree analysis): T = α · (dependent steps) + (bytes
  sent per rank) / B.
* Round model (AI Infra Book ch. 7, "Data-center networks", §7.1.2 and task
  7.2 of §7.2.1): rounds run one after another and the transfers inside a
  round in parallel, each on its own link, so
  T = Σ_rounds (α + max over the round's transfers of bytes / B_link).

The round model is evaluated here on the send log of the oracle's own
step-by-step simulations (``schedules``), so the bytes and rounds are the
schedule's, not a formula's.
"""

from __future__ import annotations

import math
from collections import defaultdict


def alpha_beta(alpha: float, steps: int, bytes_per_rank: float, bw: float) -> float:
    """T = α·steps + bytes/B."""
    return alpha * steps + bytes_per_rank / bw


def round_time(stats, alpha: float, bw_of, elem_bytes: int) -> float:
    """Round model over a simulation's send log: every step costs α plus its
    slowest transfer, bytes / bw_of(src, dst)."""
    worst = defaultdict(float)
    for step, src, dst, lo, hi in stats.sends:
        worst[step] = max(worst[step], (hi - lo) * elem_bytes / bw_of(src, dst))
    return sum(alpha + worst[s] for s in range(stats.steps))


def in_network_time(alpha: float, bytes_per_rank: float, bw: float) -> float:
    """A switch that reduces: one round, each rank sends its buffer once and
    receives the sum once (primer §4.4; AI Infra Book §7.2.1)."""
    return alpha + bytes_per_rank / bw


def ring_formula(alpha: float, n: int, size: float, bw: float) -> float:
    """Primer §4.3: T_ring = 2(N-1)α + 2(N-1)/N · S/B."""
    return 2 * (n - 1) * alpha + 2 * (n - 1) / n * size / bw


def doubling_formula(alpha: float, n: int, size: float, bw: float) -> float:
    """Primer §4.3, recursive doubling: log2 N steps of the whole buffer."""
    k = math.log2(n)
    return k * alpha + k * size / bw


def binary_tree_formula(alpha: float, n: int, size: float, bw: float) -> float:
    """Scaling ML Systems, tree all-reduce: reduce to the root, then broadcast,
    2·log2 N steps, each carrying the whole message."""
    k = math.log2(n)
    return 2 * k * alpha + 2 * k * size / bw


def crossover_ring_doubling(alpha: float, bw: float, n: int) -> float:
    """Primer §4.3: the size where T_ring = T_doubling,
    S* = αB · (2(N-1) - log2 N) / (log2 N - 2(N-1)/N)."""
    k = math.log2(n)
    return alpha * bw * (2 * (n - 1) - k) / (k - 2 * (n - 1) / n)


def crossover_ring_tree_approx(alpha: float, bw: float, n: int) -> float:
    """Scaling ML Systems: for large N the ring/tree crossover is about N·α·β / log2 N."""
    return n * alpha * bw / math.log2(n)
