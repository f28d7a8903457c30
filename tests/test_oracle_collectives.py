"""The standalone reduce-scatter and all-gather of the oracle against the
primer's table of collectives (§4.1) and against the all-reduce they compose."""

from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import numerics, schedules


def _frac(expr, N):
    # "2(N-1)/N" or "(N-1)/N"
    num = 2 if expr.startswith("2") else 1
    return Fraction(num * (N - 1), N)


def _acct(fn, N, L):
    return fn(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L)[1]


@pytest.mark.parametrize("N", [2, 3, 4, 8, 16, 64])
def test_bytes_and_steps_match_the_table(golden, N):
    d = dict(golden("collectives_table.txt"))
    L = 24 * N
    for fn, key in ((schedules.ring_reduce_scatter, "reduce_scatter_sent"),
                    (schedules.ring_allgather, "allgather_sent"),
                    (schedules.ring_allreduce, "allreduce_sent")):
        st = _acct(fn, N, L)
        assert all(Fraction(int(e), L) == _frac(d[key], N) for e in st.elements_sent), key
    rs, ag, ar = (_acct(f, N, L) for f in (schedules.ring_reduce_scatter, schedules.ring_allgather,
                                           schedules.ring_allreduce))
    assert rs.steps == ag.steps == N - 1 and ar.steps == 2 * (N - 1)
    # the all-reduce's bytes are the sum of its halves'
    assert np.array_equal(rs.elements_sent + ag.elements_sent, ar.elements_sent)


@pytest.mark.parametrize("N,L", [(1, 5), (2, 3), (4, 4), (5, 17), (8, 1000), (7, 6)])
def test_reduce_scatter_gives_rank_i_chunk_i(N, L):
    x = workloads.all_ranks(workloads.small_spec(N, L, dist="normal", seed=N + L))
    out, st = schedules.ring_reduce_scatter(x)
    b = [(c * L) // N for c in range(N + 1)]
    want = numerics.fused_sum(x, "ring_rs")
    ref = numerics.reference_sum_f64(x)
    bound = (N - 1) * 2.0 ** -24 * numerics.abs_sum_f64(x)
    for i in range(N):
        assert st.owned[i] == (b[i], b[i + 1])
        seg = slice(b[i], b[i + 1])
        np.testing.assert_array_equal(out[i, seg].view(np.uint32), want[seg].view(np.uint32))
        assert np.all(np.abs(out[i, seg].astype(np.float64) - ref[seg]) <= bound[seg])


def test_reduce_scatter_provenance():
    """With inputs 2^r, after the reduce-scatter rank i's chunk i holds all N
    contributions and every other chunk of rank i strictly fewer."""
    N = 6
    x = np.array([[float(1 << r)] * N for r in range(N)], np.float32)
    out, _ = schedules.ring_reduce_scatter(x)
    for i in range(N):
        for c in range(N):
            k = bin(int(out[i, c])).count("1")
            assert (k == N) == (c == i)


@pytest.mark.parametrize("N,L", [(2, 3), (4, 4), (5, 17), (8, 1000)])
def test_allgather_collects_every_rank_chunk(N, L):
    x = workloads.all_ranks(workloads.small_spec(N, L, dist="uniform", seed=L))
    out, _ = schedules.ring_allgather(x)
    b = [(c * L) // N for c in range(N + 1)]
    want = np.concatenate([x[c, b[c]:b[c + 1]] for c in range(N)])
    for r in range(N):
        np.testing.assert_array_equal(out[r], want)


@pytest.mark.parametrize("N,L", [(2, 9), (4, 1000), (8, 4099), (16, 333)])
def test_reduce_scatter_then_allgather_is_an_allreduce(N, L):
    """§4.1: an all-reduce is a reduce-scatter followed by an all-gather. With
    rank i owning chunk i, the composition is bit for bit the hierarchical
    order with one group of N (every chunk folded from rank c+1)."""
    x = workloads.all_ranks(workloads.small_spec(N, L, dist="normal", seed=N * L))
    rs, _ = schedules.ring_reduce_scatter(x)
    ag, _ = schedules.ring_allgather(rs)
    want = numerics.fused_sum(x, "hier", group_size=N)
    np.testing.assert_array_equal(numerics.fused_sum(x, "ring_rs"), want)
    for r in range(N):
        np.testing.assert_array_equal(ag[r].view(np.uint32), want.view(np.uint32))
    h, _ = schedules.hierarchical_allreduce(x, N)
    np.testing.assert_array_equal(h, ag)
