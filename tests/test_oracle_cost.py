"""The cost models against the numbers the pages print. Rounds and bytes come
from the oracle's step-by-step simulations; the pages' values are matched to
within half of their last printed digit."""

import math

import numpy as np
import pytest

from oracle import cost, schedules

MiB = 1 << 20
ALPHA_BOOK = 0.83e-6  # start-up per round in the AI Infra Book's example
NVLINK, NIC = 450e9, 50e9


def printed(golden_rows, key):
    """(value, tolerance) of a printed number: tolerance is half its last digit."""
    text = dict(golden_rows)[key]
    mant, _, exp = text.partition("e")
    decimals = len(mant.split(".")[1]) if "." in mant else 0
    scale = 10.0 ** int(exp) if exp else 1.0
    return float(mant) * scale, 0.5 * 10.0 ** -decimals * scale


def check(golden_rows, key, got):
    want, tol = printed(golden_rows, key)
    assert abs(got - want) <= tol * (1 + 1e-9), f"{key}: {got} vs printed {want} +- {tol}"


def _sim(fn, N, L, **kw):
    return fn(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L, **kw)[1]


def two_servers(src, dst):
    return NVLINK if src // 8 == dst // 8 else NIC


def test_task_7_2_rings_and_hierarchy(golden):
    rows = golden("cost_model.txt")
    L = (192 * MiB) // 4
    st = _sim(schedules.ring_allreduce, 16, L)
    check(rows, "continuous_ring_s", cost.round_time(st, ALPHA_BOOK, two_servers, 4))
    gpu = [(i // 2) + 8 * (i % 2) for i in range(16)]  # ring order 0, 8, 1, 9, ...
    check(rows, "interleaved_ring_s",
          cost.round_time(st, ALPHA_BOOK, lambda s, d: NVLINK if gpu[s] // 8 == gpu[d] // 8 else NIC, 4))
    st = _sim(schedules.hierarchical_allreduce, 16, L, group_size=8)
    assert st.steps == 16
    check(rows, "hierarchical_s", cost.round_time(st, ALPHA_BOOK, two_servers, 4))
    local = cost.round_time(st, 0.0, lambda s, d: NVLINK if s // 8 == d // 8 else math.inf, 4)
    net = cost.round_time(st, 0.0, lambda s, d: math.inf if s // 8 == d // 8 else NIC, 4)
    check(rows, "hierarchical_local_s", local)
    check(rows, "hierarchical_network_s", net)
    check(rows, "hierarchical_startup_s", st.steps * ALPHA_BOOK)


def test_inter_server_ring_table_and_in_network(golden):
    rows = golden("cost_model.txt")
    slice_bytes = 24 * MiB
    for key, val in rows:
        if key != "inter_server_ring":
            continue
        f = dict(kv.split("=") for kv in val.split())
        S = int(f["servers"])
        st = _sim(schedules.ring_allreduce, S, slice_bytes // 4)
        assert st.steps == int(f["rounds"])
        assert int(st.elements_sent.max()) * 4 == float(f["send_mib"]) * MiB
        check([("t", f["time_s"])], "t", cost.round_time(st, ALPHA_BOOK, lambda s, d: NIC, 4))
    check(rows, "in_network_s", cost.in_network_time(ALPHA_BOOK, slice_bytes, NIC))


def test_primer_tensor_parallel_example(golden):
    rows = golden("cost_model.txt")
    N, S, alpha = 8, 1e6, 5e-6
    st = _sim(schedules.ring_allreduce, N, int(S) // 4)
    check(rows, "tp_ring_s", cost.round_time(st, alpha, lambda s, d: NVLINK, 4))
    check(rows, "tp_ring_latency_s", st.steps * alpha)
    check(rows, "tp_ring_bandwidth_s", int(st.elements_sent.max()) * 4 / NVLINK)
    check(rows, "tp_doubling_s", cost.doubling_formula(alpha, N, S, NVLINK))


def test_crossover_and_llama_examples(golden):
    rows = golden("cost_model.txt")
    check(rows, "crossover_bytes", cost.crossover_ring_doubling(22e-6, 50e9, 128))
    bw_term = cost.ring_formula(0.0, 128, 810e9, 50e9)
    check(rows, "llama_full_copy_bandwidth_s", bw_term)
    check(rows, "llama_full_copy_latency_s", cost.ring_formula(22e-6, 128, 0.0, 50e9))
    check(rows, "llama_fsdp_shard_s", cost.ring_formula(0.0, 128, 6.3e9, 50e9))


def test_ring_versus_tree_example(golden):
    rows = golden("cost_model.txt")
    N, M, alpha, beta = 64, 1e6, 10e-6, 10e9
    check(rows, "p2_ring_s", cost.ring_formula(alpha, N, M, beta))
    check(rows, "p2_ring_latency_s", cost.ring_formula(alpha, N, 0.0, beta))
    check(rows, "p2_ring_bandwidth_s", cost.ring_formula(0.0, N, M, beta))
    check(rows, "p2_tree_s", cost.binary_tree_formula(alpha, N, M, beta))
    check(rows, "p2_crossover_bytes", cost.crossover_ring_tree_approx(alpha, beta, N))
    check(rows, "p2_crossover_100_bytes", cost.crossover_ring_tree_approx(5e-6, 50e9, 100))


@pytest.mark.parametrize("N", [2, 4, 8, 16, 64])
def test_round_model_on_uniform_links_is_the_alpha_beta_formula(N):
    """With every link alike, the round model over the simulated ring is the
    primer's closed form, and Rabenseifner has the ring's bytes in 2 log2 N
    rounds."""
    L, alpha, bw = 1024 * N, 3e-6, 100e9
    st = _sim(schedules.ring_allreduce, N, L)
    got = cost.round_time(st, alpha, lambda s, d: bw, 4)
    assert got == pytest.approx(cost.ring_formula(alpha, N, 4 * L, bw), rel=1e-12)
    rb = _sim(schedules.rabenseifner_allreduce, N, L)
    k = int(math.log2(N))
    want = 2 * k * alpha + 2 * (N - 1) / N * 4 * L / bw
    # halving/doubling rounds carry S/2, S/4, ...: the sum of the rounds' maxima is the byte total
    assert cost.round_time(rb, alpha, lambda s, d: bw, 4) == pytest.approx(want, rel=1e-12)
