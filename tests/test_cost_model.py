"""The library's cost model (ar_plan_predict, ar_select, AR_AUTO) on the host,
against the oracle's round model over its own simulations and against the
numbers the pages print. No GPU needed."""

import math

import numpy as np
import pytest

from oracle import cost, schedules
from test_oracle_cost import ALPHA_BOOK, MiB, NIC, NVLINK, check


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


def _oracle_round(fn, N, L, alpha, bw_of, **kw):
    st = fn(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L, **kw)[1]
    return cost.round_time(st, alpha, bw_of, 4)


def test_task_7_2_predictions(g, golden):
    rows = golden("cost_model.txt")
    L = (192 * MiB) // 4
    fab = g.fabric(ALPHA_BOOK, NVLINK, NIC, ranks_per_server=8)
    ring = g.ar_plan_predict(g.ar_plan(16, L, "f32", "ring"), fab)
    hier = g.ar_plan_predict(g.ar_plan(16, L, "f32", "hier", group_size=8), fab)
    check(rows, "continuous_ring_s", ring)
    check(rows, "hierarchical_s", hier)
    two = lambda s, d: NVLINK if s // 8 == d // 8 else NIC  # noqa: E731
    assert ring == pytest.approx(_oracle_round(schedules.ring_allreduce, 16, L, ALPHA_BOOK, two), rel=1e-12)
    assert hier == pytest.approx(_oracle_round(schedules.hierarchical_allreduce, 16, L, ALPHA_BOOK, two,
                                               group_size=8), rel=1e-12)


def test_inter_server_stage_and_in_network(g, golden):
    rows = golden("cost_model.txt")
    L = (24 * MiB) // 4
    for key, val in rows:
        if key == "inter_server_ring":
            f = dict(kv.split("=") for kv in val.split())
            S = int(f["servers"])
            got = g.ar_plan_predict(g.ar_plan(S, L, "f32", "ring"), g.fabric(ALPHA_BOOK, NIC, NIC, 1))
            check([("t", f["time_s"])], "t", got)
    fused = g.ar_plan(2, L, "f32", "fused")
    check(rows, "in_network_s", g.ar_plan_predict(fused, g.fabric(ALPHA_BOOK, NIC, NIC, 1, in_network=True)))
    with pytest.raises(g.ArError) as e:  # no switch reduction, no shared memory: no single pass
        g.ar_plan_predict(fused, g.fabric(ALPHA_BOOK, NIC, NIC, 1))
    assert e.value.status == g.AR_EUNSUPPORTED


def test_tensor_parallel_example(g, golden):
    rows = golden("cost_model.txt")
    check(rows, "tp_ring_s", g.ar_plan_predict(g.ar_plan(8, 250_000, "f32", "ring"), g.fabric(5e-6, NVLINK)))


@pytest.mark.parametrize("N,L,G", [(4, 1000, 2), (8, 4099, 4), (16, 777, 8), (12, 300, 3), (64, 4096, 8)])
def test_predictions_equal_the_oracle_round_model(g, N, L, G):
    alpha, loc, net = 2e-6, 300e9, 40e9
    fab = g.fabric(alpha, loc, net, ranks_per_server=G)
    bw = lambda s, d: loc if s // G == d // G else net  # noqa: E731
    algos = [("ring", schedules.ring_allreduce, {}), ("hier", schedules.hierarchical_allreduce, {"group_size": G})]
    algos.append(("dbtree", schedules.double_binary_tree_allreduce, {}))
    if N & (N - 1) == 0:
        algos.append(("rabenseifner", schedules.rabenseifner_allreduce, {}))
        algos.append(("recdoubling", schedules.recursive_doubling_allreduce, {}))
    for name, fn, kw in algos:
        got = g.ar_plan_predict(g.ar_plan(N, L, "f32", name, group_size=G), fab)
        assert got == pytest.approx(_oracle_round(fn, N, L, alpha, bw, **kw), rel=1e-12), name
    dims = (G, N // G)
    got = g.ar_plan_predict(g.ar_plan(N, L, "f32", "torus", torus_dims=dims), fab)
    assert got == pytest.approx(_oracle_round(schedules.torus_allreduce, N, L, alpha, bw, dims=dims), rel=1e-12)
    for coll, fn in (("reduce_scatter", schedules.ring_reduce_scatter), ("allgather", schedules.ring_allgather)):
        got = g.ar_plan_predict(g.ar_plan(N, L, "f32", "ring", collective=coll), fab)
        assert got == pytest.approx(_oracle_round(fn, N, L, alpha, bw), rel=1e-12), coll


def test_select_follows_the_model(g, golden):
    MiB_ = MiB
    book = g.fabric(ALPHA_BOOK, NVLINK, NIC, ranks_per_server=8)
    # 192 MiB on 2 x 8: distance-1-first halving keeps all but its last
    # round inside a server, so it carries the hierarchy's network bytes in
    # half the rounds
    algo, gs, t = g.ar_select(16, 192 * MiB_ // 4, book)
    assert algo == "rabenseifner" and t == pytest.approx(
        16 * 0 + 8 * ALPHA_BOOK + 2 * (96 + 48 + 24) * MiB_ / NVLINK + 2 * 12 * MiB_ / NIC, rel=1e-12)
    # 12 ranks (no power of two): the hierarchy beats the flat ring
    algo, gs, _ = g.ar_select(12, 192 * MiB_ // 4, g.fabric(ALPHA_BOOK, NVLINK, NIC, ranks_per_server=6))
    assert (algo, gs) == ("hier", 6)
    # small message on one server: fewer steps win. In the primer's 1 MB
    # example recursive doubling's 3 rounds beat Rabenseifner's 6 and the
    # ring's 14, at the time the page prints for doubling
    algo, _, t = g.ar_select(8, 250_000, g.fabric(5e-6, NVLINK))
    assert algo == "recdoubling"
    check(golden("cost_model.txt"), "tp_doubling_s", t)
    # 6 ranks (no doubling): the double binary tree's 6 rounds of S/2 beat
    # the ring's 10 rounds of S/6 when alpha dominates
    assert g.ar_select(6, 250_000, g.fabric(5e-6, NVLINK))[0] == "dbtree"
    assert g.ar_select(6, 250_000_000, g.fabric(5e-6, NVLINK))[0] == "ring"
    # one shared memory: the single pass
    dev = g.fabric(g.AR_DEVICE_ALPHA_S, g.AR_DEVICE_BW, shared_memory=True)
    for N in (2, 3, 16, 64):
        assert g.ar_select(N, 1 << 20, dev)[0] == "fused"
    assert g.ar_select(16, 1 << 20, dev, collective="reduce_scatter")[0] == "fused"


def test_device_model_is_launches_plus_bytes(g):
    dev = g.fabric(g.AR_DEVICE_ALPHA_S, g.AR_DEVICE_BW, shared_memory=True)
    for algo in ("ring", "rabenseifner", "fused", "recdoubling", "dbtree"):
        p = g.ar_plan(16, 50_331_648, "f32", algo)
        st = p.stats
        assert g.ar_plan_predict(p, dev) == pytest.approx(
            st["launches"] * g.AR_DEVICE_ALPHA_S + st["hbm_bytes"] / g.AR_DEVICE_BW, rel=1e-12)


def test_device_model_of_one_cta_plans(g):
    # a plan run whole in one CTA: one launch, then a block-barrier step each
    dev = g.fabric(g.AR_DEVICE_ALPHA_S, g.AR_DEVICE_BW, shared_memory=True)
    for algo, L in (("ring", 256), ("rabenseifner", 256)):
        p = g.ar_plan(16, L, "f32", algo)
        st = p.stats
        assert st["launches"] == 1 and st["steps"] > 1
        assert g.ar_plan_predict(p, dev) == pytest.approx(
            g.AR_DEVICE_ALPHA_S + st["steps"] * g.AR_DEVICE_CTA_STEP_S + st["hbm_bytes"] / g.AR_DEVICE_BW, rel=1e-12)
    # measured on GB300 (device time, buffers on chip): ring 13.2 us,
    # Rabenseifner 7.2 us, of which about 4 us are the launch and the copies
    # in and out that the model leaves out
    ring = g.ar_plan_predict(g.ar_plan(16, 256, "f32", "ring"), dev)
    rab = g.ar_plan_predict(g.ar_plan(16, 256, "f32", "rabenseifner"), dev)
    assert 8e-6 < ring < 11e-6 and 3e-6 < rab < 4.5e-6
    # 16 x 2048 fp32 does not fit on chip (8 bytes per element and rank over
    # 160 KiB): its one-CTA steps are priced at the in-memory rate
    p = g.ar_plan(16, 2048, "f32", "ring")
    st = p.stats
    assert st["launches"] == 1
    assert g.ar_plan_predict(p, dev) == pytest.approx(
        g.AR_DEVICE_ALPHA_S + st["steps"] * g.AR_DEVICE_CTA_STEP_MEM_S + st["hbm_bytes"] / g.AR_DEVICE_BW, rel=1e-12)
    # still the single pass for AR_AUTO at any size
    assert g.ar_select(16, 256, dev)[0] == "fused"


def test_auto_resolves_to_the_single_pass(g):
    for N, order in ((16, "ring"), (8, "tree"), (5, "rank")):
        p = g.ar_plan(N, 12345, "f32", "auto", order=order)
        assert g.ar_plan_desc(p)["algo"] == "fused"
    p = g.ar_plan(8, 999, "bf16", "auto", collective="allgather")
    assert g.ar_plan_desc(p)["algo"] == "fused"


def test_fabric_validation(g):
    p = g.ar_plan(4, 100, "f32", "ring")
    for bad in (g.fabric(-1, 1e9), g.fabric(1e-6, 0.0), g.fabric(1e-6, 1e9, -5.0), g.fabric(math.nan, 1e9)):
        with pytest.raises(g.ArError) as e:
            g.ar_plan_predict(p, bad)
        assert e.value.status == g.AR_EINVAL
