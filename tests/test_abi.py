"""The C ABI without a GPU: the library loads, exports every call the header
declares, rejects bad arguments before touching the device, and its host-side
schedules are the oracle's schedules step for step.

The oracle and the library share no code: the library builds its step tables
in C++ from the index rules, the oracle simulates the sends in numpy.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import workloads
from oracle import buckets as obuckets
from oracle import schedules

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


def header_functions():
    text = open(os.path.join(ROOT, "include", "ar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(ar_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(g):
    names = header_functions()
    assert len(names) >= 14, names
    lib = ctypes.CDLL(g._lib.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    # and the binding declares exactly those
    assert sorted(g._lib.SIGNATURES) == names


def test_version_and_status_strings(g):
    assert g.ar_version() >= 1
    for code in range(6):
        assert g.ar_status_string(code).startswith("AR_")


def _oracle_steps(fn, N, L, **kw):
    """The oracle's sends grouped by step: {step: set of (src, dst, lo, hi)}."""
    _, st = fn(np.zeros((N, 0), np.float32), idx=np.zeros(0, np.int64), L=L, **kw)
    steps = {}
    for step, src, dst, lo, hi in st.sends:
        if hi > lo:
            steps.setdefault(step, set()).add((src, dst, lo, hi))
    return st, steps


CASES = [(N, L) for N in (1, 2, 3, 4, 5, 8, 16) for L in (0, 1, 7, 16, 1000, 4099)] + [(64, 4096), (64, 50)]


@pytest.mark.parametrize("N,L", CASES)
def test_ring_table_matches_oracle(g, N, L):
    plan = g.ar_plan(N, L, "f32", "ring")
    st, steps = _oracle_steps(schedules.ring_allreduce, N, L)
    stats = plan.stats
    assert stats["steps"] == st.steps == 2 * (N - 1)
    for s in range(stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if s < N - 1 else "copy")
        assert set(rows) == steps.get(s, set()), s
    assert stats["bytes_sent_per_rank"] == 4 * int(st.elements_sent.max())
    assert stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


@pytest.mark.parametrize("N,L", [(N, L) for N in (1, 2, 4, 8, 16, 64) for L in (0, 3, 64, 1001)])
def test_rabenseifner_table_matches_oracle(g, N, L):
    plan = g.ar_plan(N, L, "f32", "rabenseifner")
    st, steps = _oracle_steps(schedules.rabenseifner_allreduce, N, L)
    K = N.bit_length() - 1
    stats = plan.stats
    assert stats["steps"] == st.steps == 2 * K
    for s in range(stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if s < K else "copy")
        assert set(rows) == steps.get(s, set()), s
    assert stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


@pytest.mark.parametrize("N,G,L", [(16, 8, 1000), (16, 8, 4099), (8, 2, 333), (8, 4, 64), (6, 3, 100),
                                   (8, 1, 77), (8, 8, 77), (4, 2, 3), (64, 8, 4096)])
def test_hierarchical_table_matches_oracle(g, N, G, L):
    plan = g.ar_plan(N, L, "f32", "hier", group_size=G)
    st, steps = _oracle_steps(schedules.hierarchical_allreduce, N, L, group_size=G)
    M = N // G
    stats = plan.stats
    assert stats["steps"] == st.steps == 2 * (G - 1) + 2 * (M - 1)
    n_reduce = (G - 1) + (M - 1)
    for s in range(stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if s < n_reduce else "copy")
        assert set(rows) == steps.get(s, set()), s
    assert stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


def test_headline_accounting(g):
    S = 192 << 20
    ring = g.ar_plan(16, S // 4, "f32", "ring").stats
    assert ring["bytes_sent_per_rank"] == 360 << 20
    assert ring["hbm_bytes"] == 5 * 15 * S  # 5(N-1)*S: 3 per reduce, 2 per copy element
    fused = g.ar_plan(16, S // 4, "f32", "fused").stats
    assert fused["hbm_bytes"] == 2 * 16 * S and fused["launches"] == 1
    hier = g.ar_plan(16, 96 << 20, "bf16", "hier", group_size=8).stats
    assert hier["steps"] == 16
    assert hier["workspace_bytes"] == 16 * (96 << 20) * 4
    assert g.ar_plan(16, 96 << 20, "bf16", "fused", order="hier", group_size=8).stats["workspace_bytes"] == 0


@pytest.mark.parametrize("kw", [
    dict(n_ranks=0), dict(n_ranks=65), dict(dtype=7), dict(algo=9), dict(order=9),
    dict(algo="rabenseifner", n_ranks=6), dict(order="tree", n_ranks=12),
    dict(algo="hier", group_size=0), dict(algo="hier", group_size=3),
    dict(order="hier", group_size=5), dict(scale=float("inf")), dict(scale=float("nan")),
])
def test_plan_rejects(g, kw):
    args = dict(n_ranks=8, count=100, dtype="f32", algo="fused", group_size=2, order="ring", scale=1.0)
    args.update(kw)
    with pytest.raises(g.ArError) as e:
        g.ar_plan(**args)
    assert e.value.status == g.AR_EINVAL


def test_execute_rejects_bad_pointers_without_touching_the_device(g):
    plan = g.ar_plan(4, 1024, "f32", "fused")
    good = [0x100000 * (r + 1) for r in range(4)]
    for bufs in ([0] + good[1:], [good[0] + 4] + good[1:], [good[0]] * 4,
                 [good[0], good[0] + 2048] + good[2:]):  # null, misaligned, same, overlapping
        with pytest.raises(g.ArError) as e:
            g.ar_execute(plan, bufs, stream=0)
        assert e.value.status == g.AR_EINVAL
    with pytest.raises(g.ArError):  # an output overlapping another rank's input
        g.ar_execute(plan, good, outs=[good[1]] + good[1:], stream=0)
    wplan = g.ar_plan(4, 1024, "bf16", "ring")
    with pytest.raises(g.ArError) as e:  # bf16 step plans need a workspace
        g.ar_execute(wplan, good, stream=0)
    assert e.value.status == g.AR_EINVAL
    empty = g.ar_plan(4, 0, "f32", "ring")
    g.ar_execute(empty, good, stream=0)  # count 0: nothing to do, no device call


def test_bucket_plan_matches_oracle(g):
    counts = [c for _, c in workloads.transformer_tensors()]
    of, nb = g.ar_bucket_plan(counts, 2, workloads.BUCKET_CAP_BYTES)
    want = obuckets.bucket_plan(counts, 2, workloads.BUCKET_CAP_BYTES)
    assert nb == len(want) == 81
    for b, tensors in enumerate(want):
        assert all(of[t] == b for t in tensors)
    rng = np.random.default_rng(0)
    for cap in (1, 9, 100, 10_000):
        counts = rng.integers(0, 60, 50).tolist()
        of, nb = g.ar_bucket_plan(counts, 4, cap)
        want = obuckets.bucket_plan(counts, 4, cap)
        assert nb == len(want)
        assert [[t for t in reversed(range(50)) if of[t] == b] for b in range(nb)] == want


def test_bucket_calls_reject(g):
    ok = [[0x100000 * (r * 4 + t + 1) for t in range(3)] for r in range(2)]
    with pytest.raises(g.ArError):
        g.ar_bucket_allreduce(ok, [10, 10, 10], 2, 1, "bf16", 0.5, stream=0)  # empty range
    with pytest.raises(g.ArError):
        g.ar_bucket_allreduce(ok, [10, 10, 10], 0, 4, "bf16", 0.5, stream=0)  # past the end
    bad = [row[:] for row in ok]
    bad[1][2] += 2
    with pytest.raises(g.ArError):
        g.ar_bucket_allreduce(bad, [10, 10, 10], 0, 3, "bf16", 0.5, stream=0)  # misaligned
    with pytest.raises(g.ArError):
        g.ar_bucket_pack(ok, [10, 10, 10], 0, 3, "bf16", [0x9000000, 0], stream=0)  # null bucket


@pytest.mark.parametrize("N,L", [(2, 5), (3, 7), (4, 4), (5, 4099), (8, 1000), (16, 50), (64, 4096)])
@pytest.mark.parametrize("coll", ["reduce_scatter", "allgather"])
def test_ring_collective_tables_match_oracle(g, coll, N, L):
    plan = g.ar_plan(N, L, "f32", "ring", collective=coll)
    fn = schedules.ring_reduce_scatter if coll == "reduce_scatter" else schedules.ring_allgather
    st, steps = _oracle_steps(fn, N, L)
    stats = plan.stats
    assert stats["steps"] == st.steps == N - 1
    for s in range(stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if coll == "reduce_scatter" else "copy")
        assert set(rows) == steps.get(s, set()), s
    assert stats["bytes_sent_per_rank"] == 4 * int(st.elements_sent.max())
    assert stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


def test_collective_validation(g):
    for algo in ("rabenseifner", "hier"):
        for coll in ("reduce_scatter", "allgather"):
            with pytest.raises(g.ArError) as e:
                g.ar_plan(8, 100, "f32", algo, group_size=4, collective=coll)
            assert e.value.status == g.AR_EUNSUPPORTED
    with pytest.raises(g.ArError) as e:
        g.ar_plan(8, 100, "f32", "fused", group_size=4, order="hier", collective="reduce_scatter")
    assert e.value.status == g.AR_EUNSUPPORTED
    with pytest.raises(g.ArError) as e:
        g.ar_plan(8, 100, "f32", "fused", collective=7)
    assert e.value.status == g.AR_EINVAL
    rs = g.ar_plan(16, 1 << 20, "f32", "fused", collective="reduce_scatter").stats
    ag = g.ar_plan(16, 1 << 20, "f32", "fused", collective="allgather").stats
    assert rs["hbm_bytes"] == (16 + 1) * (1 << 20) * 4 and ag["hbm_bytes"] == (16 + 1) * (1 << 20) * 4
    assert g.ar_plan(16, 1 << 20, "bf16", "ring", collective="allgather").stats["workspace_bytes"] == 0


def test_kernel_choice_validation(g):
    with pytest.raises(g.ArError) as e:
        g.ar_plan(8, 100, "f32", "fused", kernel=3)
    assert e.value.status == g.AR_EINVAL
    for bad in (dict(n_ranks=25), dict(collective="reduce_scatter")):
        args = dict(n_ranks=8, count=100, dtype="f32", algo="fused", kernel="bulk")
        args.update(bad)
        with pytest.raises(g.ArError) as e:  # the all-reduce's stages must fit in shared memory; no RS
            g.ar_plan(**args)
        assert e.value.status == g.AR_EUNSUPPORTED, bad
    for n in (2, 25, 64):  # the all-gather stages one rank's tile: any N
        assert g.ar_plan_desc(g.ar_plan(n, 100, "f32", "fused", kernel="bulk", collective="allgather"))["kernel"] == "bulk"
    for n in (1, 2, 16, 24):
        assert g.ar_plan_desc(g.ar_plan(n, 100, "bf16", "fused", kernel="bulk"))["kernel"] == "bulk"
    assert g.ar_plan_desc(g.ar_plan(64, 100, "f32", "ring", kernel="bulk"))["kernel"] == "bulk"  # ignored
    assert g.ar_plan_desc(g.ar_plan(8, 100, "f32", "fused"))["kernel"] == "auto"
    ok = [[0x100000 * (r * 4 + t + 1) for t in range(3)] for r in range(25)]
    with pytest.raises(g.ArError) as e:
        g.ar_bucket_allreduce(ok, [10, 10, 10], 0, 3, "bf16", 0.5, stream=0, kernel="bulk")
    assert e.value.status == g.AR_EUNSUPPORTED
    with pytest.raises(g.ArError) as e:
        g.ar_bucket_allreduce(ok[:4], [10, 10, 10], 0, 3, "bf16", 0.5, stream=0, kernel=7)
    assert e.value.status == g.AR_EINVAL


def _check_table(g, plan, st, steps, n_reduce):
    stats = plan.stats
    assert stats["steps"] == st.steps
    for s in range(stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if s < n_reduce else "copy"), s
        assert len(rows) == len(set(rows))
        assert set(rows) == steps.get(s, set()), s
    assert stats["bytes_sent_per_rank"] == 4 * int(st.elements_sent.max())


@pytest.mark.parametrize("N,L", [(N, L) for N in (1, 2, 4, 8, 16, 64) for L in (0, 1, 7, 1001)])
def test_recursive_doubling_table_matches_oracle(g, N, L):
    plan = g.ar_plan(N, L, "f32", "recdoubling")
    st, steps = _oracle_steps(schedules.recursive_doubling_allreduce, N, L)
    K = N.bit_length() - 1
    assert plan.stats["steps"] == K
    _check_table(g, plan, st, steps, K)
    # an exchange reads both copies and writes both once: 2 reads + 2 writes per pair
    assert plan.stats["hbm_bytes"] == (4 * 4 * (N // 2) * L * K if N > 1 else 0)


@pytest.mark.parametrize("N,L", [(N, L) for N in (1, 2, 3, 5, 8, 12, 16, 33, 64) for L in (0, 1, 2, 9, 1001)])
def test_double_binary_tree_table_matches_oracle(g, N, L):
    plan = g.ar_plan(N, L, "f32", "dbtree")
    st, steps = _oracle_steps(schedules.double_binary_tree_allreduce, N, L)
    _check_table(g, plan, st, steps, st.steps // 2)
    assert plan.stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


@pytest.mark.parametrize("dims,L", [((4, 4), 1000), ((2, 8), 77), ((8, 2), 4099), ((3, 5), 9), ((2, 3, 2), 100),
                                    ((2, 2, 2), 0), ((1, 6), 31), ((5, 1), 5), ((4, 4, 4), 4096), ((1,), 8)])
def test_torus_table_matches_oracle(g, dims, L):
    N = int(np.prod(dims))
    plan = g.ar_plan(N, L, "f32", "torus", torus_dims=dims)
    st, steps = _oracle_steps(schedules.torus_allreduce, N, L, dims=dims, trace=lambda w: None)
    assert plan.stats["steps"] == st.steps == sum(2 * (d - 1) for d in dims)
    for s in range(plan.stats["steps"]):
        op, rows = g.ar_plan_transfers(plan, s)
        assert op == ("reduce" if "reduce-scatter" in st.trace[s][0] else "copy"), s
        assert set(rows) == steps.get(s, set()), s
    assert plan.stats["bytes_sent_per_rank"] == 4 * int(st.elements_sent.max())
    assert plan.stats["hbm_bytes"] == 4 * (st.element_reads + st.element_writes)


def test_variant_validation(g):
    for N in (3, 6, 12):
        with pytest.raises(g.ArError) as e:
            g.ar_plan(N, 100, "f32", "recdoubling")
        assert e.value.status == g.AR_EINVAL
    for dims in ((4, 3), (0, 0, 0), (16, 2), (-1, 16), (65, 1, 1)):
        with pytest.raises(g.ArError) as e:
            g.ar_plan(16, 100, "f32", "torus", torus_dims=dims)
        assert e.value.status == g.AR_EINVAL, dims
    for algo in ("recdoubling", "dbtree"):
        for coll in ("reduce_scatter", "allgather"):
            with pytest.raises(g.ArError) as e:
                g.ar_plan(8, 100, "f32", algo, collective=coll)
            assert e.value.status == g.AR_EUNSUPPORTED
    with pytest.raises(g.ArError) as e:
        g.ar_plan(8, 100, "f32", 8)
    assert e.value.status == g.AR_EINVAL
    d = g.ar_plan_desc(g.ar_plan(16, 100, "f32", "torus", torus_dims=(4, 0, 4)))
    assert d["torus_dims"] == (4, 0, 4)
    assert g.ar_plan_desc(g.ar_plan(16, 100, "f32", "ring", torus_dims=(4, 4)))["torus_dims"] == (0, 0, 0)
    # bf16 step plans keep fp32 partial sums in the workspace
    assert g.ar_plan(16, 1000, "bf16", "torus", torus_dims=(4, 4)).stats["workspace_bytes"] == 16 * 1024 * 4


def test_compress_sizes_match_oracle(g):
    from oracle import compress as ocomp

    for count in (0, 1, 15, 16, 17, 1000, 4099, 1 << 20, 50_331_648):
        for b in (16, 32, 64, 128, 256, 512, 1024):
            ns, mb = g.ar_compress_sizes(count, b)
            assert ns == ocomp.n_blocks(count, b)
            assert mb == ocomp.message_bytes(count, b)
    for b in (0, 8, 15, 48, 100, 2048, -64):
        with pytest.raises(g.ArError) as e:
            g.ar_compress_sizes(100, b)
        assert e.value.status == g.AR_EINVAL


def test_compression_calls_reject_without_touching_the_device(g):
    N, L, b = 3, 1000, 64
    base = [0x1000000 * (k + 1) for k in range(20)]
    grads, codes, scales, res, outs = base[0:3], base[3:6], base[6:9], base[9:12], base[12:15]

    def rejects(fn, *a, **kw):
        with pytest.raises(g.ArError) as e:
            fn(*a, count=L, stream=0, **kw)
        assert e.value.status == g.AR_EINVAL

    for blk in (8, 100, 2048):
        rejects(g.ar_compress, grads, codes, scales, blk)
        rejects(g.ar_compressed_reduce, codes, scales, outs, blk)
        rejects(g.ar_compressed_allreduce, grads, blk)
    rejects(g.ar_compress, grads, codes, scales, b, dtype=5)
    rejects(g.ar_compress, [grads[0] + 4] + grads[1:], codes, scales, b)          # misaligned
    rejects(g.ar_compress, grads, [0] + codes[1:], scales, b)                     # null
    rejects(g.ar_compress, grads, codes, [codes[0] + 512] + scales[1:], b)        # scales overlap codes
    rejects(g.ar_compress, grads, codes, scales, b, residuals=[grads[1]] + res[1:])  # residual = a gradient
    rejects(g.ar_compressed_reduce, codes, scales, outs, b, scale=float("nan"))
    rejects(g.ar_compressed_reduce, codes, scales, [codes[1]] + outs[1:], b)      # output over codes
    rejects(g.ar_compressed_allreduce, grads, b, outs=[grads[1]] + outs[1:])      # output over another input
    rejects(g.ar_compressed_allreduce, grads, b, scale=float("inf"))
    rejects(g.ar_compressed_allreduce, grads, b, residuals=res[:2] + [res[2] + 8])
    with pytest.raises(g.ArError):
        g.ar_compressed_allreduce([grads[0]] * 65, b, count=L, stream=0)          # too many ranks
    # count 0 validates and enqueues nothing (no device call on this GPU-less host)
    g.ar_compress(grads, codes, scales, b, count=0, stream=0)
    g.ar_compressed_reduce(codes, scales, outs, b, count=0, stream=0)
    g.ar_compressed_allreduce(grads, b, residuals=res, outs=grads, count=0, stream=0)


def test_bind_validates_without_touching_the_device(g):
    plan = g.ar_plan(4, 1024, "f32", "ring")
    good = [0x100000 * (r + 1) for r in range(4)]
    for bufs in ([0] + good[1:], [good[0] + 4] + good[1:], [good[0]] * 4):
        with pytest.raises(g.ArError) as e:
            g.ar_bind(plan, bufs)
        assert e.value.status == g.AR_EINVAL
    wplan = g.ar_plan(4, 1024, "bf16", "ring")
    with pytest.raises(g.ArError) as e:  # bf16 step plans need a workspace
        g.ar_bind(wplan, good)
    assert e.value.status == g.AR_EINVAL
    empty = g.ar_plan(4, 0, "f32", "ring")
    b = g.ar_bind(empty, good)  # count 0: no graph, no CUDA call
    g.ar_execute_bound(b, stream=0)
    del b
    with pytest.raises(g.ArError):
        g._check(g._lib.load().ar_execute_bound(None, None), "ar_execute_bound")


def test_plan_query_makes_no_device_call(g):
    # A plan that never ran reports nothing, without any CUDA call (there is
    # no GPU here); an empty execution does not count as running.
    plan = g.ar_plan(4, 1024, "f32", "ring")
    assert g.ar_plan_query(plan) == g.AR_OK
    empty = g.ar_plan(4, 0, "f32", "fused")
    g.ar_execute(empty, [0x100000 * (r + 1) for r in range(4)], stream=0)
    assert g.ar_plan_query(empty) == g.AR_OK
    assert g._lib.load().ar_plan_query(None) == g.AR_EINVAL


def test_small_step_plans_are_one_launch(g):
    # a step plan whose every step moves at most 2048 elements runs the whole
    # schedule in one CTA: one launch, the same steps and bytes
    for algo, N, G, small_L in (("ring", 16, 0, 2048), ("rabenseifner", 16, 0, 256), ("hier", 8, 4, 1024),
                                ("recdoubling", 4, 0, 1024)):
        small = g.ar_plan(N, small_L, "f32", algo, group_size=G).stats
        big = g.ar_plan(N, small_L + 1, "f32", algo, group_size=G).stats
        assert small["launches"] == 1 and big["launches"] == big["steps"] >= small["steps"] > 0, algo
        assert small["hbm_bytes"] < big["hbm_bytes"]
    assert g.ar_plan(16, 2048, "bf16", "ring").stats["launches"] == 1
    assert g.ar_plan(64, 20, "f32", "ring").stats["launches"] == 126  # 126 x 64 transfers: too many for one table
    assert g.ar_plan(1, 100, "f32", "ring").stats["launches"] == 0
