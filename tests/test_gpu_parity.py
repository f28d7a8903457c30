"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by
element, bit for bit, at sizes the oracle finishes in seconds: several tiles,
ragged chunk boundaries and tails, tiny and degenerate cases."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, expected, to_device, to_host, widened
from oracle import numerics, schedules

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    assert torch.cuda.is_available()
    return g


SIZES = [(1, 5), (2, 1), (2, 2), (3, 7), (4, 1000), (5, 4099), (8, 20003), (16, 100003), (7, 3),
         (64, 4109), (64, 70), (16, 1 << 18)]


def _group(N):
    for G in (8, 4, 2, 3):
        if N % G == 0 and G < N:
            return G
    return N


def _run(g, x, dtype, algo, order="ring", group_size=0, scale=1.0, out_of_place=False):
    N, L = x.shape
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [torch.empty_like(d) for d in devs] if out_of_place else None
    plan = g.ar_plan(N, L, dtype, algo, group_size=group_size, order=order, scale=scale)
    ws = g.workspace_for(plan)
    if ws is not None:
        ws.fill_(0xFF)  # the workspace's contents on entry must not matter
    g.ar_execute(plan, devs, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    res = outs if out_of_place else devs
    got = [to_host(t, dtype) for t in res]
    if out_of_place:  # inputs untouched
        for r in range(N):
            np.testing.assert_array_equal(to_host(devs[r], dtype), x[r])
    return got


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["ring", "rank", "tree", "hier"])
@pytest.mark.parametrize("N,L", SIZES)
def test_fused_matches_oracle(g, dtype, order, N, L):
    if order == "tree" and N & (N - 1):
        pytest.skip("tree order needs a power-of-two rank count")
    G = _group(N) if order == "hier" else 0
    scale = 0.125 if (N + L) % 2 else 1.0
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=N * 7 + L))
    got = _run(g, x, dtype, "fused", order, G, scale, out_of_place=(L % 3 == 0))
    want = expected("fused", order, x, dtype, G, scale)
    for r in range(N):
        assert_bits_equal(got[r], want, f"rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["ring", "rabenseifner", "hier"])
@pytest.mark.parametrize("N,L", SIZES)
def test_step_executor_matches_oracle(g, dtype, algo, N, L):
    if algo == "rabenseifner" and N & (N - 1):
        pytest.skip("Rabenseifner needs a power-of-two rank count")
    G = _group(N) if algo == "hier" else 0
    scale = 0.5 if (N * L) % 3 == 1 else 1.0
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "uniform", seed=N * 11 + L))
    got = _run(g, x, dtype, algo, group_size=G, scale=scale, out_of_place=(L % 2 == 1))
    want = expected(algo, "ring", x, dtype, G, scale)
    for r in range(N):
        assert_bits_equal(got[r], want, f"rank {r}")


@pytest.mark.parametrize("N,G", [(16, 8), (8, 2), (8, 1), (8, 8), (12, 3), (64, 8)])
def test_hierarchical_shapes(g, N, G):
    L = 30011
    x = workloads.all_ranks(workloads.small_spec(N, L, "bf16", "normal", seed=G))
    want = expected("hier", "ring", x, "bf16", G)
    for algo, order in (("hier", "ring"), ("fused", "hier")):
        got = _run(g, x, "bf16", algo, order, G)
        for r in range(N):
            assert_bits_equal(got[r], want, f"{algo} rank {r}")


@pytest.mark.parametrize("algo,order", [("ring", "ring"), ("rabenseifner", "ring"), ("hier", "ring"),
                                        ("fused", "ring"), ("fused", "rank"), ("fused", "tree"),
                                        ("fused", "hier")])
def test_integer_inputs_exact(g, algo, order):
    """Integer inputs: every algorithm and order gives the exact sum."""
    N, L = 8, 262_147
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "int"))
    want = numerics.reference_sum_f64(x).astype(np.float32)
    got = _run(g, x, "f32", algo, order, group_size=4)
    for r in range(N):
        assert_bits_equal(got[r], want, f"rank {r}")


def test_fused_orders_reproduce_schedules_on_gpu(g):
    """The fused single pass in a schedule's order equals that schedule run
    step by step, bit for bit, on the GPU alone."""
    N, L = 16, 1 << 20
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=3))
    for algo, order, G in (("ring", "ring", 0), ("rabenseifner", "tree", 0), ("hier", "hier", 4)):
        a = _run(g, x, "f32", algo, group_size=G)
        b = _run(g, x, "f32", "fused", order, group_size=G)
        assert_bits_equal(a[5], b[5], algo)


def test_bf16_rounding_ties_on_gpu(g):
    """bf16 sums that land exactly halfway between two bf16 values round to
    even, as the format definition says: a bf16 value a plus half its ulp is
    exact in fp32 and a tie for bf16."""
    rng = np.random.default_rng(11)
    K = 8192
    a32 = (rng.uniform(1, 2, K) * 2.0 ** rng.integers(-30, 30, K) * rng.choice([-1, 1], K)).astype(np.float32)
    a16 = numerics.f32_to_bf16_rne(a32)
    a = numerics.bf16_to_f32(a16)
    e = np.floor(np.log2(np.abs(a.astype(np.float64))))
    half = (2.0 ** (e - 8) * rng.choice([-1, 1], K)).astype(np.float32)  # bf16 ulp is 2^(e-7)
    b16 = numerics.f32_to_bf16_rne(half)
    s = (a + numerics.bf16_to_f32(b16)).astype(np.float32)
    tie = (s.view(np.uint32) & np.uint32(0xFFFF)) == 0x8000
    assert tie.sum() > K // 3
    odd = (s.view(np.uint32) >> np.uint32(16)) & np.uint32(1)
    assert odd[tie].min() == 0 and odd[tie].max() == 1  # ties to both neighbours
    x = np.stack([a16[tie], b16[tie]])
    got = _run(g, x, "bf16", "fused", "rank")
    want = numerics.f32_to_bf16_rne(s[tie])
    assert_bits_equal(got[0], want, "ties")
    assert_bits_equal(got[1], want, "ties")


def test_buckets_pack_ring_unpack_and_fused(g):
    """Bucketed sync: pack + ring + unpack, and the fused no-pack pass, both
    against the oracle, with tensor sizes that leave ragged vectors and
    packed offsets that are not 16-byte aligned."""
    from oracle import buckets as ob

    N = 8
    counts = [5, 1000, 37, 4096, 9, 2051, 777, 64, 3, 10_000]
    scale = 1.0 / N
    rng = np.random.default_rng(7)
    grads = [[numerics.f32_to_bf16_rne((rng.standard_normal(c) * 1e-3).astype(np.float32)) for c in counts]
             for _ in range(N)]
    plan = ob.bucket_plan(counts, 2, 2 * 3000)
    of, nb = g.ar_bucket_plan(counts, 2, 2 * 3000)
    assert nb == len(plan)
    for b in plan:
        lo, hi = min(b), max(b) + 1
        assert sorted(b) == list(range(lo, hi))
        want = ob.sync_bucket(grads, b, counts, scale)
        Lb = sum(counts[t] for t in b)
        # path 1: pack -> ring (fp32) -> unpack
        dev = [[to_device(grads[r][t], "bf16") for t in range(len(counts))] for r in range(N)]
        bucket = [torch.empty(Lb, dtype=torch.float32, device="cuda") for _ in range(N)]
        g.ar_bucket_pack(dev, counts, lo, hi, "bf16", bucket)
        ring = g.ar_plan(N, Lb, "f32", "ring")
        g.ar_execute(ring, bucket)
        g.ar_bucket_unpack(bucket, scale, "bf16", dev, counts, lo, hi)
        torch.cuda.synchronize()
        for t in b:
            for r in range(N):
                assert_bits_equal(to_host(dev[r][t], "bf16"), want[(t, 0)][r], f"pack path t={t} r={r}")
        # path 2: fused, no pack buffer
        dev = [[to_device(grads[r][t], "bf16") for t in range(len(counts))] for r in range(N)]
        g.ar_bucket_allreduce(dev, counts, lo, hi, "bf16", scale)
        torch.cuda.synchronize()
        for t in b:
            for r in range(N):
                assert_bits_equal(to_host(dev[r][t], "bf16"), want[(t, 0)][r], f"fused t={t} r={r}")
        # tensors outside the bucket are untouched
        for t in range(len(counts)):
            if t not in b:
                assert_bits_equal(to_host(dev[0][t], "bf16"), grads[0][t], "outside bucket")


def test_pack_unpack_f32_roundtrip(g):
    N = 3
    counts = [17, 8, 1]
    rng = np.random.default_rng(1)
    grads = [[rng.standard_normal(c).astype(np.float32) for c in counts] for _ in range(N)]
    dev = [[to_device(grads[r][t], "f32") for t in range(3)] for r in range(N)]
    bucket = [torch.empty(26, dtype=torch.float32, device="cuda") for _ in range(N)]
    g.ar_bucket_pack(dev, counts, 0, 3, "f32", bucket)
    torch.cuda.synchronize()
    for r in range(N):  # descending tensor id inside the bucket
        np.testing.assert_array_equal(to_host(bucket[r], "f32"),
                                      np.concatenate([grads[r][2], grads[r][1], grads[r][0]]))
    g.ar_bucket_unpack(bucket, 2.0, "f32", dev, counts, 0, 3)
    torch.cuda.synchronize()
    for r in range(N):
        for t in range(3):
            np.testing.assert_array_equal(to_host(dev[r][t], "f32"), grads[r][t] * np.float32(2.0))


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("algo", ["fused", "ring"])
def test_execute_host_roundtrip(g, algo, pinned):
    """Host buffers in and out: pinned buffers are read and written directly by
    the fused kernel; pageable ones are staged through the device buffers in
    several slabs."""
    N, L = 4, 9 * (1 << 20) + 5
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=9))
    host_in = [torch.from_numpy(x[r].copy()) for r in range(N)]
    host_out = [torch.empty(L, dtype=torch.float32) for _ in range(N)]
    if pinned:
        host_in = [t.pin_memory() for t in host_in]
        host_out = [t.pin_memory() for t in host_out]
    dev = [torch.empty(L, dtype=torch.float32, device="cuda") for _ in range(N)]
    plan = g.ar_plan(N, L, "f32", algo, order="ring")
    g.ar_execute_host(plan, host_in, host_out, dev)
    want = expected(algo, "ring", x, "f32")
    for r in range(N):
        assert_bits_equal(host_out[r].numpy(), want, f"rank {r}")
        np.testing.assert_array_equal(host_in[r].numpy(), x[r])


def test_device_status_is_clear(g):
    assert g.ar_device_status(clear=True) == g.AR_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["ring", "rank", "tree", "hier"])
@pytest.mark.parametrize("N,L", [(2, 1), (2, 70001), (3, 7), (4, 1000), (5, 4099), (8, 20003), (16, 100003),
                                 (16, 1 << 18), (24, 50000), (12, 777)])
@pytest.mark.parametrize("sm_budget", [0, 7])
def test_fused_bulk_copy_pipeline_matches_oracle(g, dtype, order, N, L, sm_budget):
    """The bulk-copy (TMA) kernel gives the register pipeline's result, bit for
    bit, on the whole GPU and on a few SMs."""
    if order == "tree" and N & (N - 1):
        pytest.skip("tree order needs a power-of-two rank count")
    G = _group(N) if order == "hier" else 0
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=N * 3 + L))
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [torch.empty_like(d) for d in devs] if L % 2 else None
    plan = g.ar_plan(N, L, dtype, "fused", group_size=G, order=order, scale=0.5, sm_budget=sm_budget,
                     kernel="bulk")
    g.ar_execute(plan, devs, outs=outs)
    torch.cuda.synchronize()
    want = expected("fused", order, x, dtype, G, 0.5)
    for r in range(N):
        assert_bits_equal(to_host((outs or devs)[r], dtype), want, f"rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["ring", "rank", "hier", "tree"])
@pytest.mark.parametrize("N,L", [(1, 9), (1, 40001), (2, 70001), (3, 1001), (4, 12345), (5, 4099), (8, 20003),
                                 (12, 33333), (16, 100003), (32, 7777), (64, 5001)])
def test_fused_register_pipeline_with_sm_budget(g, dtype, order, N, L):
    """A launch held to fewer SMs than the GPU has runs the variants with more
    loads in flight per thread (in ring, rank and tree order the next tile's
    first batch is loaded during this tile's stores); their result is the
    oracle's, bit for bit, in and out of place."""
    if order == "hier" and N % 2:
        pytest.skip("the hierarchical order needs a group size that divides N")
    if order == "tree" and (N < 2 or N & (N - 1)):
        pytest.skip("the tree order needs a power-of-two rank count")
    G = _group(N) if order == "hier" else 0
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=N * 5 + L))
    want = expected("fused", order, x, dtype, G, 0.5)
    for out_of_place in (False, True):
        devs = [to_device(x[r], dtype) for r in range(N)]
        outs = [torch.empty_like(d) for d in devs] if out_of_place else None
        plan = g.ar_plan(N, L, dtype, "fused", group_size=G, order=order, scale=0.5, sm_budget=7, kernel="loads")
        g.ar_execute(plan, devs, outs=outs)
        torch.cuda.synchronize()
        for r in range(N):
            assert_bits_equal(to_host((outs or devs)[r], dtype), want, f"rank {r}")


@pytest.mark.parametrize("order", ["ring", "rank", "hier", "tree"])
def test_execute_host_slabs_with_sm_budget(g, order):
    """Pageable host buffers go through the device in slabs, one launch per
    element range; the ranges cut the ring's chunks mid-way, and the launches
    held to a few SMs still give the oracle's bits."""
    N, L = 8, 5 * (1 << 20) + 3
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=21))
    host_in = [torch.from_numpy(x[r].copy()) for r in range(N)]
    host_out = [torch.empty(L, dtype=torch.float32) for _ in range(N)]
    dev = [torch.empty(L, dtype=torch.float32, device="cuda") for _ in range(N)]
    G = 4 if order == "hier" else 0
    plan = g.ar_plan(N, L, "f32", "fused", order=order, group_size=G, sm_budget=6, kernel="loads")
    g.ar_execute_host(plan, host_in, host_out, dev)
    want = expected("fused", order, x, "f32", G)
    for r in range(N):
        assert_bits_equal(host_out[r].numpy(), want, f"rank {r}")


@pytest.mark.parametrize("kernel", ["auto", "loads", "bulk"])
@pytest.mark.parametrize("sm_budget", [0, 9])
def test_bucket_paths_with_sm_budget(g, sm_budget, kernel):
    from oracle import buckets as ob

    N = 8
    counts = [5, 1000, 37, 40960, 9, 2051, 777, 64, 3, 100_000]
    rng = np.random.default_rng(sm_budget + 1)
    grads = [[numerics.f32_to_bf16_rne((rng.standard_normal(c) * 1e-3).astype(np.float32)) for c in counts]
             for _ in range(N)]
    cap = 2 * 50_000
    dev = [[to_device(grads[r][t], "bf16") for t in range(len(counts))] for r in range(N)]
    for b in ob.bucket_plan(counts, 2, cap):
        lo, hi = min(b), max(b) + 1
        g.ar_bucket_allreduce(dev, counts, lo, hi, "bf16", 1.0 / N, sm_budget=sm_budget, kernel=kernel)
        torch.cuda.synchronize()
        want = ob.sync_bucket(grads, b, counts, 1.0 / N)
        for t in b:
            for r in range(N):
                assert_bits_equal(to_host(dev[r][t], "bf16"), want[(t, 0)][r], f"t={t} r={r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo", ["ring", "rabenseifner", "dbtree", "recdoubling"])
def test_step_executor_on_16_byte_aligned_buffers(g, dtype, algo):
    """Buffers that are 16- but not 32-byte aligned (views 16 bytes into a
    larger allocation) take the 16-byte access path of the step kernel; the
    result is the same bits."""
    N, L = 8, 20011
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=41))
    esz = 2 if dtype == "bf16" else 4
    shift = 16 // esz
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    big = [torch.empty(L + 64, dtype=tdt, device="cuda") for _ in range(N)]
    devs = [b[shift:shift + L] for b in big]
    for r in range(N):
        devs[r].copy_(to_device(x[r], dtype))
        assert devs[r].data_ptr() % 32 == 16
    plan = g.ar_plan(N, L, dtype, algo, scale=0.5)
    ws = g.workspace_for(plan)
    g.ar_execute(plan, devs, workspace=ws)
    torch.cuda.synchronize()
    want = expected(algo, "ring", x, dtype, scale=0.5)
    for r in range(N):
        assert_bits_equal(to_host(devs[r].contiguous(), dtype), want, f"rank {r}")


@pytest.mark.parametrize("sm_budget", [0, 5])
@pytest.mark.parametrize("N,dtype", [(8, "bf16"), (12, "f32"), (5, "bf16"), (2, "f32"), (4, "bf16")])
@pytest.mark.parametrize("aligned32", [True, False])
def test_bucket_allreduce_vector_widths(g, aligned32, N, dtype, sm_budget):
    """The fused bucket pass moves 32-byte vectors when every tensor is
    32-byte aligned (more than 4 ranks) and 16-byte vectors otherwise
    (tensors placed 16 bytes into larger allocations); both give the oracle's
    bits, ragged tensor sizes included, at full width and held to a few SMs
    (the kernels that load the next tile during this tile's stores)."""
    from oracle import buckets as ob

    counts = [5, 1000, 37, 4096, 9, 2051, 777, 64, 3, 30_011]
    scale = 1.0 / N
    rng = np.random.default_rng(17 + N)
    host = [[(rng.standard_normal(c) * 1e-3).astype(np.float32) for c in counts] for _ in range(N)]
    if dtype == "bf16":
        host = [[numerics.f32_to_bf16_rne(a) for a in row] for row in host]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    shift = 0 if aligned32 else 16 // (2 if dtype == "bf16" else 4)  # 16 bytes
    keep, dev = [], []
    for r in range(N):
        row = []
        for t, c in enumerate(counts):
            big = torch.empty(c + 64, dtype=tdt, device="cuda")
            keep.append(big)
            v = big[shift:shift + c]
            v.copy_(to_device(host[r][t], dtype))
            assert (v.data_ptr() % 32 == 0) == aligned32
            row.append(v)
        dev.append(row)
    lo, hi = 0, len(counts)
    g.ar_bucket_allreduce(dev, counts, lo, hi, dtype, scale, sm_budget=sm_budget)
    torch.cuda.synchronize()
    bucket = list(range(hi - 1, lo - 1, -1))  # packed in reverse forward order
    if dtype == "bf16":
        want = ob.sync_bucket(host, bucket, counts, scale)
    else:  # fp32 packs as is: the ring all-reduce of the packed bucket, times the scale
        offs = ob.bucket_offsets(bucket, counts)
        Lb = sum(counts[t] for t in bucket)
        packed = np.zeros((N, Lb), np.float32)
        for r in range(N):
            for t in bucket:
                packed[r, offs[t]:offs[t] + counts[t]] = host[r][t]
        reduced, _ = schedules.ring_allreduce(packed)
        out = reduced * np.float32(scale)
        want = {(t, 0): out[:, offs[t]:offs[t] + counts[t]] for t in bucket}
    for t in range(lo, hi):
        for r in range(N):
            assert_bits_equal(to_host(dev[r][t].contiguous(), dtype), want[(t, 0)][r], f"t={t} r={r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,order", [("fused", "ring"), ("fused", "tree"), ("ring", "ring"),
                                        ("rabenseifner", "ring"), ("hier", "ring"), ("dbtree", "ring")])
def test_mixed_in_and_out_of_place(g, dtype, algo, order):
    """outs[r] may equal bufs[r] rank by rank: even ranks in place, odd ranks
    into separate outputs, in one call. Every rank gets the oracle's bits and
    the odd ranks' inputs are untouched."""
    N, L = 8, 50_021
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=23))
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [devs[r] if r % 2 == 0 else torch.empty_like(devs[r]) for r in range(N)]
    plan = g.ar_plan(N, L, dtype, algo, order=order, group_size=4 if algo == "hier" else 0, scale=0.25)
    ws = g.workspace_for(plan)
    g.ar_execute(plan, devs, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    want = expected(algo, order, x, dtype, group_size=4 if algo == "hier" else 0, scale=0.25)
    for r in range(N):
        assert_bits_equal(to_host(outs[r], dtype), want, f"rank {r}")
        if r % 2:
            np.testing.assert_array_equal(to_host(devs[r], dtype), x[r])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,N,G,dims", [("ring", 16, 0, None), ("rabenseifner", 8, 0, None), ("hier", 8, 4, None),
                                           ("recdoubling", 4, 0, None), ("dbtree", 6, 0, None),
                                           ("torus", 8, 0, (2, 4))])
def test_one_cta_and_per_step_executors_agree(g, algo, N, G, dims, dtype):
    """Plans whose steps move at most 2048 elements run every step in one CTA
    with a block barrier per step; larger ones run one kernel per step. Both
    give the oracle's bits, in place and out of place, around the boundary."""
    for L in (5, 256, 257, 777, 1024, 1025, 2048, 2049, 8193):
        x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=L + N))
        want = expected(algo, "ring", x, dtype, group_size=G, scale=0.5, torus_dims=dims)
        plan = g.ar_plan(N, L, dtype, algo, group_size=G, scale=0.5, torus_dims=dims or (0, 0, 0))
        assert plan.stats["launches"] in (1, plan.stats["steps"])
        for out_of_place in (False, True):
            bufs = [to_device(x[r], dtype) for r in range(N)]
            outs = [torch.empty_like(b) for b in bufs] if out_of_place else None
            g.ar_execute(plan, bufs, outs=outs, workspace=g.workspace_for(plan))
            torch.cuda.synchronize()
            for r in range(N):
                got = to_host((outs if out_of_place else bufs)[r], dtype)
                assert_bits_equal(got, want, f"{algo} L={L} rank {r} {'out' if out_of_place else 'in'}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,coll,N,G,L", [
    ("ring", "allreduce", 16, 0, 256), ("ring", "allreduce", 16, 0, 2048),
    ("ring", "allreduce", 16, 0, 1280), ("ring", "allreduce", 16, 0, 1281), ("rabenseifner", "allreduce", 64, 0, 64),
    ("rabenseifner", "allreduce", 8, 0, 100), ("hier", "allreduce", 8, 4, 300), ("dbtree", "allreduce", 6, 0, 77),
    ("ring", "reduce_scatter", 16, 0, 1000), ("ring", "allgather", 16, 0, 999)])
def test_one_cta_plans_on_and_off_chip(g, dtype, algo, coll, N, G, L):
    """Plans whose steps all fit one CTA run with their buffers in shared
    memory when 8 bytes per element and rank fit in 160 KiB (16 x 1280
    elements does, 16 x 1281 does not), else from global memory. Either way:
    the oracle's bits on every rank (a reduce-scatter: in the chunk each
    rank owns), with even ranks in place and odd ranks out of place in one
    call, and the odd ranks' inputs untouched."""
    from oracle.chunks import chunk_bounds

    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=N * 1000 + L))
    plan = g.ar_plan(N, L, dtype, algo, group_size=G, scale=0.5 if coll == "allreduce" else 1.0, collective=coll)
    assert plan.stats["launches"] == 1
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [devs[r] if r % 2 == 0 else torch.full_like(devs[r], 7.0) for r in range(N)]
    ws = g.workspace_for(plan)
    g.ar_execute(plan, devs, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    xf = widened(x, dtype)
    b = chunk_bounds(L, N)
    if coll == "allreduce":
        want = expected(algo, "ring", x, dtype, group_size=G, scale=0.5)
        rows = [want] * N
    elif coll == "reduce_scatter":
        finish = schedules.finish_bf16(1.0) if dtype == "bf16" else None
        out, _ = schedules.ring_reduce_scatter(xf, finish=finish)
        rows = [numerics.f32_to_bf16_rne(out[r]) if dtype == "bf16" else out[r] for r in range(N)]
    else:
        out, _ = schedules.ring_allgather(x if dtype == "f32" else x)
        rows = [out[r] for r in range(N)]
    for r in range(N):
        got = to_host(outs[r], dtype)
        if coll == "reduce_scatter":
            seg = slice(b[r], b[r + 1])
            assert_bits_equal(got[seg], rows[r][seg], f"rank {r}")  # the rest is unspecified
        else:
            assert_bits_equal(got, rows[r], f"rank {r}")
        if r % 2:
            assert_bits_equal(to_host(devs[r], dtype), x[r], f"input of rank {r}")
