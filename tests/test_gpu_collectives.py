"""GPU parity of the standalone reduce-scatter and all-gather (ZeRO/FSDP halves)
against the oracle: step-by-step ring and fused single pass, fp32 and bf16, in
place and out of place, ragged chunk boundaries."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, to_device, to_host, widened
from oracle import numerics, schedules
from oracle.chunks import chunk_bounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


SIZES = [(1, 9), (2, 7), (3, 1000), (4, 4099), (8, 20003), (16, 100003), (64, 5000)]


def _run(g, x, dtype, algo, coll, order="ring", scale=1.0, out_of_place=False, kernel="auto", sm_budget=0):
    N, L = x.shape
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [torch.full_like(d, 7.0) for d in devs] if out_of_place else None
    plan = g.ar_plan(N, L, dtype, algo, order=order, scale=scale, collective=coll, kernel=kernel,
                     sm_budget=sm_budget)
    ws = g.workspace_for(plan)
    if ws is not None:
        ws.fill_(0xFF)
    g.ar_execute(plan, devs, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    if out_of_place:
        for r in range(N):
            np.testing.assert_array_equal(to_host(devs[r], dtype), x[r])
    return [to_host(t, dtype) for t in (outs if out_of_place else devs)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,order,sm_budget", [("ring", "ring", 0), ("fused", "ring", 0), ("fused", "rank", 0),
                                                  ("fused", "tree", 0), ("fused", "ring", 7), ("fused", "rank", 7),
                                                  ("fused", "tree", 7)])
@pytest.mark.parametrize("N,L", SIZES)
def test_reduce_scatter(g, dtype, algo, order, sm_budget, N, L):
    """Every rank's own chunk of the reduced sum; held to a few SMs the fused
    pass runs the kernel that loads the next tile during this tile's store."""
    if order == "tree" and N & (N - 1):
        pytest.skip("tree order needs a power-of-two rank count")
    scale = 0.25 if L % 2 else 1.0
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=N + 3 * L))
    got = _run(g, x, dtype, algo, "reduce_scatter", order, scale, out_of_place=(N % 2 == 0), sm_budget=sm_budget)
    xf = widened(x, dtype)
    if algo == "ring":
        finish = schedules.finish_bf16(scale) if dtype == "bf16" else schedules.finish_scale(scale)
        out, _ = schedules.ring_reduce_scatter(xf, finish=finish)
        want_rows = [numerics.f32_to_bf16_rne(out[r]) if dtype == "bf16" else out[r] for r in range(N)]
    else:
        s = numerics.fused_sum(xf, "ring_rs" if order == "ring" else order, scale=scale)
        w = numerics.f32_to_bf16_rne(s) if dtype == "bf16" else s
        want_rows = [w] * N
    b = chunk_bounds(L, N)
    for r in range(N):
        seg = slice(b[r], b[r + 1])
        assert_bits_equal(got[r][seg], want_rows[r][seg], f"rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("algo,kernel", [("ring", "auto"), ("fused", "auto"), ("fused", "loads")])
@pytest.mark.parametrize("N,L", SIZES)
@pytest.mark.parametrize("out_of_place", [False, True])
def test_allgather(g, dtype, algo, kernel, N, L, out_of_place):
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "uniform", seed=N * 5 + L))
    got = _run(g, x, dtype, algo, "allgather", scale=3.0, out_of_place=out_of_place,  # scale is ignored
               kernel=kernel)
    want, _ = schedules.ring_allgather(x)
    b = chunk_bounds(L, N)
    assert np.array_equal(want[0], np.concatenate([x[c, b[c]:b[c + 1]] for c in range(N)]))
    for r in range(N):
        assert_bits_equal(got[r], want[r], f"rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,L", SIZES + [(5, 1), (7, 3), (16, 37), (12, (1 << 20) + 13)])
@pytest.mark.parametrize("out_of_place", [False, True])
def test_allgather_bulk_copies(g, dtype, N, L, out_of_place):
    """The all-gather through bulk copies (one load, N stores per tile) gives
    the oracle's result, ragged chunk heads and tails included, under an SM
    budget too."""
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "uniform", seed=N * 7 + L))
    want, _ = schedules.ring_allgather(x)
    for sm_budget in (0, 5):
        got = _run(g, x, dtype, "fused", "allgather", out_of_place=out_of_place, kernel="bulk", sm_budget=sm_budget)
        for r in range(N):
            assert_bits_equal(got[r], want[r], f"rank {r} (sm_budget {sm_budget})")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,L", [(3, 1000), (8, 20003), (16, 100003), (5, 3), (16, 1 << 16), (6, 30000)])
def test_ring_allgather_mixed_in_and_out_of_place(g, dtype, N, L):
    """Even ranks in place, odd ranks into separate outputs, in one call: the
    first ring step writes each sent chunk to the sender's own output only for
    the ranks whose output is separate (bf16 chunks with even bounds move as
    fp32 pairs). Every output is the oracle's and every separate input is left
    as it was."""
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "uniform", seed=N + L))
    devs = [to_device(x[r], dtype) for r in range(N)]
    outs = [d if r % 2 == 0 else torch.full_like(d, 7.0) for r, d in enumerate(devs)]
    plan = g.ar_plan(N, L, dtype, "ring", collective="allgather")
    g.ar_execute(plan, devs, outs=outs)
    torch.cuda.synchronize()
    want, _ = schedules.ring_allgather(x)
    for r in range(N):
        assert_bits_equal(to_host(outs[r], dtype), want[r], f"rank {r}")
        if r % 2:
            np.testing.assert_array_equal(to_host(devs[r], dtype), x[r])


def test_allgather_bulk_from_host_slabs(g):
    """ar_execute_host on pageable memory runs the all-gather in element-range
    slabs: each slab's chunk pieces go through the bulk pipeline."""
    N, L = 6, (3 << 20) + 17
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "uniform", seed=11))
    want, _ = schedules.ring_allgather(x)
    plan = g.ar_plan(N, L, "f32", "fused", collective="allgather", kernel="bulk")
    host_in = [torch.from_numpy(x[r].copy()) for r in range(N)]
    host_out = [torch.zeros(L) for _ in range(N)]
    dev = [torch.empty(L, device="cuda") for _ in range(N)]
    g.ar_execute_host(plan, host_in, host_out, dev)
    for r in range(N):
        assert_bits_equal(host_out[r].numpy(), want[r], f"rank {r}")


def test_allgather_bulk_full_size(g):
    """16 ranks x 192 MiB fp32, in the launch configuration the timings use:
    every output chunk is a bit-for-bit copy of its owner's chunk (the
    definition), checked on the device over the whole buffers."""
    N, L = 16, 50_331_648
    b = chunk_bounds(L, N)
    devs = [torch.randn(L, device="cuda") for _ in range(N)]
    outs = [torch.zeros_like(d) for d in devs]
    plan = g.ar_plan(N, L, "f32", "fused", collective="allgather", kernel="bulk")
    g.ar_execute(plan, devs, outs=outs)
    torch.cuda.synchronize()
    for r in range(N):
        for c in range(N):
            assert torch.equal(outs[r][b[c]:b[c + 1]].view(torch.int32), devs[c][b[c]:b[c + 1]].view(torch.int32))
    del devs, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_then_allgather_equals_allreduce(g, dtype):
    """The two halves in sequence give the all-reduce in the order of one
    hierarchical group of N, bit for bit (primer §4.1)."""
    N, L = 16, 1 << 20
    x = workloads.all_ranks(workloads.small_spec(N, L, dtype, "normal", seed=77))
    devs = [to_device(x[r], dtype) for r in range(N)]
    rs = g.ar_plan(N, L, dtype, "ring", collective="reduce_scatter")
    ag = g.ar_plan(N, L, dtype, "ring", collective="allgather")
    g.ar_execute(rs, devs, workspace=g.workspace_for(rs))
    g.ar_execute(ag, devs)
    torch.cuda.synchronize()
    plan = g.ar_plan(N, L, dtype, "fused", order="hier", group_size=N)
    ref = [to_device(x[r], dtype) for r in range(N)]
    g.ar_execute(plan, ref)
    torch.cuda.synchronize()
    for r in (0, 9):
        assert_bits_equal(to_host(devs[r], dtype), to_host(ref[r], dtype), f"rank {r}")
