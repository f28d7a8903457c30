"""ar_execute_noalloc: the all-reduce for callers that cannot allocate device
memory (their memory belongs to another allocator, or cudaMalloc could
synchronise the device on their path). It must give exactly what ar_execute
gives with a caller-provided workspace, call after call, although every call
reuses the library's one static workspace array and finds the previous call's
leftovers in it.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


@pytest.mark.parametrize("algo,G", [("ring", 0), ("hier", 4), ("rabenseifner", 0)])
def test_noalloc_matches_ar_execute_on_two_calls_in_a_row(g, algo, G):
    N, L = 8, 100_003
    plan = g.ar_plan(N, L, "bf16", algo, group_size=G)
    assert 0 < plan.stats["workspace_bytes"] <= g.AR_STATIC_WORKSPACE_BYTES
    inputs = [workloads.all_ranks(workloads.small_spec(N, L, "bf16", "normal", seed=100 + call))
              for call in range(2)]
    # reference: the existing entry point with a workspace the caller allocated
    want = []
    for x in inputs:
        bufs = [to_device(x[r], "bf16") for r in range(N)]
        ws = g.workspace_for(plan)
        g.ar_execute(plan, bufs, workspace=ws)
        torch.cuda.synchronize()
        want.append([to_host(b, "bf16") for b in bufs])
    # the no-allocation entry point, twice in a row on one stream
    got = []
    for x in inputs:
        bufs = [to_device(x[r], "bf16") for r in range(N)]
        g.ar_execute_noalloc(plan, bufs)
        got.append(bufs)
    torch.cuda.synchronize()
    for call in range(2):
        for r in range(N):
            assert_bits_equal(to_host(got[call][r], "bf16"), want[call][r], f"call {call} rank {r}")


def test_noalloc_out_of_place_and_no_workspace_plans(g):
    N, L = 4, 4099
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "uniform", seed=5))
    for algo in ("fused", "ring"):  # plans that need no workspace run as with ar_execute
        plan = g.ar_plan(N, L, "f32", algo)
        a = [to_device(x[r], "f32") for r in range(N)]
        b = [to_device(x[r], "f32") for r in range(N)]
        outs = [torch.empty_like(t) for t in b]
        g.ar_execute(plan, a)
        g.ar_execute_noalloc(plan, b, outs=outs)
        torch.cuda.synchronize()
        for r in range(N):
            assert_bits_equal(to_host(outs[r], "f32"), to_host(a[r], "f32"), f"{algo} rank {r}")
            np.testing.assert_array_equal(to_host(b[r], "f32"), x[r])


def test_noalloc_rejects_plans_larger_than_its_workspace(g):
    N = 16
    L = g.AR_STATIC_WORKSPACE_BYTES // (4 * N) + 64  # one more row of partials than fits
    plan = g.ar_plan(N, L, "bf16", "ring")
    assert plan.stats["workspace_bytes"] > g.AR_STATIC_WORKSPACE_BYTES
    bufs = [torch.empty(L, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    with pytest.raises(g.ArError) as e:
        g.ar_execute_noalloc(plan, bufs)
    assert e.value.status == g.AR_EINVAL
