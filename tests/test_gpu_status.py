"""The failure path of the bounded device-side waits, on the GPU without any
fault: a wait that nothing satisfies gives up, the status word reports a
timeout, and the context keeps working."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal, expected, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from gradient_sync_gb300 import build

    build.build()
    import gradient_sync_gb300 as g

    return g


def test_bounded_wait_times_out_and_reports(g):
    assert g.ar_device_status(clear=True) == g.AR_OK
    g.ar_selftest_wait_timeout(polls=2000)
    assert g.ar_device_status(clear=False) == g.AR_ETIMEOUT  # sticky
    assert g.ar_device_status(clear=True) == g.AR_ETIMEOUT
    assert g.ar_device_status(clear=True) == g.AR_OK
    # the context is still usable: a bulk-copy all-reduce runs and is right
    N, L = 8, 123_457
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=1))
    bufs = [to_device(x[r], "f32") for r in range(N)]
    g.ar_execute(g.ar_plan(N, L, "f32", "fused", kernel="bulk"), bufs)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(bufs[3], "f32"), expected("fused", "ring", x, "f32"), "after timeout")
    assert g.ar_device_status(clear=True) == g.AR_OK


def test_timeout_is_sticky_per_plan_and_blocks_execution_until_cleared(g):
    assert g.ar_device_status(clear=True) == g.AR_OK
    N, L = 4, 40_000
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=2))
    bufs = [to_device(x[r], "f32") for r in range(N)]
    fused = g.ar_plan(N, L, "f32", "fused")
    ring = g.ar_plan(N, L, "f32", "ring")
    idle = g.ar_plan(N, L, "f32", "fused")  # never executed
    g.ar_execute(fused, bufs)
    bound = g.ar_bind(ring, bufs)
    torch.cuda.synchronize()
    assert g.ar_plan_query(fused) == g.AR_OK
    assert g.ar_plan_query(ring) == g.AR_OK
    # a wait that nothing satisfies runs out; the host-visible word is read
    # without synchronising the device, once the stream has drained
    g.ar_selftest_wait_timeout(polls=2000)
    torch.cuda.synchronize()
    assert g.ar_plan_query(fused) == g.AR_ETIMEOUT
    assert g.ar_plan_query(ring) == g.AR_ETIMEOUT  # bound on this device
    assert g.ar_plan_query(idle) == g.AR_OK  # never ran on a device
    # every executing call refuses, and enqueues nothing
    y = [to_device(x[r], "f32") for r in range(N)]
    calls = [lambda: g.ar_execute(fused, y), lambda: g.ar_execute(ring, y),
             lambda: g.ar_execute_noalloc(ring, y), lambda: g.ar_execute_bound(bound),
             lambda: g.ar_bind(ring, y),
             lambda: g.ar_bucket_allreduce([[t] for t in y], [L], 0, 1, "f32", 1.0)]
    for call in calls:
        with pytest.raises(g.ArError) as e:
            call()
        assert e.value.status == g.AR_ETIMEOUT
    torch.cuda.synchronize()
    for r in range(N):
        np.testing.assert_array_equal(to_host(y[r], "f32"), x[r])
    assert g.ar_plan_query(fused) == g.AR_ETIMEOUT  # querying does not clear
    # clearing restores execution
    assert g.ar_device_status(clear=True) == g.AR_ETIMEOUT
    assert g.ar_plan_query(fused) == g.AR_OK
    assert g.ar_plan_query(ring) == g.AR_OK
    g.ar_execute(fused, y)
    torch.cuda.synchronize()
    assert_bits_equal(to_host(y[1], "f32"), expected("fused", "ring", x, "f32"), "after clearing")
    assert g.ar_device_status(clear=True) == g.AR_OK


def test_selftest_rejects_zero_polls(g):
    with pytest.raises(g.ArError):
        g.ar_selftest_wait_timeout(polls=0)
