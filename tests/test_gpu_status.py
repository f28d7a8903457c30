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


def test_selftest_rejects_zero_polls(g):
    with pytest.raises(g.ArError):
        g.ar_selftest_wait_timeout(polls=0)
