"""Overlapped bucketed sync: the same bits as the sync without overlap and as
the oracle, whatever the SM budget; and the product's critical-path
prediction equals the oracle's model."""

import numpy as np
import pytest
import torch

import workloads
from _gpu import assert_bits_equal
from oracle import buckets as ob
from oracle import numerics
from oracle import overlap as omodel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ov():
    from gradient_sync_gb300 import build

    build.build()
    from gradient_sync_gb300 import overlap

    return overlap


@pytest.mark.parametrize("sm_budget", [0, 4, 37])
def test_overlapped_sync_matches_serial_and_oracle(ov, sm_budget):
    N = 4
    tensors = workloads.transformer_tensors(layers=2, hidden=256, ffn=1024, vocab=1000)
    counts = [c for _, c in tensors]
    rng = np.random.default_rng(sm_budget)
    host = [[numerics.f32_to_bf16_rne((rng.standard_normal(c) * 1e-3).astype(np.float32)) for c in counts]
            for _ in range(N)]

    def dev():
        return [[torch.from_numpy(h.view(np.int16)).cuda().view(torch.bfloat16) for h in row] for row in host]

    a, b = dev(), dev()
    cap = 2 * 300_000  # several buckets at this size
    red_a = ov.BucketedReducer(a, counts, cap_bytes=cap, sm_budget=sm_budget)
    red_b = ov.BucketedReducer(b, counts, cap_bytes=cap)
    bwd = ov.SyntheticBackward(tensors, tokens=512, hidden=256)
    bwd.run(red_a.ready)  # overlapped with the synthetic backward
    red_a.finish()
    red_b.sync_all()  # no overlap
    torch.cuda.synchronize()
    assert len(red_a.buckets) > 2
    for bk in ob.bucket_plan(counts, 2, cap):
        want = ob.sync_bucket(host, bk, counts, 1.0 / N)
        for t in bk:
            for r in range(N):
                got_a = a[r][t].view(torch.int16).cpu().numpy().view(np.uint16)
                got_b = b[r][t].view(torch.int16).cpu().numpy().view(np.uint16)
                assert_bits_equal(got_a, want[(t, 0)][r], f"overlapped t={t} r={r}")
                assert_bits_equal(got_b, got_a, f"serial t={t} r={r}")


def test_critical_path_matches_the_oracle_model(ov):
    rng = np.random.default_rng(3)
    for _ in range(50):
        k = int(rng.integers(1, 20))
        ready = np.sort(rng.uniform(0, 10, k)).tolist()
        dur = rng.uniform(0, 2, k).tolist()
        tc = float(rng.uniform(0, 15))
        assert ov.critical_path(ready, dur, tc) == pytest.approx(omodel.step_time(ready, dur, tc), rel=1e-12)


def test_sm_budget_does_not_change_results():
    import gradient_sync_gb300 as g
    from _gpu import expected, to_device, to_host

    N, L = 16, 1 << 20
    x = workloads.all_ranks(workloads.small_spec(N, L, "f32", "normal", seed=11))
    for algo in ("fused", "ring"):
        plan = g.ar_plan(N, L, "f32", algo, sm_budget=3)
        bufs = [to_device(x[r], "f32") for r in range(N)]
        g.ar_execute(plan, bufs)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(bufs[7], "f32"), expected(algo, "ring", x, "f32"), algo)
