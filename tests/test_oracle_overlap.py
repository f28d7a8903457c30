"""The critical-path model of overlapped communication against the AI Infra
Book's printed timelines (§7.6.1, §7.6.2)."""

import pytest

from oracle import overlap


def _rows(golden, kind):
    out = []
    for key, val in golden("overlap_model.txt"):
        if key == kind:
            f = dict(kv.split("=") for kv in val.split())
            out.append(f)
    return out


def test_readiness_skew(golden):
    for f in _rows(golden, "skew"):
        ready = [float(v) for v in f["ready_ms"].split(",")]
        got = overlap.group_completion(ready, float(f["exchange_ms"]))
        assert got == pytest.approx(float(f["done_ms"]), abs=0.05)


def test_sequential_and_overlapped_steps(golden):
    for f in _rows(golden, "sequential"):  # ready when the computation ends: no overlap
        got = overlap.step_time([float(f["compute_ms"])], [float(f["comm_ms"])], float(f["compute_ms"]),
                                float(f["update_ms"]))
        assert got == pytest.approx(float(f["step_ms"]), abs=0.05)
    for f in _rows(golden, "overlap"):
        got = overlap.step_time([float(f["ready_ms"])], [float(f["comm_ms"])], float(f["compute_ms"]),
                                float(f["update_ms"]))
        assert got == pytest.approx(float(f["step_ms"]), abs=0.05)


def test_latest_hidden_readiness(golden):
    f = _rows(golden, "latest_ready_hidden")[0]
    tc, tn, r = float(f["compute_ms"]), float(f["comm_ms"]), float(f["ready_ms"])
    assert overlap.exposed([r], [tn], tc) == pytest.approx(0.0, abs=1e-12)
    assert overlap.exposed([r + 0.01], [tn], tc) > 0


def test_communication_speedup_reduction(golden):
    f = _rows(golden, "reduction")[0]
    comm = 1 - 1.3 / 7.6
    step = 1 - 23.3 / 29.6
    assert round(comm * 100) == int(f["comm_pct"]) and round(step * 100) == int(f["step_pct"])
    # the whole-step speedup formula gives the same step: T_c = 22 ms unaffected, T_n = 7.6 ms, s = 7.6/1.3
    assert overlap.speedup(22.0, 7.6, 7.6 / 1.3) == pytest.approx(29.6 / 23.3, rel=1e-12)


def test_buckets_serialise_on_one_stream():
    # three buckets ready at 1, 2, 3 taking 2 each: 1-3, 3-5, 5-7
    assert overlap.comm_timeline([1, 2, 3], [2, 2, 2]) == [(1, 3), (3, 5), (5, 7)]
    assert overlap.step_time([1, 2, 3], [2, 2, 2], compute_end=4.0, update=1.0) == 8.0
    assert overlap.exposed([1, 2, 3], [2, 2, 2], compute_end=4.0) == 3.0
    # communication shorter than the gaps: only the last bucket's tail shows
    assert overlap.exposed([1, 2, 3], [0.5, 0.5, 0.5], compute_end=3.2) == pytest.approx(0.3)
