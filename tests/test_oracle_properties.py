"""The oracle against mathematics: exact sums, error bounds, cross-checks between
independent formulations, and bf16 rounding against its format definition."""

import functools

import numpy as np
import pytest

import workloads
from oracle import buckets, chunks, numerics, schedules

U32 = 2.0 ** -24  # unit roundoff of fp32


def _inputs(N, L, dist="uniform", seed=0):
    return workloads.all_ranks(workloads.small_spec(N, L, dist=dist, seed=seed), threads=1)


def _algorithms(N):
    out = [("ring", lambda x, **k: schedules.ring_allreduce(x, **k), "ring", {})]
    if N & (N - 1) == 0:
        out.append(("rabenseifner", lambda x, **k: schedules.rabenseifner_allreduce(x, **k), "tree", {}))
    for G in range(1, N + 1):
        if N % G == 0:
            out.append((f"hier G={G}",
                        lambda x, G=G, **k: schedules.hierarchical_allreduce(x, G, **k), "hier",
                        {"group_size": G}))
    return out


BRUTE = [(N, L) for N in range(1, 9) for L in (1, 2, 3, 5, 7, 8, 13, 16, 31, 64)]


@pytest.mark.parametrize("N,L", BRUTE)
def test_brute_force_every_algorithm(N, L):
    """Every schedule, every rank: bitwise identical across ranks, within the
    Higham bound (N-1)*u*sum|g| of the fp64 sum, and bitwise equal to the fused
    sum in that schedule's order (an independent formulation)."""
    x = _inputs(N, L, seed=N * 100 + L)
    ref = numerics.reference_sum_f64(x)
    bound = (N - 1) * U32 * numerics.abs_sum_f64(x)
    for name, fn, order, kw in _algorithms(N):
        out, st = fn(x)
        for r in range(1, N):
            np.testing.assert_array_equal(out[r].view(np.uint32), out[0].view(np.uint32), err_msg=name)
        assert np.all(np.abs(out[0].astype(np.float64) - ref) <= bound), name
        fused = numerics.fused_sum(x, order, **kw)
        np.testing.assert_array_equal(out[0].view(np.uint32), fused.view(np.uint32), err_msg=name)


@pytest.mark.parametrize("N", [2, 3, 4, 8, 16])
def test_integer_inputs_are_exact(N):
    """Integers in [-8, 8]: every partial sum is an exactly representable integer,
    so every algorithm and every order equals the direct sum bit for bit."""
    L = 1000 + N
    x = _inputs(N, L, dist="int")
    want = numerics.reference_sum_f64(x).astype(np.float32)
    for name, fn, order, kw in _algorithms(N):
        out, _ = fn(x)
        np.testing.assert_array_equal(out, np.broadcast_to(want, out.shape), err_msg=name)
    for order in ["ring", "rank"] + (["tree"] if N & (N - 1) == 0 else []):
        np.testing.assert_array_equal(numerics.fused_sum(x, order), want)


def test_ring_order_is_left_fold_from_chunk_rank():
    """The ring carries chunk c from rank c around to rank c-1; check the fold
    order against a per-element brute force with Python fp32 scalars."""
    N, L = 5, 17
    x = _inputs(N, L, dist="normal", seed=7)
    out, _ = schedules.ring_allreduce(x)
    c_of = chunks.chunk_of(np.arange(L), L, N)
    for e in range(L):
        c = int(c_of[e])
        acc = np.float32(x[c, e])
        for i in range(1, N):
            acc = np.float32(acc + x[(c + i) % N, e])
        assert acc.view(np.uint32) == out[0, e].view(np.uint32)


def test_orders_differ_in_low_bits():
    """The orders are genuinely different (otherwise the bit-exact tests above
    could not tell a schedule from another)."""
    x = _inputs(8, 4096, dist="normal")
    r = numerics.fused_sum(x, "ring")
    k = numerics.fused_sum(x, "rank")
    t = numerics.fused_sum(x, "tree")
    h = numerics.fused_sum(x, "hier", group_size=4)
    assert (r != k).any() and (r != t).any() and (k != t).any() and (h != r).any()


@pytest.mark.parametrize("name", ["ring", "rabenseifner", "hier"])
def test_sampled_run_equals_full_run(name):
    fn = {"ring": schedules.ring_allreduce,
          "rabenseifner": schedules.rabenseifner_allreduce,
          "hier": functools.partial(schedules.hierarchical_allreduce, group_size=4)}[name]
    N, L = 8, 1003
    x = _inputs(N, L, dist="normal", seed=3)
    full, st_full = fn(x)
    rng = np.random.default_rng(1)
    idx = np.sort(rng.choice(L, 97, replace=False))
    part, st = fn(x[:, idx], idx=idx, L=L)
    np.testing.assert_array_equal(part, full[:, idx])
    np.testing.assert_array_equal(st.elements_sent, st_full.elements_sent)
    assert st.steps == st_full.steps


def test_scale_and_bf16_finish_applied_once():
    N, L = 8, 999
    x = _inputs(N, L, dist="normal")
    out, _ = schedules.ring_allreduce(x, finish=schedules.finish_scale(0.125))
    np.testing.assert_array_equal(out[3], numerics.fused_sum(x, "ring", scale=0.125))
    xb = numerics.bf16_to_f32(numerics.f32_to_bf16_rne(x))
    out, _ = schedules.hierarchical_allreduce(xb, 4, finish=schedules.finish_bf16())
    want = numerics.bf16_to_f32(numerics.f32_to_bf16_rne(numerics.fused_sum(xb, "hier", group_size=4)))
    np.testing.assert_array_equal(out, np.broadcast_to(want, out.shape))


# ----------------------------------------------------------------- bf16


def _f(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("f32_bits,bf16_bits", [
    (0x3F800000, 0x3F80),  # 1.0 exactly
    (0x3F808000, 0x3F80),  # 1 + 2^-8: halfway, last kept bit 0 -> stays (ties to even)
    (0x3F818000, 0x3F82),  # 1 + 3*2^-8: halfway, last kept bit 1 -> rounds up to even
    (0x3F808001, 0x3F81),  # just above halfway -> up
    (0x3F807FFF, 0x3F80),  # just below halfway -> down
    (0xBF818000, 0xBF82),  # negative tie, odd -> away from zero to even
    (0xBF808000, 0xBF80),  # negative tie, even -> stays
    (0x3F7FFFFF, 0x3F80),  # carry into the exponent: 0.99999994 -> 1.0
    (0x7F7FFFFF, 0x7F80),  # largest fp32 is past the last bf16 midpoint -> +inf
    (0x7F7F7FFF, 0x7F7F),  # below that midpoint -> largest bf16
    (0x00008000, 0x0000),  # subnormal tie, even
    (0x00018000, 0x0002),  # subnormal tie, odd -> up
    (0x80000000, 0x8000),  # -0 keeps its sign
])
def test_bf16_rne_hand_built(f32_bits, bf16_bits):
    assert int(numerics.f32_to_bf16_rne(_f(f32_bits))[0]) == bf16_bits


def test_bf16_widen_then_narrow_is_identity():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = numerics.bf16_to_f32(bits)
    finite = np.isfinite(f)
    np.testing.assert_array_equal(numerics.f32_to_bf16_rne(f[finite]), bits[finite])
    # widening is exact: the low half of the fp32 word is zero
    assert np.all((f.view(np.uint32) & 0xFFFF) == 0)


def test_bf16_rne_matches_torch_conversion():
    """Cross-check with an independent implementation of the same rounding."""
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32),
        (rng.standard_normal(100_000) * 1e-3).astype(np.float32),
        # exact ties (low 16 bits 0x8000) over many exponents, both signs
        ((rng.integers(0x0080, 0xFF00, 20_000, dtype=np.uint32) << np.uint32(16)) | np.uint32(0x8000))
        .view(np.float32),
    ])
    x = x[np.isfinite(x)]
    want = workloads.f32_to_bf16_bits_torch(x)
    np.testing.assert_array_equal(numerics.f32_to_bf16_rne(x), want)


def test_bf16_rne_error_bound():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(50_000).astype(np.float32)
    y = numerics.bf16_to_f32(numerics.f32_to_bf16_rne(x)).astype(np.float64)
    assert np.all(np.abs(y - x) <= 2.0 ** -9 * 2 * np.abs(x.astype(np.float64)))


# ----------------------------------------------------------------- buckets


def test_transformer_bucket_layout():
    tensors = workloads.transformer_tensors()
    counts = [c for _, c in tensors]
    names = [n for n, _ in tensors]
    assert sum(counts) == 1_139_343_360
    plan = buckets.bucket_plan(counts, 2, workloads.BUCKET_CAP_BYTES)
    assert len(plan) == 81
    flat = [t for b in plan for t in b]
    assert sorted(flat) == list(range(len(counts)))  # every tensor exactly once
    assert flat == list(reversed(range(len(counts))))  # reverse forward order
    sizes = sorted(sum(counts[t] for t in b) for b in plan)
    want = sorted([16_777_216] * 48 + [12_584_960] * 16 + [4_196_352] * 16 + [65_536_000])
    assert sizes == want
    assert [names[t] for t in plan[0]] == ["layers.15.w2"]
    assert [names[t] for t in plan[3]] == ["layers.15.norm2", "layers.15.wo", "layers.15.wv", "layers.15.wk"]
    assert [names[t] for t in plan[4]] == ["layers.15.wq", "layers.15.norm1"]
    assert [names[t] for t in plan[-1]] == ["embedding"]
    cap = workloads.BUCKET_CAP_BYTES // 2
    for b in plan:  # only single oversize tensors exceed the cap
        assert sum(counts[t] for t in b) <= cap or len(b) == 1


@pytest.mark.parametrize("cap", [1, 10, 37, 1000])
def test_bucket_plan_invariants(cap):
    rng = np.random.default_rng(cap)
    counts = rng.integers(1, 50, 40).tolist()
    plan = buckets.bucket_plan(counts, 2, cap * 2)
    flat = [t for b in plan for t in b]
    assert flat == list(reversed(range(len(counts))))
    for i, b in enumerate(plan):
        size = sum(counts[t] for t in b)
        assert size <= cap or len(b) == 1
        if i + 1 < len(plan):  # greedy: the next tensor did not fit
            assert size + counts[plan[i + 1][0]] > cap


def test_bucketed_sync_integer_mean():
    """Integer gradients on 8 ranks: the fp32 sums are exact, and x 1/8 is exact,
    so each output is the bf16 rounding of the exact mean."""
    N = 8
    counts = [5, 17, 3, 64, 9]
    rng = np.random.default_rng(2)
    grads = [[numerics.f32_to_bf16_rne(rng.integers(-8, 9, c).astype(np.float32)) for c in counts]
             for _ in range(N)]
    plan = buckets.bucket_plan(counts, 2, 60)
    for b in plan:
        res = buckets.sync_bucket(grads, b, counts, 0.125)
        for t in b:
            vals = np.stack([numerics.bf16_to_f32(grads[r][t]) for r in range(N)])
            mean = numerics.reference_sum_f64(vals) / 8
            want = workloads.f32_to_bf16_bits_torch(mean.astype(np.float32))
            for r in range(N):
                np.testing.assert_array_equal(res[(t, 0)][r], want)


def test_bucketed_sync_windows_match_full():
    N = 4
    counts = [100, 37, 250]
    rng = np.random.default_rng(3)
    grads = [[numerics.f32_to_bf16_rne(rng.standard_normal(c).astype(np.float32)) for c in counts]
             for _ in range(N)]
    b = [2, 1, 0]
    full = buckets.sync_bucket(grads, b, counts, 0.25)
    wins = [(2, 10, 40), (1, 0, 37), (0, 90, 100)]
    part_grads = [{(t, lo): grads[r][t][lo:hi] for t, lo, hi in wins} for r in range(N)]
    part = buckets.sync_bucket(part_grads, b, counts, 0.25, windows=wins)
    for t, lo, hi in wins:
        np.testing.assert_array_equal(part[(t, lo)], full[(t, 0)][:, lo:hi])


def test_bucket_sum_order_is_ring_over_packed_bucket():
    """The bucket's elements are summed in ring order over the packed bucket:
    chunk boundaries follow the bucket length, not the tensor boundaries."""
    N = 4
    counts = [7, 5]
    rng = np.random.default_rng(4)
    grads = [[numerics.f32_to_bf16_rne(rng.standard_normal(c).astype(np.float32)) for c in counts]
             for _ in range(N)]
    b = [1, 0]
    res = buckets.sync_bucket(grads, b, counts, 1.0)
    packed = np.stack([np.concatenate([numerics.bf16_to_f32(grads[r][t]) for t in b]) for r in range(N)])
    want = numerics.f32_to_bf16_rne(numerics.fused_sum(packed, "ring"))
    np.testing.assert_array_equal(res[(1, 0)][0], want[:5])
    np.testing.assert_array_equal(res[(0, 0)][0], want[5:])


def test_workload_blocks_are_addressable():
    spec = workloads.small_spec(3, 3 * workloads.BLOCK + 17, dist="normal")
    full = workloads.rank_buffer(spec, 2)
    lo, hi = workloads.BLOCK - 5, 2 * workloads.BLOCK + 9
    np.testing.assert_array_equal(workloads.rank_buffer(spec, 2, lo, hi), full[lo:hi])
    assert full.dtype == np.float32 and abs(float(full.std()) - 1e-3) < 2e-5
