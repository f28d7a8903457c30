"""Pins of the oracle's blockwise INT8 compression and error feedback against
the numbers the compression section of Scaling ML Systems prints, exact
arithmetic and brute force."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import compress as C
from oracle import numerics

F32 = np.float32


def _rows(golden):
    return dict(golden("compression.txt"))


def test_message_size_and_ratio(golden):
    rows = _rows(golden)
    rng = np.random.default_rng(0)
    for d, b in ((1000, 128), (4096, 64), (129, 128), (1, 16), (5000, 1024)):
        q, s = C.quantize_blockwise(rng.standard_normal(d).astype(F32), b)
        assert q.nbytes + s.nbytes == C.message_bytes(d, b) == d + 4 * -(-d // b)
        assert q.dtype == np.int8 and s.dtype == np.float32
    assert round(C.compression_ratio(128), 2) == float(rows["ratio_b128"])
    for b in map(int, rows["typical_blocks"].split()):
        d = 1 << 20
        assert C.compression_ratio(b) == pytest.approx(4 * d / C.message_bytes(d, b), rel=1e-12)
    assert C.compression_ratio(1 << 30) == pytest.approx(float(rows["ratio_limit"]), rel=1e-8)


def _heavy(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n) * 1e-3
    out = rng.choice(n, max(1, n // 200), replace=False)
    x[out] *= rng.uniform(50, 500, out.size)  # a heavy tail
    return x.astype(F32)


@pytest.mark.parametrize("b", [16, 64, 128, 1024])
def test_error_within_half_a_block_scale(b, golden):
    """|x - code * scale| <= scale / 2, up to the fp32 rounding of the quotient
    and of the product."""
    half = float(_rows(golden)["max_error_in_scales"])
    x = _heavy(20_011, b)
    q, s = C.quantize_blockwise(x, b)
    err = np.abs(x.astype(np.float64) - C.dequantize(q, s, b).astype(np.float64))
    sb = np.repeat(s.astype(np.float64), b)[: x.size]
    assert np.all(err <= half * sb * (1 + 2.0 ** -20) + np.abs(x) * 2.0 ** -23)
    assert np.abs(q.astype(int)).max() <= int(_rows(golden)["int8_max_code"])
    for k in range(s.size):  # the block's largest element maps to the largest code
        assert np.abs(q[k * b:(k + 1) * b].astype(int)).max() == 127


def test_exact_grid_values():
    """Values k * 2^j with some |k| = 127 in every block: the scale is 2^j
    exactly, the codes are k and dequantization is exact."""
    rng = np.random.default_rng(1)
    b, nb = 64, 50
    k = rng.integers(-127, 128, b * nb)
    k[::b] = 127 * rng.choice([-1, 1], nb)
    j = np.repeat(rng.integers(-30, 10, nb), b)
    x = (k * np.exp2(j)).astype(F32)
    q, s = C.quantize_blockwise(x, b)
    np.testing.assert_array_equal(q, k.astype(np.int8))
    np.testing.assert_array_equal(s, np.exp2(j[::b]).astype(F32))
    np.testing.assert_array_equal(C.dequantize(q, s, b), x)


def test_codes_are_the_nearest_level_brute_force():
    """For every element the code is the integer q in [-127, 127] nearest to x
    in exact rational arithmetic, q * s against x with the block's fp32 scale
    (the closest of the 255 levels), except within 1e-5 of a tie, where the
    fp32 quotient may round either way."""
    rng = np.random.default_rng(2)
    b = 16
    x = (rng.standard_normal(16 * 40) * np.exp2(rng.integers(-20, 5, 16 * 40))).astype(F32)
    q, s = C.quantize_blockwise(x, b)
    checked = 0
    for i, xv in enumerate(x):
        sv = Fraction(float(s[i // b]))
        ratio = Fraction(float(xv)) / sv
        frac = ratio - (ratio.numerator // ratio.denominator)
        if abs(frac - Fraction(1, 2)) < Fraction(1, 100000):
            continue
        best = min(range(-127, 128), key=lambda c: abs(Fraction(float(xv)) - c * sv))
        assert int(q[i]) == best, (i, float(xv), float(s[i // b]))
        checked += 1
    assert checked > 600


def test_zero_tiny_and_ragged_blocks():
    x = np.zeros(40, F32)
    x[32:] = [1e-44, -2e-45, 0, 0, 0, 0, 0, 0]  # max / 127 underflows to 0
    x[20] = 3.0
    q, s = C.quantize_blockwise(x, 16)
    assert s[0] == 0 and s[2] == 0 and s[1] == F32(F32(3.0) / F32(127))
    assert not q[:16].any() and not q[32:].any() and q[20] == 127
    # the last block is short: its scale is the largest of its own elements
    y = np.arange(1, 38, dtype=F32)  # blocks 0..15, 16..31, 32..36
    _, s = C.quantize_blockwise(y, 16)
    np.testing.assert_array_equal(s, (np.array([16, 32, 37], F32) / F32(127)).astype(F32))


def test_blocks_beat_one_scale_on_heavy_tails():
    """One scale for the whole tensor loses the small gradients (the page's
    reason for blocks); with blocks the mean error is several times lower."""
    x = _heavy(1 << 16, 7)
    per_tensor = np.abs(x - C.int8_compressor(x.size)(x)).mean()
    blockwise = np.abs(x - C.int8_compressor(128)(x)).mean()
    assert per_tensor / blockwise > 2


def _one_bit(threshold):
    return lambda x: np.where(x >= threshold, 1.0, 0.0)


def test_error_feedback_worked_example(golden):
    """Any 5 gradients below 0.5 that add to 1.6: the naive compressor sends 0,
    error feedback sends 2 and keeps -0.4 (the totals the page prints are
    forced: what is sent is a whole number and the residual stays in
    [-0.5, 0.5))."""
    rows = _rows(golden)
    K, thr = int(rows["ef_steps"]), float(rows["ef_threshold"])
    total = float(rows["ef_true_total"])
    c = _one_bit(thr)
    rng = np.random.default_rng(3)
    for _ in range(20):
        while True:
            w = rng.uniform(0.5, 1.0, K)
            g = w / w.sum() * total
            if g.max() < thr:
                break
        naive = sum(float(c(np.float64(gt))) for gt in g)
        e, sent = 0.0, 0.0
        for gt in g:
            v, e = C.error_feedback_step(np.float64(gt), np.float64(e), c)
            sent += float(v)
        assert naive == float(rows["ef_naive_sent"])
        assert sent == float(rows["ef_feedback_sent"])
        assert e == pytest.approx(float(rows["ef_residual"]), abs=1e-12)
        assert sent + e == pytest.approx(g.sum(), abs=1e-12)  # telescoping


def test_error_feedback_telescopes_with_int8():
    """Sum of transmitted = sum of gradients + e_1 - e_{K+1}, and the residual
    stays within half a block scale."""
    rng = np.random.default_rng(4)
    b, d, K = 64, 4096, 20
    comp = C.int8_compressor(b)
    e = np.zeros(d, F32)
    sent = np.zeros(d, np.float64)
    gsum = np.zeros(d, np.float64)
    for _ in range(K):
        g = (rng.standard_normal(d) * 1e-3).astype(F32)
        v, e_new = C.error_feedback_step(g, e, comp)
        q, s = C.quantize_blockwise((g + e).astype(F32), b)
        assert np.all(np.abs(e_new) <= np.repeat(s, b)[:d] * 0.5 * (1 + 2.0 ** -20) + 1e-12)
        e = e_new.astype(F32)
        sent += v
        gsum += g
    assert np.allclose(sent + e, gsum, rtol=0, atol=1e-8)


def test_compressed_allreduce_on_exact_values():
    """Grid values: compression is lossless, the residuals are zero and the
    result is the exact sum; in general it is within the compression error."""
    rng = np.random.default_rng(5)
    N, b, L = 6, 32, 32 * 9 + 5
    k = rng.integers(-127, 128, (N, L))
    k[:, ::b] = 127
    x = (k * 2.0 ** -10).astype(F32)
    out, e, _, _ = C.compressed_allreduce(x, np.zeros_like(x), b)
    np.testing.assert_array_equal(out, numerics.reference_sum_f64(x).astype(F32))
    assert not e.any()
    y = _heavy(N * L, 9).reshape(N, L)
    out, _, codes, scales = C.compressed_allreduce(y, None, b, scale=1.0)
    bound = sum(np.repeat(s.astype(np.float64), b)[:L] * 0.5 for s in scales)
    ref = numerics.reference_sum_f64(y)
    assert np.all(np.abs(out - ref) <= bound * (1 + 1e-5) + N * 2.0 ** -23 * numerics.abs_sum_f64(y))
    # one rank: the result is its own dequantized message
    one, _, q1, s1 = C.compressed_allreduce(y[:1], None, b)
    np.testing.assert_array_equal(one, C.dequantize(q1[0], s1[0], b))
