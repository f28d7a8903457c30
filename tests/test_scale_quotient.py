"""The block scale max|x| / 127 without a division, checked with exact
rational arithmetic on the CPU: q0 = RN(m * c) with c = RN(1/127), the
remainder m - q0 * 127 (one FMA), and q0 + remainder * c (one FMA) must be
the correctly rounded quotient RN(m / 127). This is the method the kernels
use (its exhaustive comparison with the IEEE division over every float runs
on the GPU); here each operation is rounded exactly from its rational value."""

from fractions import Fraction

import numpy as np
import pytest


def rn32(q: Fraction) -> Fraction:
    """Round a rational to the nearest fp32 value, ties to even (finite range,
    subnormals included)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)  # below the normal range the spacing stays 2^-149
    scale = Fraction(2) ** (23 - e)
    n = a * scale
    f = n.numerator // n.denominator
    rem = n - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return sign * Fraction(f) / scale


def f32(q: Fraction) -> float:
    return float(np.float32(float(q)))


C = rn32(Fraction(1, 127))


def div127(m: Fraction) -> Fraction:
    q0 = rn32(m * C)
    rem = rn32(m - q0 * 127)
    assert rem == m - q0 * 127, "the remainder is exact"
    return rn32(rem * C + q0)


def test_reciprocal_constant():
    assert f32(C) == float.fromhex("0x1.020408p-7")
    assert abs(C - Fraction(1, 127)) <= Fraction(1, 2) * Fraction(2) ** -30  # half an ulp at 2^-7


def _cases():
    rng = np.random.default_rng(5)
    bits = [0, 1, 2, 3, 0x007FFFFF, 0x00800000, 0x00800001, 0x3F800000, 0x42FE0000, 0x7F7FFFFF, 0x7F7FFFFE,
            0x3C010204, 0x3C010205, 0x0B7E0000, 0x00FE0000, 0x01000000]
    bits += rng.integers(0, 0x7F800000, 3000).tolist()
    bits += rng.integers(0, 0x02000000, 1000).tolist()  # subnormal and lowest normal quotients
    # m = k * 127 * 2^e and its neighbours: exact quotients and near-ties
    for k in rng.integers(1 << 23, 1 << 24, 300).tolist():
        for e in (-150, -140, -100, -10, 0, 30, 90):
            m = np.float32(float(Fraction(k * 127) * Fraction(2) ** e))
            if np.isfinite(m):
                u = int(np.array(m, np.float32).view(np.uint32))
                bits += [u - 1, u, u + 1]
    return sorted({b for b in bits if 0 <= b < 0x7F800000})


def test_division_free_quotient_is_correctly_rounded():
    bad = []
    for u in _cases():
        m = Fraction(float(np.array(u, np.uint32).view(np.float32)))
        if div127(m) != rn32(m / 127):
            bad.append(hex(u))
    assert not bad, f"{len(bad)} mismatches, first {bad[:5]}"
