"""Numerics of the all-reduce: the definition of the sum, the declared summation
orders of the fused single pass, and bf16 widening/narrowing.

The problem (primer ch. 4 "Collective communication: algorithms, cost and the
library that runs them", §4.1, table of collectives): every rank starts with a
buffer of S bytes and every rank ends with the element-wise sum of all N
buffers. Scaling ML Systems ("Collective communication", section on the
collective API's numeric contract) adds that the order of the reduction is
part of the contract, because floating-point addition is not associative:
different algorithms may differ in their low bits.

So there is one exact definition (``reference_sum_f64``, used with an error
bound) and one bit-exact fp32 result per declared order (``fused_sum``).
"""

from __future__ import annotations

import numpy as np

from .chunks import chunk_bounds, chunk_of

# ----------------------------------------------------------------- bf16


def bf16_to_f32(bits) -> np.ndarray:
    """Widen bf16 bit patterns to fp32. bf16 is the upper half of an fp32 word,
    so widening appends 16 zero bits and is exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne(x) -> np.ndarray:
    """Round fp32 to bf16, round to nearest, ties to even, from the bit layout.

    bf16 keeps the sign, the 8 exponent bits and the top 7 mantissa bits of an
    fp32 word. The dropped low 16 bits decide the rounding: above half (0x8000)
    rounds up, below half rounds down, exactly half rounds to the neighbour
    whose last kept bit is 0. A carry out of the mantissa increments the
    exponent, which is the correct next bf16 value (up to +/-inf). Inputs must
    be finite.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("bf16 narrowing expects finite inputs")
    bits = x.view(np.uint32)
    low = bits & np.uint32(0xFFFF)
    high = bits >> np.uint32(16)
    half = np.uint32(0x8000)
    round_up = (low > half) | ((low == half) & ((high & np.uint32(1)) == 1))
    return (high + round_up.astype(np.uint32)).astype(np.uint16)


# ----------------------------------------------------------------- the sum


def reference_sum_f64(x) -> np.ndarray:
    """The definition: out[e] = sum over ranks r of g_r[e], accumulated in fp64."""
    x = np.asarray(x)
    acc = np.zeros(x.shape[1:], dtype=np.float64)
    for r in range(x.shape[0]):
        acc = acc + x[r].astype(np.float64)
    return acc


def abs_sum_f64(x) -> np.ndarray:
    """sum over ranks of |g_r[e]| in fp64 (the scale of the rounding-error bound)."""
    x = np.asarray(x)
    acc = np.zeros(x.shape[1:], dtype=np.float64)
    for r in range(x.shape[0]):
        acc = acc + np.abs(x[r].astype(np.float64))
    return acc


def _left_fold(x, ranks, cols=slice(None)):
    """((x[ranks[0]] + x[ranks[1]]) + x[ranks[2]]) + ... in fp32, on columns ``cols``."""
    acc = np.array(x[ranks[0], cols], dtype=np.float32, copy=True)
    for r in ranks[1:]:
        acc = acc + np.asarray(x[r, cols], dtype=np.float32)
    return acc


def _tree(values):
    """Pairwise sum of adjacent entries, level by level: (v0+v1), (v2+v3), ... then
    ((v0+v1)+(v2+v3)), ... The number of entries must be a power of two."""
    vals = list(values)
    while len(vals) > 1:
        vals = [vals[2 * m] + vals[2 * m + 1] for m in range(len(vals) // 2)]
    return vals[0]


def fused_sum(x, order: str, idx=None, L: int | None = None, group_size: int = 0,
              scale: float = 1.0) -> np.ndarray:
    """The fp32 sum of all ranks' elements in a declared order, times ``scale``.

    ``x`` is [N, K] fp32: the values of K elements of every rank, whose indices
    in the full buffer of L elements are ``idx`` (default: all of them).

    Orders (each is the per-element summation order of one schedule):

    * ``"ring"``: an element of chunk c is folded starting at rank c:
      ((g_c + g_{c+1}) + ...) + g_{c-1}, rank indices mod N. This is the order
      in which the ring's reduce-scatter carries chunk c around the ring (the
      primer, §4.2: rank i sends chunk (i - s) mod N at step s).
    * ``"ring_rs"``: an element of chunk c is folded starting at rank c+1:
      ((g_{c+1} + g_{c+2}) + ...) + g_c, the order of the standalone ring
      reduce-scatter in which rank c ends with chunk c.
    * ``"rank"``: ((g_0 + g_1) + ...) + g_{N-1} for every element.
    * ``"tree"``: a balanced binary tree over ranks in index order, the order
      of recursive halving with partners at distance 1 first (the primer,
      §4.3, Fig. 4.5 and Animation 4.2). N must be a power of two.
    * ``"hier"``: groups of G consecutive ranks. An element of slice k (the
      buffer cut into G slices) and sub-chunk j (slice k cut into M = N/G
      sub-chunks) is first folded inside every group starting at local rank
      k+1: ((g_{k+1} + g_{k+2}) + ...) + g_k, then the M group partials are
      folded starting at group j. This is the order of the three-phase
      hierarchical all-reduce (primer §4.4, Fig. 4.8 and Animation 4.3).

    The result is multiplied by ``scale`` once, in fp32.
    """
    x = np.asarray(x, dtype=np.float32)
    N, K = x.shape
    idx = np.arange(K) if idx is None else np.asarray(idx, dtype=np.int64)
    L = K if L is None else L
    out = np.empty(K, dtype=np.float32)
    if order == "rank":
        out[:] = _left_fold(x, list(range(N)))
    elif order in ("ring", "ring_rs"):
        c_of = chunk_of(idx, L, N)
        first = 0 if order == "ring" else 1
        for c in range(N):
            cols = np.nonzero(c_of == c)[0]
            if cols.size:
                out[cols] = _left_fold(x, [(c + first + i) % N for i in range(N)], cols)
    elif order == "tree":
        if N & (N - 1):
            raise ValueError("tree order needs a power-of-two rank count")
        out[:] = _tree([x[r] for r in range(N)])
    elif order == "hier":
        G = group_size
        if G < 1 or N % G:
            raise ValueError("hier order needs a group size that divides N")
        M = N // G
        s_of = chunk_of(idx, L, G)
        sb = chunk_bounds(L, G)
        for k in range(G):
            Lk = sb[k + 1] - sb[k]
            in_slice = np.nonzero(s_of == k)[0]
            if not in_slice.size:
                continue
            j_of = chunk_of(idx[in_slice] - sb[k], Lk, M)
            for j in range(M):
                cols = in_slice[j_of == j]
                if not cols.size:
                    continue
                partials = [
                    _left_fold(x, [g * G + (k + 1 + i) % G for i in range(G)], cols)
                    for g in range(M)
                ]
                acc = partials[j % M].copy()
                for i in range(1, M):
                    acc = acc + partials[(j + i) % M]
                out[cols] = acc
    else:
        raise ValueError(f"unknown order {order!r}")
    if scale != 1.0:
        out = out * np.float32(scale)
    return out
