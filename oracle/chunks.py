"""How one rank's buffer is cut into N chunks.

The primer (ch. 4 "Collective communication: algorithms, cost and the library
that runs them", §4.2 "The ring, one step at a time") cuts each rank's buffer
into N chunks numbered 0..N-1 but does not say where the cuts fall when N does
not divide the element count. Reading taken here: chunk c covers elements
[floor(c*L/N), floor((c+1)*L/N)). Chunks then differ in length by at most one
element and are empty only when L < N.
"""

from __future__ import annotations

import numpy as np


def chunk_bounds(L: int, n: int) -> list[int]:
    """The n+1 cut points of a buffer of L elements cut into n chunks."""
    if n < 1:
        raise ValueError("n must be >= 1")
    return [(c * L) // n for c in range(n + 1)]


def chunk_range(L: int, n: int, c: int) -> tuple[int, int]:
    b = chunk_bounds(L, n)
    return b[c], b[c + 1]


def chunk_of(idx, L: int, n: int) -> np.ndarray:
    """For every element index in ``idx``, the chunk that contains it.

    Found by searching the cut points: the chunk is the last c whose start is
    <= the index (empty chunks are skipped automatically).
    """
    bounds = np.asarray(chunk_bounds(L, n), dtype=np.int64)
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= L):
        raise IndexError("element index outside the buffer")
    return np.searchsorted(bounds, idx, side="right") - 1
