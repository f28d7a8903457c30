"""CPU oracle for the gradient all-reduce: TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement of what the
all-reduce computes, written from the pages and checked against the values
and closed forms they print (``tests/test_oracle_*.py``). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it.
The GPU library (``gradient_sync_gb300``) never imports it and shares no code
with it; both take their inputs from ``workloads``.

Arithmetic: fp32 adds in numpy (one IEEE binary32 addition per element, no
fusion, no reassociation), fp64 for the reference sum, and bf16 rounding
written out from the bf16 bit layout.

Modules:

* ``chunks``    -- how a buffer of L elements is cut into N chunks.
* ``numerics``  -- bf16 widening/narrowing, the fp64 definition of the sum,
                   and the fused single-pass sums in each declared order.
* ``schedules`` -- step-by-step simulations of the ring, Rabenseifner,
                   hierarchical, recursive-doubling, double-binary-tree and
                   torus (dimension-ordered) all-reduce, and of the standalone
                   ring reduce-scatter and all-gather, with per-rank mailboxes
                   and byte/step counters.
* ``buckets``   -- DDP-style bucket assignment and the bucketed gradient sync.
* ``compress``  -- blockwise INT8 quantization, error feedback, and the
                   compressed all-reduce (every rank's message dequantized and
                   summed in rank order).

Parity pins: every function here is pinned by a test against a value the
pages print, a closed form or brute force, except the bucket packing order
inside one bucket, which the pages do not fix (parity unpinned beyond the
invariants listed in ``buckets``).
"""

from . import buckets, chunks, compress, numerics, schedules  # noqa: F401
from .chunks import chunk_bounds, chunk_of  # noqa: F401
from .numerics import (bf16_to_f32, f32_to_bf16_rne, fused_sum, reference_sum_f64,  # noqa: F401
                       abs_sum_f64)
from .schedules import (hierarchical_allreduce, rabenseifner_allreduce,  # noqa: F401
                        ring_allgather, ring_allreduce, ring_reduce_scatter, RunStats,
                        recursive_doubling_allreduce, double_binary_tree_allreduce, torus_allreduce)
