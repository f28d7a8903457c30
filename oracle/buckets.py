"""DDP-style bucketed gradient sync.

Scaling ML Systems ("Collective communication", section "Bucket fusion"):
parameter gradients are grouped into buckets of a capped size (25 MB is the
usual PyTorch default, set by ``bucket_cap_mb``), parameters are assigned to
buckets in the reverse of their forward order (the order in which backward
produces their gradients), and one all-reduce is issued per bucket.

Readings taken where the pages are silent:

* The cap counts the bytes of the gradients as stored (bf16: 2 bytes each).
* A bucket is closed when adding the next tensor would take it over the cap;
  a tensor larger than the cap gets a bucket of its own; tensors are never
  split.
* Inside a bucket, tensors are packed in the order they were added (reverse
  forward order). This packing order is not fixed by the pages: parity
  unpinned beyond the invariants (every tensor in exactly one bucket, bucket
  sizes sum to the parameter count, buckets follow reverse forward order).
* Each bucket is widened to fp32, ring all-reduced in fp32, multiplied by 1/N
  and rounded once to bf16.
"""

from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f32, f32_to_bf16_rne
from .schedules import ring_allreduce


def bucket_plan(counts, elem_bytes: int, cap_bytes: int) -> list[list[int]]:
    """Assign tensors (given in forward order) to buckets, filled in reverse order.

    Returns the buckets in the order they fill (the first is the last layer's);
    each bucket lists its tensor indices in packing order.
    """
    buckets, cur, cur_bytes = [], [], 0
    for t in reversed(range(len(counts))):
        nbytes = int(counts[t]) * elem_bytes
        if cur and cur_bytes + nbytes > cap_bytes:
            buckets.append(cur)
            cur, cur_bytes = [], 0
        cur.append(t)
        cur_bytes += nbytes
    if cur:
        buckets.append(cur)
    return buckets


def bucket_offsets(bucket, counts) -> dict:
    """Packed offset of every tensor of a bucket (tensors laid end to end in bucket order)."""
    off, out = 0, {}
    for t in bucket:
        out[t] = off
        off += int(counts[t])
    return out


def sync_bucket(grads, bucket, counts, scale: float, windows=None):
    """All-reduce one bucket of bf16 gradients: pack (widen to fp32), ring
    all-reduce in fp32, unpack (multiply by ``scale`` in fp32, round to bf16).

    ``grads[r][t]`` is rank r's gradient of tensor t as bf16 bits. With
    ``windows`` = list of (t, lo, hi), only those elements are computed and
    ``grads[r][t]`` holds just elements [lo, hi) of tensor t for those
    windows (keyed by (t, lo)). Returns {(t, lo): [N, hi-lo] bf16 bits}.
    """
    N = len(grads)
    offs = bucket_offsets(bucket, counts)
    Lb = sum(int(counts[t]) for t in bucket)
    if windows is None:
        windows = [(t, 0, int(counts[t])) for t in bucket]
        get = lambda r, t, lo, hi: grads[r][t]  # noqa: E731
    else:
        get = lambda r, t, lo, hi: grads[r][(t, lo)]  # noqa: E731
    idx = np.concatenate([np.arange(offs[t] + lo, offs[t] + hi, dtype=np.int64)
                          for t, lo, hi in windows])
    packed = np.stack([
        np.concatenate([bf16_to_f32(get(r, t, lo, hi)) for t, lo, hi in windows]) for r in range(N)
    ])
    reduced, _ = ring_allreduce(packed, idx=idx, L=Lb)
    out_bits = np.stack([f32_to_bf16_rne(reduced[r] * np.float32(scale)) for r in range(N)])
    res, pos = {}, 0
    for t, lo, hi in windows:
        res[(t, lo)] = out_bits[:, pos:pos + hi - lo]
        pos += hi - lo
    return res
