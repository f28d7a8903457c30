"""Seeded synthetic inputs for the gradient all-reduce.

This module is the one place that both the CPU oracle (``oracle/``) and the
GPU path (``gradient_sync_gb300``) take their inputs from. It holds no
arithmetic of the all-reduce itself: it only draws random numbers and rounds
them to the storage type of a rank's gradient buffer.

Recipe (the same for every workload):

* A rank buffer is cut into blocks of ``BLOCK`` elements. Block ``b`` of the
  buffer with key ``key`` (``(rank,)`` for a flat buffer, ``(rank, tensor)``
  for one parameter's gradient) is drawn from its own PCG64 stream,
  ``numpy.random.default_rng(SeedSequence(seed, spawn_key=key + (b,)))``.
  Blocks are therefore independent and can be drawn in any order, in
  parallel, or one window at a time.
* ``"int"``: ``integers(-8, 9)`` (both ends included), stored as fp32. Sums of
  up to 2^20 such values are exact in fp32.
* ``"normal"``: ``standard_normal() * std`` in fp64, rounded to fp32
  (round to nearest even); for bf16 buffers the fp32 value is then rounded to
  bf16 by ``torch`` (round to nearest even).
* ``"uniform"``: ``uniform(-1, 1)`` in fp64, rounded to fp32.

bf16 buffers are held on the host as ``numpy.uint16`` bit patterns.

The workloads are the ones the pages use: a 192 MiB fp32 gradient (the
[12288, 4096] FFN gate projection) on 16 ranks (AI Infra Book ch. 7, "Data-center
networks", §7.2.1), and DDP buckets of about 25 MB over a transformer's
parameter gradients (Scaling ML Systems, "Collective communication",
section "Bucket fusion").
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK = 1 << 20  # elements per independently seeded block

MiB = 1 << 20
KiB = 1 << 10
GiB = 1 << 30


@dataclass(frozen=True)
class Spec:
    """A flat all-reduce workload: ``n_ranks`` buffers of ``count`` elements."""

    name: str
    n_ranks: int
    count: int
    dtype: str  # "f32" or "bf16"
    dist: str  # "int", "normal" or "uniform"
    std: float = 1e-3
    seed: int = 0
    group_size: int = 0  # hierarchical: ranks per group (0 = flat)
    extra: dict = field(default_factory=dict)

    @property
    def itemsize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def bytes_per_rank(self) -> int:
        return self.count * self.itemsize


# The named workloads, with the sizes the pages' examples use.
RING_N4_INT = Spec("ring all-reduce, 4 ranks x 1,048,576 fp32 integers in [-8, 8]",
                   n_ranks=4, count=1_048_576, dtype="f32", dist="int")
RING_N16_192MIB = Spec("ring all-reduce, 16 ranks x 192 MiB fp32 (50,331,648 values), N(0, 1e-3^2)",
                       n_ranks=16, count=50_331_648, dtype="f32", dist="normal", std=1e-3)
HIER_2X8_BF16 = Spec("hierarchical all-reduce, 16 ranks as 2 groups of 8, 96 Mi bf16 values per rank, N(0, 1e-3^2)",
                     n_ranks=16, count=100_663_296, dtype="bf16", dist="normal", std=1e-3, group_size=8)

SWEEP_RANKS = (2, 4, 8, 16, 64)
SWEEP_BYTES = tuple(KiB * 4 ** k for k in range(11))  # 1 KiB .. 1 GiB in powers of 4
SWEEP_TOTAL_CAP = 64 * GiB


def sweep_specs():
    """The size/algorithm sweep: every (N, S) pair with N*S <= 64 GiB, fp32 uniform [-1, 1]."""
    out = []
    for n in SWEEP_RANKS:
        for s in SWEEP_BYTES:
            if n * s <= SWEEP_TOTAL_CAP:
                out.append(Spec(f"sweep N={n} S={s} B", n_ranks=n, count=s // 4,
                                dtype="f32", dist="uniform"))
    return out


# ---------------------------------------------------------------- transformer

TRANSFORMER = dict(layers=16, hidden=2048, ffn=8192, vocab=32000)


def transformer_tensors(layers=16, hidden=2048, ffn=8192, vocab=32000):
    """Parameter gradients of the 16-layer transformer, in forward (registration) order.

    Returns a list of (name, element count). Per layer: norm1, Wq, Wk, Wv, Wo
    (hidden x hidden), norm2, W1, W3 (hidden x ffn) and W2 (ffn x hidden); the
    token embedding (vocab x hidden) comes first. No untied output head.
    """
    out = [("embedding", vocab * hidden)]
    for layer in range(layers):
        out += [
            (f"layers.{layer}.norm1", hidden),
            (f"layers.{layer}.wq", hidden * hidden),
            (f"layers.{layer}.wk", hidden * hidden),
            (f"layers.{layer}.wv", hidden * hidden),
            (f"layers.{layer}.wo", hidden * hidden),
            (f"layers.{layer}.norm2", hidden),
            (f"layers.{layer}.w1", hidden * ffn),
            (f"layers.{layer}.w3", hidden * ffn),
            (f"layers.{layer}.w2", ffn * hidden),
        ]
    return out


BUCKET_CAP_BYTES = 25 * MiB
BUCKETED_N8 = Spec("bucketed gradient sync, 8 ranks, 16-layer transformer (hidden 2048, FFN 8192, "
                   "vocab 32000) bf16 gradients N(0, 1e-3^2), 25 MiB buckets",
                   n_ranks=8, count=sum(c for _, c in transformer_tensors()), dtype="bf16",
                   dist="normal", std=1e-3, extra={"cap_bytes": BUCKET_CAP_BYTES})


# ---------------------------------------------------------------- generation

def _rng(seed: int, key: tuple, block: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=tuple(key) + (block,)))


def _draw_f32(dist: str, rng: np.random.Generator, n: int, std: float) -> np.ndarray:
    if dist == "int":
        return rng.integers(-8, 9, size=n).astype(np.float32)
    if dist == "normal":
        return (rng.standard_normal(n) * std).astype(np.float32)
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, n).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def f32_to_bf16_bits_torch(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 with torch's own conversion; returns uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def default_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def window(dist: str, dtype: str, seed: int, key: tuple, lo: int, hi: int, std: float = 1e-3,
           threads: int | None = None) -> np.ndarray:
    """Elements [lo, hi) of the buffer with ``key``; only the blocks that cover them are drawn."""
    if hi <= lo:
        return np.zeros(0, np.float32 if dtype == "f32" else np.uint16)
    b0, b1 = lo // BLOCK, (hi - 1) // BLOCK

    def one(b):
        return _draw_f32(dist, _rng(seed, key, b), BLOCK, std)

    blocks = list(range(b0, b1 + 1))
    nthreads = threads or default_threads()
    if len(blocks) == 1 or nthreads == 1:
        parts = [one(b) for b in blocks]
    else:
        with ThreadPoolExecutor(min(nthreads, len(blocks))) as ex:
            parts = list(ex.map(one, blocks))
    flat = parts[0] if len(parts) == 1 else np.concatenate(parts)
    out = flat[lo - b0 * BLOCK: hi - b0 * BLOCK]
    if dtype == "bf16":
        return f32_to_bf16_bits_torch(out)
    return np.ascontiguousarray(out)


def rank_buffer(spec: Spec, rank: int, lo: int = 0, hi: int | None = None, threads=None) -> np.ndarray:
    """Rank ``rank``'s buffer of a flat workload (or elements [lo, hi) of it)."""
    hi = spec.count if hi is None else hi
    return window(spec.dist, spec.dtype, spec.seed, (rank,), lo, hi, spec.std, threads)


def all_ranks(spec: Spec, threads=None) -> np.ndarray:
    """All ranks' buffers as one [n_ranks, count] array (small workloads only)."""
    return np.stack([rank_buffer(spec, r, threads=threads) for r in range(spec.n_ranks)])


def tensor_grad(spec: Spec, rank: int, tensor: int, count: int, lo: int = 0, hi: int | None = None,
                threads=None) -> np.ndarray:
    """Rank ``rank``'s gradient of parameter ``tensor`` (forward order index)."""
    hi = count if hi is None else hi
    return window(spec.dist, spec.dtype, spec.seed, (rank, tensor), lo, hi, spec.std, threads)


RESIDUAL_KEY = 1 << 24  # second key component of the residual streams (distinct from tensor ids)


def residual_buffer(spec: Spec, rank: int, lo: int = 0, hi: int | None = None, threads=None) -> np.ndarray:
    """An fp32 error-feedback residual for rank ``rank`` of a flat workload (or
    elements [lo, hi) of it): normal with 1/100 of the gradients' std, the
    size of a residual left by a block of a few std (half a scale is about
    2 std / 127)."""
    hi = spec.count if hi is None else hi
    return window("normal", "f32", spec.seed, (rank, RESIDUAL_KEY), lo, hi, spec.std * 1e-2, threads)


def small_spec(n_ranks: int, count: int, dtype: str = "f32", dist: str = "uniform", seed: int = 0,
               group_size: int = 0, std: float = 1e-3) -> Spec:
    """An ad-hoc workload for tests (ragged sizes, tiny N, edge cases)."""
    return Spec(f"test N={n_ranks} L={count} {dtype} {dist}", n_ranks=n_ranks, count=count,
                dtype=dtype, dist=dist, seed=seed, group_size=group_size, std=std)
