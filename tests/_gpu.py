"""Helpers for the GPU tests: move seeded inputs to the device and results back,
and compute the oracle's expected values (full or on sampled windows)."""

from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import numerics, schedules


def to_device(arr: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def widened(x: np.ndarray, dtype: str) -> np.ndarray:
    """The fp32 values of the inputs (bf16 widened exactly)."""
    return numerics.bf16_to_f32(x) if dtype == "bf16" else np.asarray(x, np.float32)


def expected(algo: str, order: str, x: np.ndarray, dtype: str, group_size: int = 0, scale: float = 1.0,
             idx=None, L=None, torus_dims=None) -> np.ndarray:
    """The oracle's result for one rank (all ranks are identical), as stored
    (fp32 values or bf16 bits)."""
    xf = widened(x, dtype)
    if algo == "fused":
        s = numerics.fused_sum(xf, order, idx=idx, L=L, group_size=group_size, scale=scale)
        return numerics.f32_to_bf16_rne(s) if dtype == "bf16" else s
    finish = schedules.finish_bf16(scale) if dtype == "bf16" else schedules.finish_scale(scale)
    if algo == "ring":
        out, _ = schedules.ring_allreduce(xf, idx=idx, L=L, finish=finish)
    elif algo == "rabenseifner":
        out, _ = schedules.rabenseifner_allreduce(xf, idx=idx, L=L, finish=finish)
    elif algo == "hier":
        out, _ = schedules.hierarchical_allreduce(xf, group_size, idx=idx, L=L, finish=finish)
    elif algo == "recdoubling":
        out, _ = schedules.recursive_doubling_allreduce(xf, idx=idx, L=L, finish=finish)
    elif algo == "dbtree":
        out, _ = schedules.double_binary_tree_allreduce(xf, idx=idx, L=L, finish=finish)
    elif algo == "torus":
        out, _ = schedules.torus_allreduce(xf, torus_dims, idx=idx, L=L, finish=finish)
    else:
        raise ValueError(algo)
    for r in range(1, out.shape[0]):
        assert np.array_equal(out[r].view(np.uint32), out[0].view(np.uint32))
    return numerics.f32_to_bf16_rne(out[0]) if dtype == "bf16" else out[0]


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    g = got.view(np.uint16 if got.dtype == np.uint16 else np.uint32)
    w = want.view(np.uint16 if want.dtype == np.uint16 else np.uint32)
    if not np.array_equal(g, w):
        bad = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {bad.size} of {g.size} elements differ; first at {bad[:8].tolist()}: "
                             f"got {got[bad[:4]]} want {want[bad[:4]]}")


def sample_windows(L: int, n_chunks: int, window: int = 1024, n_random: int = 64, seed: int = 0):
    """Sorted unique element indices: the first and last `window` elements of
    every chunk plus `n_random` random windows."""
    from oracle.chunks import chunk_bounds

    b = chunk_bounds(L, n_chunks)
    parts = []
    for c in range(n_chunks):
        lo, hi = b[c], b[c + 1]
        parts.append(np.arange(lo, min(hi, lo + window)))
        parts.append(np.arange(max(lo, hi - window), hi))
    rng = np.random.default_rng(seed)
    for s in rng.integers(0, max(1, L - window), n_random):
        parts.append(np.arange(s, min(L, s + window)))
    return np.unique(np.concatenate(parts).astype(np.int64))


def device_inputs(spec: workloads.Spec, idx=None):
    """Every rank's full buffer on the device, plus the sampled values at idx
    ([N, len(idx)], or the full host array when idx is None)."""
    devs, sampled = [], []
    for r in range(spec.n_ranks):
        host = workloads.rank_buffer(spec, r)
        devs.append(to_device(host, spec.dtype))
        sampled.append(host if idx is None else host[idx])
        del host
    return devs, np.stack(sampled)
