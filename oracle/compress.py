"""Blockwise INT8 gradient compression with error feedback, and the compressed
all-reduce built on it.

Scaling ML Systems, "Collective communication", the section on gradient
compression when bandwidth is scarce:

* "Quantization: reducing precision", INT8: a scale s = max|g| / 127 and codes
  round(g / s); the receiver reconstructs codes * s.
* "Blockwise quantization for gradient communication": the tensor is cut into
  blocks of b elements (typically 64 or 128), each with its own scale; the
  message is d bytes of codes plus 4 bytes of fp32 scale per block, a
  compression of 4b / (b + 4) against fp32 (3.88 at b = 128); the largest
  error of an element is half its block's scale.
* "Error feedback and residual accumulation": each worker keeps a residual
  e_t; it compresses x = g_t + e_t, transmits v_t = C(x) and keeps
  e_{t+1} = x - v_t, so that the sum of what it transmits telescopes to the
  sum of its gradients minus the last residual.

Readings where the page leaves a step open (each is a test below):

* Arithmetic is fp32, in the page's order: the scale is the fp32 quotient
  max|x| / 127, each code the fp32 quotient x / s rounded to the nearest
  integer with ties to even, clamped to [-127, 127]; dequantization is the fp32
  product code * s. The last block of a tensor may be shorter than b.
* A block whose scale is 0 (all zeros, or a maximum so small that max / 127
  underflows) gets codes 0.
* The compressed all-reduce: every rank compresses its own x_r = g_r + e_r
  once, and the reducer sums the N dequantized messages in fp32 in rank order,
  ((d_0 + d_1) + ...) + d_{N-1}, scales once and rounds once to the output
  type. No partial sum is requantised (the page's "interfaces that fuse
  quantization and reduction").

Plain numpy, one element at a time where it matters; test infrastructure
only (see the package docstring).
"""

from __future__ import annotations

import numpy as np

from .numerics import f32_to_bf16_rne

F32 = np.float32


def n_blocks(count: int, block: int) -> int:
    return (count + block - 1) // block


def message_bytes(count: int, block: int) -> int:
    """Bytes of one compressed message: a 1-byte code per element plus an fp32
    scale per block."""
    return count + 4 * n_blocks(count, block)


def compression_ratio(block: int) -> float:
    """fp32 bytes over message bytes for a length that is a multiple of b:
    4d / (d + 4d/b) = 4b / (b + 4)."""
    return 4 * block / (block + 4)


def quantize_blockwise(x: np.ndarray, block: int):
    """Codes (int8, one per element) and scales (fp32, one per block) of x."""
    x = np.asarray(x, F32)
    nb = n_blocks(x.size, block)
    codes = np.zeros(x.size, np.int8)
    scales = np.zeros(nb, F32)
    for k in range(nb):
        xb = x[k * block:(k + 1) * block]
        m = np.max(np.abs(xb)) if xb.size else F32(0)
        s = F32(F32(m) / F32(127))
        scales[k] = s
        if s == 0:
            continue  # codes stay 0
        q = np.rint((xb / s).astype(F32))
        codes[k * block:(k + 1) * block] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, block: int) -> np.ndarray:
    """code * scale of its block, as fp32 products."""
    s = np.repeat(np.asarray(scales, F32), block)[: codes.size]
    return (codes.astype(F32) * s).astype(F32)


def error_feedback_step(g, e, compress):
    """One step of error feedback: x = g + e is compressed to the transmitted
    v = compress(x); the new residual is x - v. Returns (v, e_new)."""
    x = g + e
    v = compress(x)
    return v, x - v


def int8_compressor(block: int):
    """The blockwise INT8 compressor as a function x -> transmitted values
    (fp32 in, fp32 out)."""

    def c(x):
        q, s = quantize_blockwise(x, block)
        return dequantize(q, s, block)

    return c


def compress_rank(g: np.ndarray, e: np.ndarray | None, block: int):
    """What one rank sends: codes and scales of x = g + e (fp32), and its new
    residual x - dequantized (None without error feedback)."""
    x = np.asarray(g, F32) if e is None else (np.asarray(g, F32) + np.asarray(e, F32)).astype(F32)
    q, s = quantize_blockwise(x, block)
    e_new = None if e is None else (x - dequantize(q, s, block)).astype(F32)
    return q, s, e_new


def dequant_allreduce(codes, scales, block: int, scale: float = 1.0, out_dtype: str = "f32"):
    """The reducer: sum of the N ranks' dequantized messages in rank order,
    times `scale` once, rounded once to the output type (bf16 as bits)."""
    N = len(codes)
    acc = dequantize(codes[0], scales[0], block)
    for r in range(1, N):
        acc = (acc + dequantize(codes[r], scales[r], block)).astype(F32)
    if scale != 1.0:
        acc = (acc * F32(scale)).astype(F32)
    return f32_to_bf16_rne(acc) if out_dtype == "bf16" else acc


def compressed_allreduce(grads, errors, block: int, scale: float = 1.0, out_dtype: str = "f32"):
    """Every rank compresses g_r + e_r, all messages are summed in rank order.
    grads: [N, L] fp32 values (bf16 inputs widened by the caller); errors:
    [N, L] fp32 residuals or None. Returns (result, new residuals or None,
    codes, scales)."""
    codes, scales, new_e = [], [], []
    for r in range(len(grads)):
        q, s, e = compress_rank(grads[r], None if errors is None else errors[r], block)
        codes.append(q)
        scales.append(s)
        new_e.append(e)
    out = dequant_allreduce(codes, scales, block, scale, out_dtype)
    return out, (None if errors is None else np.stack(new_e)), codes, scales
