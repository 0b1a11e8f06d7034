"""MXFP8 (E4M3 values, E8M0 block scales) quantisation of bf16 rows (test infrastructure).

Written from "vLLM PR #65508" (the ROCm MXFP8 epilogue on the sparse-decode
attention output), its description of the epilogue's arithmetic:

* one MX block is 32 consecutive elements of a row;
* the block's amax is taken on the bf16 values' integer bit patterns (the
  magnitude bits, sign cleared: for finite values the integer order is the
  magnitude order);
* the block's E8M0 scale byte is clamp(exponent_field - 8 + (mantissa > 0.75),
  0, 254), exponent_field and mantissa (as a fraction in [0, 1)) being those
  of the amax; the page states that this equals ceil(log2(amax / 448)) + 127,
  448 = 1.75 * 2^8 being the largest E4M3 value;
* every element is multiplied by the exact power of two 2^(127 - scale) and
  converted to E4M3 with round-to-nearest-even;
* scales are stored row-major, one byte per block.

The conversion here is the saturating E4M3 encoder of ``oracle.formats``
(finite values of a block scaled this way never exceed 448, so saturation
only matters for non-finite inputs: an infinity becomes +-448, a NaN 0x7F).
"""

from __future__ import annotations

import numpy as np

from .formats import e4m3_encode

MX_BLOCK = 32


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (bf16 is the top half of float32)."""
    b32 = (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).astype(np.uint32)
    return b32.view(np.float32).astype(np.float64)


def block_scale(block_bits: np.ndarray) -> int:
    """E8M0 scale byte of one 32-element block of bf16 bit patterns."""
    amax = int((np.asarray(block_bits, dtype=np.uint16) & np.uint16(0x7FFF)).max())
    exponent_field = (amax >> 7) & 0xFF
    mantissa_above = (amax & 0x7F) > 96  # mantissa fraction m / 128 > 0.75
    return max(0, min(254, exponent_field - 8 + (1 if mantissa_above else 0)))


def mxfp8_quantize(bits: np.ndarray):
    """bf16 rows [rows, cols] (uint16 bit patterns, cols a multiple of 32) ->
    (E4M3 bytes [rows, cols], E8M0 scale bytes [rows, cols / 32])."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % MX_BLOCK:
        raise ValueError("columns must be a multiple of 32")
    nb = cols // MX_BLOCK
    scales = np.zeros((rows, nb), dtype=np.uint8)
    out = np.zeros((rows, cols), dtype=np.uint8)
    x = bf16_values(bits)
    for r in range(rows):
        for k in range(nb):
            sl = slice(k * MX_BLOCK, (k + 1) * MX_BLOCK)
            sb = block_scale(bits[r, sl])
            scales[r, k] = sb
            out[r, sl] = e4m3_encode(x[r, sl] * 2.0 ** (127 - sb))
    return out, scales
