"""E4M3 and E2M1 number formats, from their definitions (test infrastructure).

E4M3 ("float8_e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits, no infinities; exponent field 15 with mantissa 7 is NaN, so the largest
finite magnitude is 1.75 * 2^8 = 448.  Exponent field 0 holds subnormals
m * 2^-9.

E2M1 (the NVFP4 element code): 1 sign bit (bit 3), 2 exponent bits with bias
1, 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.

The page "vllm.models.minimax_m3.nvidia.ops.gather_nvfp4_index_k" (module
docstring) fixes the dequantisation rule as e4m3_rn_satfinite(e2m1 * scale):
the exact product, rounded once to the nearest E4M3 value with ties to the
even mantissa, saturating finite overflow to +-448.  ``e4m3_encode`` below is
that rounding written as "nearest member of the finite E4M3 set".
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(b: int) -> float:
    """Value of one E4M3 byte, from the bit fields."""
    sign = -1.0 if (b >> 7) & 1 else 1.0
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# value of every byte; NaN for 0x7F and 0xFF
E4M3_VALUES = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)

# E2M1 code -> value: bit 3 is the sign, bits 0-2 index the magnitudes
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
E2M1_VALUES = np.array([(-1.0 if c & 8 else 1.0) * _E2M1_MAG[c & 7] for c in range(16)], dtype=np.float64)

# The non-negative finite E4M3 set, ascending, with its bytes 0x00..0x7E.
_POS_BYTES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = E4M3_VALUES[:0x7F].copy()
assert np.all(np.diff(_POS_VALUES) > 0)


def e4m3_encode(x) -> np.ndarray:
    """Round exact values to E4M3 bytes: nearest finite value, ties to even,
    saturate |x| > 448 to 448, keep the sign of zero, NaN -> 0x7F.

    Vectorised over a float64 array.  Every input that arises in this path
    (an E2M1 x E4M3 product, or a float32) is exact in float64, so the
    comparison of distances below is exact.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    nan = np.isnan(x)
    a = np.abs(np.where(nan, 0.0, x))
    neg = np.signbit(x) & ~nan
    i = np.searchsorted(_POS_VALUES, a, side="left")  # first value >= a
    i = np.clip(i, 1, len(_POS_VALUES) - 1)
    lo = _POS_VALUES[i - 1]
    hi = _POS_VALUES[i]
    d_lo = a - lo
    d_hi = hi - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_BYTES[i] & 1) == 0))
    mag = np.where(take_hi, _POS_BYTES[i], _POS_BYTES[i - 1]).astype(np.uint8)
    mag = np.where(a == 0.0, np.uint8(0), mag)
    mag = np.where(a >= E4M3_MAX, np.uint8(0x7E), mag)  # satfinite
    out = mag | np.where(neg, np.uint8(0x80), np.uint8(0)).astype(np.uint8)
    out = np.where(nan, np.uint8(0x7F), out).astype(np.uint8)
    return out


def e4m3_encode_rational(v: Fraction | float) -> int:
    """Second, independent E4M3 encoder: exact rational arithmetic.

    Picks the binade, scales by its quantum (2^(e-3), or 2^-9 below the
    normal range), rounds the quotient half-to-even (Python's ``round`` on a
    Fraction) and saturates.  Used only to pin ``e4m3_encode``.
    """
    if isinstance(v, float):
        if v != v:
            return 0x7F
        sign = 0x80 if math.copysign(1.0, v) < 0 else 0
        if math.isinf(v):
            return sign | 0x7E
    else:
        sign = 0x80 if v < 0 else 0
    a = abs(Fraction(v))
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -6)
    quantum = Fraction(2) ** (e - 3)
    r = round(a / quantum)  # half to even
    if r == 16:  # carried into the next binade
        e += 1
        r = 8
    if r == 0:
        return sign
    if e > 8 or (e == 8 and r > 14):
        return sign | 0x7E
    if r < 8:  # subnormal (only reachable at e == -6)
        return sign | r
    return sign | ((e + 7) << 3) | (r - 8)
