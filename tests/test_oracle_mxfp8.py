"""Pins of the MXFP8 quantisation oracle ("vLLM PR #65508", the epilogue's
arithmetic): the bit formula of the E8M0 scale against its definition
ceil(log2(amax / 448)) + 127 in exact rational arithmetic, the worked edge
blocks of the description (zeros, subnormals, 446/448/450 around the largest
E4M3 value, the 1.75 mantissa boundary), and the no-saturation property of
the scaled blocks."""

from fractions import Fraction

import numpy as np

from oracle.formats import E4M3_VALUES
from oracle.mxfp8 import MX_BLOCK, bf16_values, block_scale, mxfp8_quantize


def _exact(bits: int) -> Fraction:
    """Exact value of a finite bf16 bit pattern, from its fields."""
    e, m = (bits >> 7) & 0xFF, bits & 0x7F
    mag = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -mag if bits & 0x8000 else mag


def _scale_by_definition(block) -> int:
    """ceil(log2(amax / 448)) + 127, clamped to [0, 254]: the smallest k with
    amax <= 448 * 2^k, found by exact comparisons."""
    amax = max(abs(_exact(int(b))) for b in block)
    if amax == 0:
        return 0
    k = -300
    while amax > 448 * Fraction(2) ** k:
        k += 1
    return max(0, min(254, k + 127))


def _finite_bits(rng, n):
    b = rng.integers(0, 1 << 16, size=n, dtype=np.uint32).astype(np.uint16)
    exp = (b >> 7) & 0xFF
    return np.where(exp == 0xFF, b & np.uint16(0x807F), b).astype(np.uint16)  # no inf / NaN


def test_scale_formula_equals_its_definition_on_random_and_edge_blocks():
    rng = np.random.default_rng(7)
    blocks = [_finite_bits(rng, MX_BLOCK) for _ in range(2000)]
    # narrow dynamic ranges too: blocks whose exponents sit close together
    for _ in range(1000):
        e = int(rng.integers(1, 254))
        b = ((rng.integers(max(1, e - 3), min(254, e + 1) + 1, size=MX_BLOCK) << 7)
             | rng.integers(0, 128, size=MX_BLOCK) | (rng.integers(0, 2, size=MX_BLOCK) << 15))
        blocks.append(b.astype(np.uint16))
    edges = [0x0000, 0x8000, 0x0001, 0x007F, 0x0080, 0x43DF, 0x43E0, 0x43E1, 0x3FE0, 0x3FE1, 0x7F7F, 0x0400, 0x04E1]
    for v in edges:
        blocks.append(np.full(MX_BLOCK, v, dtype=np.uint16))
        blk = np.zeros(MX_BLOCK, dtype=np.uint16)
        blk[5] = v
        blocks.append(blk)
    for blk in blocks:
        assert block_scale(blk) == _scale_by_definition(blk), [hex(int(x)) for x in blk[:4]]


def test_worked_edge_blocks():
    def one(v, fill=0x0000):
        blk = np.full((1, MX_BLOCK), fill, dtype=np.uint16)
        blk[0, 0] = v
        return mxfp8_quantize(blk)

    q, s = one(0x0000)  # all zeros: scale 0, every byte +0
    assert s[0, 0] == 0 and (q == 0).all()
    q, s = one(0x8000)  # -0 keeps its sign
    assert s[0, 0] == 0 and q[0, 0] == 0x80
    q, s = one(0x43E0)  # 448 = 1.75 * 2^8: exponent 135, mantissa exactly 0.75 -> scale 127, 448 -> 0x7E
    assert s[0, 0] == 127 and q[0, 0] == 0x7E
    q, s = one(0x43E1)  # 450: mantissa 97/128 > 0.75 -> scale 128; 225 rounds to 224 = 0x76
    assert s[0, 0] == 128 and q[0, 0] == 0x76
    q, s = one(0x43DF)  # 446: scale 127; nearest E4M3 is 448
    assert s[0, 0] == 127 and q[0, 0] == 0x7E
    q, s = one(0xC3E1)  # -450: the sign passes through
    assert s[0, 0] == 128 and q[0, 0] == 0xF6
    q, s = one(0x0001)  # smallest subnormal, 2^-133: scale clamps to 0, 2^-133 * 2^127 = 2^-6 -> 0x08
    assert s[0, 0] == 0 and q[0, 0] == 0x08
    q, s = one(0x3F80, fill=0x3F00)  # amax 1.0 (exponent 127): scale 119, 1.0 * 2^8 = 256 -> 0x78; 0.5 -> 128 -> 0x70
    assert s[0, 0] == 119 and q[0, 0] == 0x78 and (q[0, 1:] == 0x70).all()


def test_scaled_blocks_stay_within_e4m3_range_and_round_to_nearest():
    rng = np.random.default_rng(8)
    bits = _finite_bits(rng, 64 * MX_BLOCK).reshape(64, MX_BLOCK)
    q, s = mxfp8_quantize(bits)
    x = bf16_values(bits)
    for r in range(64):
        scaled = x[r] * 2.0 ** (127 - int(s[r, 0]))
        assert np.abs(scaled).max() <= 448.0  # no block needs saturation
        back = E4M3_VALUES[q[r]]
        # round to nearest: no finite E4M3 value is closer than the chosen one
        finite = E4M3_VALUES[np.isfinite(E4M3_VALUES)]
        best = np.abs(finite[None, :] - scaled[:, None]).min(axis=1)
        assert np.array_equal(np.abs(back - scaled), best)


def test_rows_are_blocks_in_order():
    rng = np.random.default_rng(9)
    bits = _finite_bits(rng, 3 * 4 * MX_BLOCK).reshape(3, 4 * MX_BLOCK)
    q, s = mxfp8_quantize(bits)
    assert q.shape == bits.shape and s.shape == (3, 4)
    for r in range(3):
        for k in range(4):
            qb, sb = mxfp8_quantize(bits[r:r + 1, k * MX_BLOCK:(k + 1) * MX_BLOCK])
            assert sb[0, 0] == s[r, k] and np.array_equal(qb[0], q[r, k * MX_BLOCK:(k + 1) * MX_BLOCK])
