"""Pins for the oracle's number formats and NVFP4 dequantisation.

Checked against things other than the oracle itself: torch's float8_e4m3fn
decode and cast, the E2M1 bit-field definition, a second rational encoder,
worked values, and a hand-built page (tests/golden/nvfp4_page_layout.txt).
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle.formats import E2M1_VALUES, E4M3_VALUES, e4m3_encode, e4m3_encode_rational
from oracle.indexer import dequant_page, gather_dequant, page_fields, ST_BLOCK_OOR, ST_BAD_OUTPUT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_values_match_torch_decode():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(E4M3_VALUES))
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(ref[~nan], E4M3_VALUES[~nan])
    # signed zeros
    assert math.copysign(1.0, E4M3_VALUES[0x80]) < 0 and math.copysign(1.0, E4M3_VALUES[0]) > 0
    assert E4M3_VALUES[0x7E] == 448.0 and E4M3_VALUES[0x01] == 2.0 ** -9


def test_e2m1_values_from_bit_fields():
    # E2M1: sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0;
    # exponent 0 is subnormal (m * 2^-1).
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        v = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        v = -v if s else v
        assert E2M1_VALUES[c] == v and math.copysign(1, E2M1_VALUES[c]) == math.copysign(1, v if v else (-1 if s else 1))
    assert sorted(set(np.abs(E2M1_VALUES))) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize(
    "x,byte",
    [
        (6 * 448.0, 0x7E),  # saturates
        (-6 * 448.0, 0xFE),
        (448.0, 0x7E),
        (464.0, 0x7E),  # tie between 448 and 480: even -> 448
        (2.0 ** -10, 0x00),  # tie between 0 and 2^-9: even -> 0
        (-(2.0 ** -10), 0x80),  # keeps the sign of zero
        (1.5 * 2.0 ** -9, 0x02),  # tie between 1 and 2 units: even -> 2
        (2.5 * 2.0 ** -9, 0x02),  # tie between 2 and 3 units: even -> 2
        (3.5 * 2.0 ** -9, 0x04),
        (0.75 * 2.0 ** -9, 0x01),
        (1.0, 0x38),
        (1.0625, 0x38),  # tie between 1.0 (m=0) and 1.125 (m=1): even -> 1.0
        (1.1875, 0x3A),  # tie between 1.125 (m=1) and 1.25 (m=2): even -> 1.25
        (2.0 ** -6, 0x08),  # smallest normal
        (7.5 * 2.0 ** -9, 0x08),  # rounds up into the normal range (tie, even)
        (0.0, 0x00),
        (-0.0, 0x80),
        (float("nan"), 0x7F),
        (float("inf"), 0x7E),
    ],
)
def test_e4m3_encode_worked_values(x, byte):
    assert int(e4m3_encode(np.array([x]))[0]) == byte
    assert e4m3_encode_rational(x) == byte


def _all_products():
    codes = np.repeat(np.arange(16), 256)
    scales = np.tile(np.arange(256), 16)
    return codes, scales, E2M1_VALUES[codes] * E4M3_VALUES[scales]


def test_encoder_agrees_with_rational_encoder_on_all_4096_products():
    codes, scales, x = _all_products()
    got = e4m3_encode(x)
    for c, s, v, g in zip(codes, scales, x, got):
        if math.isnan(v):
            assert g == 0x7F
            continue
        if v == 0:
            want = e4m3_encode_rational(float(v))
        else:
            want = e4m3_encode_rational(Fraction(float(v)))
        assert g == want, (c, s, v)


def test_encoder_agrees_with_rational_encoder_on_random_and_midpoints():
    rng = np.random.default_rng(123)
    x = np.ldexp(rng.uniform(1, 2, 4000), rng.integers(-14, 11, 4000)) * rng.choice([-1, 1], 4000)
    # exact midpoints between adjacent E4M3 values
    pos = E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([x, mids, -mids])
    got = e4m3_encode(x)
    for v, g in zip(x, got):
        assert g == e4m3_encode_rational(Fraction(float(v))) or (v < 0 and g == e4m3_encode_rational(float(v)))


def test_encoder_matches_torch_cast_below_overflow():
    # torch's cast is round-to-nearest-even; it saturates only up to the 464 tie
    # and returns NaN above, so compare where |x| <= 464.
    _, _, x = _all_products()
    rng = np.random.default_rng(7)
    r = np.ldexp(rng.uniform(1, 2, 20000), rng.integers(-14, 9, 20000)) * rng.choice([-1, 1], 20000)
    x = np.concatenate([x, r]).astype(np.float32).astype(np.float64)
    x = x[~np.isnan(x) & (np.abs(x) <= 464)]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x), ref)


def _load_page_fixture():
    page = np.zeros(9216, dtype=np.uint8)
    expect = {}
    with open(os.path.join(GOLDEN, "nvfp4_page_layout.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "set":
                page[int(line[1])] = int(line[2], 16)
            elif line[0] == "expect":
                expect[(int(line[1]), int(line[2]))] = int(line[3], 16)
    return page, expect


def test_dequant_matches_hand_built_page():
    page, expect = _load_page_fixture()
    out = dequant_page(page)
    want = np.zeros((128, 128), dtype=np.uint8)
    for (t, d), b in expect.items():
        want[t, d] = b
    assert np.array_equal(out, want), np.argwhere(out != want)[:10]


def test_page_fields_layout_on_hand_built_page():
    page, _ = _load_page_fixture()
    codes, scales = page_fields(page.reshape(128, 72))
    assert codes[3, 4] == 0xA and codes[3, 5] == 0x7
    assert codes[127, 50] == 7 and codes[127, 51] == 0
    assert scales[3, 0] == 0x38 and scales[5, 7] == 0x30 and scales[127, 3] == 0x7E


def test_dequant_every_pair_inside_a_page():
    # all 16 codes x 256 scales laid into real pages: element (t, d) uses scale (t, d // 16)
    codes, scales, x = _all_products()
    pages = np.zeros((1, 9216), dtype=np.uint8)
    page = pages[0]
    # put pair k at token k // 32 ... one scale per group: 16 codes per group
    # 4096 pairs = 256 groups of 16 codes (group shares one scale).
    for gidx in range(256):
        t, g = divmod(gidx, 8)
        page[8192 + t * 8 + g] = gidx  # scale byte = gidx
        for j in range(16):
            d = g * 16 + j
            c = j
            b = t * 64 + d // 2
            if d % 2 == 0:
                page[b] = (page[b] & 0xF0) | c
            else:
                page[b] = (page[b] & 0x0F) | (c << 4)
    out = dequant_page(page)
    for gidx in range(256):
        t, g = divmod(gidx, 8)
        for j in range(16):
            v = E2M1_VALUES[j] * E4M3_VALUES[gidx]
            want = 0x7F if math.isnan(v) else e4m3_encode_rational(float(v) if v == 0 else Fraction(float(v)))
            assert out[t, g * 16 + j] == want


def test_gather_semantics_and_status():
    rng = np.random.default_rng(5)
    kv = rng.integers(0, 256, size=(6, 9216), dtype=np.uint8)
    kv[:, 8192:] = 0x38
    bt = np.array([[4, 1, 9, 0], [2, 3, 5, 5]], dtype=np.int32)  # 9 is out of range
    num_pages = np.array([3, 2], dtype=np.int32)
    page_offsets = np.array([0, 3], dtype=np.int32)
    out, status = gather_dequant(kv, bt, num_pages, page_offsets, 3, 5)
    assert status == ST_BLOCK_OOR
    assert np.array_equal(out[0], dequant_page(kv[4]))
    assert np.array_equal(out[1], dequant_page(kv[1]))
    assert not out[2].any()  # skipped (block 9)
    assert np.array_equal(out[3], dequant_page(kv[2]))
    assert np.array_equal(out[4], dequant_page(kv[3]))
    # output index past the buffer
    out, status = gather_dequant(kv, bt[1:], num_pages[1:], np.array([4]), 3, 5)
    assert status == ST_BAD_OUTPUT and np.array_equal(out[4], dequant_page(kv[2]))
    # max_num_pages bounds the gather
    out, status = gather_dequant(kv, bt, np.array([4, 4]), np.array([0, 1]), 1, 5)
    assert np.array_equal(out[0], dequant_page(kv[4])) and np.array_equal(out[1], dequant_page(kv[2]))
    assert not out[2:].any()
