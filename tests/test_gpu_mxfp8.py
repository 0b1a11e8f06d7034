"""GPU parity: MXFP8 quantisation of bf16 rows is bit-exact against the oracle
(values and E8M0 scales), on random rows over a wide dynamic range, the
worked edge blocks, non-finite inputs, strided rows and the decode-batch
shape of the pages (K = 2048 per rank)."""

import numpy as np
import pytest
import torch

from helpers import dev, host
from oracle.mxfp8 import mxfp8_quantize

pytestmark = pytest.mark.gpu


def _bits(rng, rows, cols, lo=-40, hi=40):
    # bf16 values over ~2^80 of dynamic range, both signs, some zeros
    x = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(lo, hi, size=(rows, 1)))).astype(np.float32)
    x[rng.random(x.shape) < 0.02] = 0.0
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _run(lib, bits, x_stride=None, out_stride=None, scale_stride=None):
    rows, cols = bits.shape
    xs = x_stride or cols
    buf = np.zeros((rows, xs), dtype=np.uint16)
    buf[:, :cols] = bits
    x = dev(buf).view(torch.bfloat16)
    out = torch.full((rows, out_stride or cols), 0xA5, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows, scale_stride or cols // 32), 0xA5, dtype=torch.uint8, device="cuda")
    lib.idx_mxfp8_quantize(x[:, :cols] if xs != cols else x, out[:, :cols] if out_stride else out,
                           sc[:, :cols // 32] if scale_stride else sc)
    torch.cuda.synchronize()
    return host(out), host(sc)


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (16, 2048), (37, 4096), (200, 2048)])
def test_random_rows(lib, rows, cols):
    bits = _bits(np.random.default_rng(rows * 7 + cols), rows, cols)
    q, s = _run(lib, bits)
    want_q, want_s = mxfp8_quantize(bits)
    assert np.array_equal(s, want_s)
    assert np.array_equal(q, want_q)


def test_edge_and_non_finite_blocks(lib):
    edges = [0x0000, 0x8000, 0x0001, 0x807F, 0x0080, 0x43DF, 0x43E0, 0x43E1, 0xC3E1, 0x3FE0, 0x3FE1, 0x7F7F,
             0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0x3F80]
    rows = []
    for v in edges:
        rows.append(np.full(32, v, dtype=np.uint16))
        blk = np.full(32, 0x3F00, dtype=np.uint16)
        blk[7] = v
        rows.append(blk)
    bits = np.stack(rows)  # one block per row
    q, s = _run(lib, bits)
    want_q, want_s = mxfp8_quantize(bits)
    assert np.array_equal(s, want_s)
    assert np.array_equal(q, want_q)


def test_strided_rows_leave_padding_untouched(lib):
    bits = _bits(np.random.default_rng(5), 9, 256)
    q, s = _run(lib, bits, x_stride=264, out_stride=272, scale_stride=11)
    want_q, want_s = mxfp8_quantize(bits)
    assert np.array_equal(q[:, :256], want_q) and (q[:, 256:] == 0xA5).all()
    assert np.array_equal(s[:, :8], want_s) and (s[:, 8:] == 0xA5).all()


@pytest.mark.slow
def test_large_batch_sampled_rows(lib):
    """16,384 rows x 2,048: every row's scales against the oracle, the values
    of 64 sampled rows, and repeated launches bit-identical."""
    bits = _bits(np.random.default_rng(11), 16384, 2048)
    q, s = _run(lib, bits)
    rng = np.random.default_rng(12)
    for r in rng.integers(0, 16384, size=64):
        wq, ws = mxfp8_quantize(bits[r:r + 1])
        assert np.array_equal(q[r], wq[0]) and np.array_equal(s[r], ws[0])
    amax = (bits & 0x7FFF).reshape(16384, 64, 32).max(axis=2).astype(np.int64)
    want_s = np.clip(((amax >> 7) & 0xFF) - 8 + ((amax & 0x7F) > 96), 0, 254)
    assert np.array_equal(s, want_s.astype(np.uint8))
    q2, s2 = _run(lib, bits)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
