"""GPU parity: gather/dequant bytes are bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from helpers import dev, host, status_word
from oracle.formats import E2M1_VALUES, E4M3_VALUES, e4m3_encode
from oracle.indexer import dequant_page, gather_dequant
from sparse_attention_indexer_nvfp4_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(lib, wl, out_pages=None, sentinel=0xA5):
    out_pages = wl["out_pages"] if out_pages is None else out_pages
    out = torch.full((out_pages, 128, 128), sentinel, dtype=torch.uint8, device="cuda")
    st = status_word()
    lib.idx_dequant_nvfp4_pages(dev(wl["kv"]), dev(wl["bt"]), dev(wl["num_pages"]), dev(wl["page_offsets"]),
                                wl["max_num_pages"], out, st)
    torch.cuda.synchronize()
    return host(out), int(st.item())


def test_every_code_scale_pair(lib):
    # 256 scale groups x 16 codes: all 4,096 (code, scale) pairs, NaN scales included
    page = np.zeros(9216, dtype=np.uint8)
    for gidx in range(256):
        t, g = divmod(gidx, 8)
        page[8192 + t * 8 + g] = gidx
        for j in range(16):
            d = g * 16 + j
            b = t * 64 + d // 2
            page[b] |= j if d % 2 == 0 else j << 4
    kv = page.reshape(1, 128, 72)
    wl = dict(kv=kv, bt=np.zeros((1, 1), np.int32), num_pages=np.ones(1, np.int32),
              page_offsets=np.zeros(1, np.int32), max_num_pages=1, out_pages=1)
    out, st = _run(lib, wl)
    assert st == 0
    want = dequant_page(page)
    assert np.array_equal(out[0], want)
    # NaN scales give the canonical 0x7F for every code
    for s in (0x7F, 0xFF):
        t, g = divmod(s, 8)
        assert (out[0, t, g * 16:(g + 1) * 16] == 0x7F).all()


def test_scaled_gather_with_special_scales(lib):
    wl = W.gather_workload(seed=21, num_reqs=24, max_pages=60, num_blocks=3000, special_frac=0.05)
    out, st = _run(lib, wl)
    want, st_ref = gather_dequant(wl["kv"], wl["bt"], wl["num_pages"], wl["page_offsets"], wl["max_num_pages"],
                                  wl["out_pages"])
    assert st == st_ref == 0
    assert np.array_equal(out, want)


def test_status_and_untouched_pages(lib):
    wl = W.gather_workload(seed=22, num_reqs=3, max_pages=5, num_blocks=50, min_pages=5)
    wl["bt"][0, 1] = 999  # out of range
    wl["bt"][2, 0] = -3
    wl["page_offsets"] = np.array([0, 5, 12], dtype=np.int32)  # request 2 runs past a 15-page buffer
    out, st = _run(lib, wl, out_pages=15)
    want = np.full((15, 128, 128), 0xA5, dtype=np.uint8)
    want, st_ref = gather_dequant(wl["kv"], wl["bt"], wl["num_pages"], wl["page_offsets"], 5, 15, out=want)
    assert st == st_ref and st & 1 and st & 4
    assert np.array_equal(out, want)
    assert (out[1] == 0xA5).all()  # skipped page untouched


def test_max_num_pages_and_table_width_bound(lib):
    wl = W.gather_workload(seed=23, num_reqs=4, max_pages=8, num_blocks=100, min_pages=8)
    wl["max_num_pages"] = 3
    out, st = _run(lib, wl)
    want = np.full_like(out, 0xA5)
    want, _ = gather_dequant(wl["kv"], wl["bt"], wl["num_pages"], wl["page_offsets"], 3, wl["out_pages"], out=want)
    assert np.array_equal(out, want)


def test_empty_work_launches_nothing(lib):
    wl = W.gather_workload(seed=24, num_reqs=2, max_pages=4, num_blocks=10)
    out = torch.zeros((8, 128, 128), dtype=torch.uint8, device="cuda")
    assert lib.idx_dequant_nvfp4_pages(dev(wl["kv"]), dev(wl["bt"]), dev(wl["num_pages"]), dev(wl["page_offsets"]),
                                       0, out) == 0
    torch.cuda.synchronize()
    assert not out.any()


@pytest.mark.slow
def test_full_size_gather(lib):
    """256 requests, num_pages U[1,1344], 200,000-page pool, 2% special scales:
    every output byte is written (two sentinels give identical outputs) and
    every gathered page equals the oracle's byte for byte."""
    from oracle import pool as oracle_pool

    wl = W.gather_workload(seed=1)
    args = (dev(wl["kv"]), dev(wl["bt"]), dev(wl["num_pages"]), dev(wl["page_offsets"]), wl["max_num_pages"])
    outs = []
    for sentinel in (0xA5, 0x5A):
        out = torch.full((wl["out_pages"], 128, 128), sentinel, dtype=torch.uint8, device="cuda")
        st = status_word()
        lib.idx_dequant_nvfp4_pages(*args, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    got = host(outs[0])
    del outs, args
    torch.cuda.empty_cache()
    bad, examples, st_ref = oracle_pool.gather_mismatches(wl, got)
    print(f"\ngather: {wl['out_pages']} pages compared, {bad} differ")
    assert st_ref == 0
    assert bad == 0, examples
