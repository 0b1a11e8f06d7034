"""Shared helpers for the GPU parity tests (device copies, sentinels, checks)."""

import numpy as np
import torch

SENTINEL_BITS = 0x7FBADBAD  # a NaN payload the kernels never write


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def sentinel_f32(shape) -> torch.Tensor:
    return torch.full(shape, SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)


def untouched(a: np.ndarray) -> np.ndarray:
    return a.view(np.int32) == SENTINEL_BITS


def status_word() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def decode_args(wl: dict):
    return dict(
        q=dev(wl["q"]), q_scale=dev(wl["q_scale"]), kv=dev(wl["kv"]), block_table=dev(wl["bt"]),
        seq_lens=dev(wl["seq_lens"]),
    )


def check_scores(gpu: np.ndarray, ref: np.ndarray, written: np.ndarray, bound: np.ndarray) -> dict:
    """Written entries within tolerance; every other entry untouched."""
    assert np.array_equal(~untouched(gpu), written), "written/untouched pattern differs"
    g, r, b = gpu[written], ref[written], bound[written]
    nan_r = np.isnan(r)
    assert np.array_equal(np.isnan(g), nan_r), "NaN pattern differs"
    err = np.abs(g[~nan_r].astype(np.float64) - r[~nan_r].astype(np.float64))
    bad = err > b[~nan_r]
    assert not bad.any(), f"{int(bad.sum())} scores outside tolerance; worst {err.max()}"
    rel = err / np.maximum(b[~nan_r], 1e-30)
    return dict(n=int(written.sum()), max_err_over_bound=float(rel.max()) if rel.size else 0.0)


def selection_within_tolerance(gpu_out: np.ndarray, ref_out: np.ndarray, ref_scores: np.ndarray,
                               ref_bound: np.ndarray, query_len: int) -> int:
    """End-to-end decode rows vs the oracle's own: rows may differ only where the
    oracle scores of the differing pages are within tolerance of each other.
    Returns the number of rows that differ (each explained by such a near-tie)."""
    B = gpu_out.shape[0]
    differ = 0
    for b in range(B):
        for i in range(query_len):
            slot = 8 - query_len + i
            for h in range(4):
                g, r = gpu_out[b, i, h], ref_out[b, i, h]
                if np.array_equal(g, r):
                    continue
                differ += 1
                assert g[15] == r[15]
                row = slot * 4 + h
                gs = sorted((float(ref_scores[b, row, p]) for p in g[:15] if p >= 0), reverse=True)
                rs = sorted((float(ref_scores[b, row, p]) for p in r[:15] if p >= 0), reverse=True)
                tol = 2 * float(ref_bound[b, row].max())
                assert len(gs) == len(rs) and all(abs(x - y) <= tol for x, y in zip(gs, rs)), (b, i, h)
    return differ


def topk_within_tolerance(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_scores: np.ndarray,
                          ref_bound: np.ndarray) -> int:
    """Top-16 rows of the GPU's scores vs the oracle's own: a row may differ
    only where the oracle scores of the two selections agree within twice the
    row's tolerance, rank by rank.  Returns the number of rows that differ."""
    differ = 0
    for r in range(gpu_idx.shape[0]):
        g, w = gpu_idx[r], ref_idx[r]
        if np.array_equal(g, w):
            continue
        differ += 1
        gs = sorted((float(ref_scores[r, c]) for c in g if c >= 0), reverse=True)
        ws = sorted((float(ref_scores[r, c]) for c in w if c >= 0), reverse=True)
        tol = 2 * float(np.nanmax(ref_bound[r]))
        assert len(gs) == len(ws) and all(abs(x - y) <= tol for x, y in zip(gs, ws)), r
    return differ
