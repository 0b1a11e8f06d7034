"""The CPU oracle over full-size workloads on every host core (test infrastructure).

The oracle is used as it stands.  Each workload is cut into independent
pieces (a run of one request's pages, one request's gathered pages, one
token of the multi-token scorer) and every piece is one call of the
oracle's own function on a sub-batch that holds only that piece's inputs.
The pieces' results are put back together here, which is bookkeeping, not
arithmetic: the union of the pieces is the whole workload, and no piece
depends on another.

Workers are started with the 'spawn' method, so none inherits a CUDA
context from the test process; the large inputs (the index-K pool, the key
blocks, the GPU's gathered pages) reach them through shared memory, not
through pickling.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_W: dict = {}  # per-worker inputs
_SHM: list = []  # keeps the worker's shared-memory handles alive


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class Shared:
    """numpy arrays placed in shared memory for the workers."""

    def __init__(self, arrays: dict):
        self.blocks, self.spec = [], {}
        for name, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, a.dtype, buffer=shm.buf)[...] = a
            self.blocks.append(shm)
            self.spec[name] = (shm.name, a.shape, a.dtype.str)

    def close(self):
        for shm in self.blocks:
            shm.close()
            shm.unlink()
        self.blocks = []


def _init(spec: dict, small: dict):
    _W.clear()
    _W.update(small)
    for name, (shm_name, shape, dtype) in spec.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _SHM.append(shm)
        _W[name] = np.ndarray(shape, np.dtype(dtype), buffer=shm.buf)


def _run(spec: dict, small: dict, fn, tasks: list, chunksize: int = 1):
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=min(cores(), max(1, len(tasks))), initializer=_init, initargs=(spec, small)) as pool:
        return pool.map(fn, tasks, chunksize=chunksize)


# ---------------------------------------------------------------------------
# decode scores
# ---------------------------------------------------------------------------

def _decode_piece(task):
    from oracle.indexer import decode_scores

    b, j0, j1 = task
    w = _W
    s, wr, bd, st = decode_scores(w["q"][b:b + 1], w["q_scale"][b:b + 1], w["kv"], w["bt"][b:b + 1],
                                  w["seq_lens"][b:b + 1], w["query_len"], w["width"], w["max_blocks"],
                                  pages=[(0, j) for j in range(j0, j1)], page_tokens=w["page_tokens"])
    return b, j0, j1, s[0, :, j0:j1], wr[0, :, j0:j1], bd[0, :, j0:j1], st


def decode_scores_full(wl: dict, query_len: int = 8, piece: int = 128):
    """decode_scores over every page of the workload, on all host cores.

    Returns (scores, written, bound, status) exactly as one call of
    oracle.indexer.decode_scores on the whole batch would.
    """
    from oracle.indexer import ROWS, scored_pages

    B, width, mb = len(wl["seq_lens"]), int(wl["width"]), int(wl["max_blocks"])
    pt = int(wl.get("page_tokens", 128))
    tasks = []
    for b in range(B):
        n = scored_pages(wl["seq_lens"][b], mb, width, pt)
        tasks += [(b, j, min(j + piece, n)) for j in range(0, n, piece)]
        if n == 0:
            tasks.append((b, 0, 0))  # the request's status bits still count
    shared = Shared({"kv": wl["kv"]})
    try:
        small = {k: wl[k] for k in ("q", "q_scale", "bt", "seq_lens")}
        small.update(query_len=query_len, width=width, max_blocks=mb, page_tokens=pt)
        parts = _run(shared.spec, small, _decode_piece, tasks)
    finally:
        shared.close()
    scores = np.full((B, ROWS, width), np.nan, dtype=np.float32)
    written = np.zeros((B, ROWS, width), dtype=bool)
    bound = np.zeros((B, ROWS, width), dtype=np.float64)
    status = 0
    for b, j0, j1, s, wr, bd, st in parts:
        scores[b, :, j0:j1] = s
        written[b, :, j0:j1] = wr
        bound[b, :, j0:j1] = bd
        status |= st
    return scores, written, bound, status


# ---------------------------------------------------------------------------
# gather / dequant
# ---------------------------------------------------------------------------

def _gather_piece(task):
    from oracle.indexer import gather_dequant

    r, p0, p1 = task
    w = _W
    n = p1 - p0
    want, st = gather_dequant(w["kv"], w["bt"][r:r + 1, p0:p1], np.array([n], np.int32), np.zeros(1, np.int32),
                              n, n)
    got = w["gpu_out"][int(w["page_offsets"][r]) + p0:int(w["page_offsets"][r]) + p1]
    bad = np.nonzero((got != want).reshape(n, -1).any(axis=1))[0]
    return r, p0, int(len(bad)), [int(p0 + x) for x in bad[:4]], st


def gather_mismatches(g: dict, gpu_out: np.ndarray, piece: int = 256):
    """Compare every gathered output page with the oracle's dequantisation of
    its source page (byte for byte).  Returns (mismatched pages, examples,
    status)."""
    tasks = []
    for r in range(len(g["num_pages"])):
        n = min(int(g["num_pages"][r]), int(g["max_num_pages"]), g["bt"].shape[1])
        tasks += [(r, p, min(p + piece, n)) for p in range(0, n, piece)]
    shared = Shared({"kv": g["kv"], "gpu_out": gpu_out})
    try:
        parts = _run(shared.spec, {"bt": g["bt"], "page_offsets": g["page_offsets"]}, _gather_piece, tasks)
    finally:
        shared.close()
    bad = sum(p[2] for p in parts)
    examples = [(p[0], x) for p in parts for x in p[3]][:8]
    status = 0
    for p in parts:
        status |= p[4]
    return bad, examples, status


# ---------------------------------------------------------------------------
# multi-token scorer
# ---------------------------------------------------------------------------

def _mtp_piece(t):
    from oracle.indexer import mtp_scores

    w = _W
    s, bd = mtp_scores(w["q"], w["q_scale"], w["k"], w["k_scale"], w["bt"], w["num_keys"], w["cu_tokens"],
                       w["max_keys"], tokens=[t])
    return t, s[t], bd[t]


def mtp_scores_full(m: dict):
    """mtp_scores over every token of the workload, on all host cores."""
    T = int(m["cu_tokens"][-1])
    shared = Shared({"k": m["k"], "k_scale": m["k_scale"], "q": m["q"]})
    try:
        small = {k: m[k] for k in ("q_scale", "bt", "num_keys", "cu_tokens", "max_keys")}
        parts = _run(shared.spec, small, _mtp_piece, list(range(T)))
    finally:
        shared.close()
    out = np.full((T, m["max_keys"]), np.nan, dtype=np.float32)
    bound = np.zeros((T, m["max_keys"]), dtype=np.float64)
    for t, s, bd in parts:
        out[t], bound[t] = s, bd
    return out, bound


# ---------------------------------------------------------------------------
# timed samples (the CPU baseline of the benchmark)
# ---------------------------------------------------------------------------

def _decode_piece_count(task):
    b, j0, j1, _, wr, _, _ = _decode_piece(task)
    return int(wr.sum()), j1 - j0


class DecodeSampler:
    """A pool of workers holding one decode workload, timing the oracle on
    random pieces of it (each piece: one request's run of `piece` pages,
    dequantised and scored for all 32 rows)."""

    def __init__(self, wl: dict, query_len: int = 8, piece: int = 8, processes: int | None = None):
        from oracle.indexer import scored_pages

        self.piece = piece
        self.cores = processes or cores()
        pt = int(wl.get("page_tokens", 128))
        self.n = [scored_pages(s, wl["max_blocks"], wl["width"], pt) for s in wl["seq_lens"]]
        self.shared = Shared({"kv": wl["kv"]})
        small = {k: wl[k] for k in ("q", "q_scale", "bt", "seq_lens")}
        small.update(query_len=query_len, width=int(wl["width"]), max_blocks=int(wl["max_blocks"]), page_tokens=pt)
        self.pool = mp.get_context("spawn").Pool(processes=self.cores, initializer=_init,
                                                 initargs=(self.shared.spec, small))
        first = next(b for b, n in enumerate(self.n) if n > 0)
        self.pool.map(_decode_piece_count, [(first, 0, 1)] * self.cores)  # workers up and warm

    def rate(self, seconds: float, seed: int = 0):
        """Scores per second over about `seconds` with every worker busy,
        pieces handed out in rounds of a few per worker; returns (rate, pages,
        wall seconds)."""
        import time

        rng = np.random.default_rng(seed)
        live = [b for b, n in enumerate(self.n) if n > 0]
        done = pages = 0
        t0 = time.perf_counter()
        while True:
            tasks = []
            for _ in range(4 * self.cores):
                b = int(rng.choice(live))
                j0 = int(rng.integers(0, max(1, self.n[b] - self.piece + 1)))
                tasks.append((b, j0, min(self.n[b], j0 + self.piece)))
            for written, np_ in self.pool.map(_decode_piece_count, tasks, chunksize=1):
                done += written
                pages += np_
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        return done / dt, pages, dt

    def close(self):
        self.pool.terminate()
        self.pool.join()
        self.shared.close()
