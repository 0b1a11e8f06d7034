#!/usr/bin/env python3
"""Benchmark of the sparse-attention indexer decode path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--quick]

A step is one indexer decode step (score every page below each query's own
page, then the exact top-16 rows) over the batched-decode workload: 64
requests, seq_len U[8K, 168K], 8 query slots x 4 index heads x depth 128,
1,344-column score rows, 1% duplicated pages.  Inputs are synthetic
(seeded), resident in HBM before the timed region; the 415 MB index-K pool
is larger than the 129 MB L2, so L2 is not flushed between steps.

The JSON line also carries: the dominant kernel's roofline (decode scorer,
algorithmic bytes / CUDA-event time, against MEASURED_PEAKS.json), the CPU
oracle timed on a bounded sample of the same workload, an end-to-end number
through the C ABI with host buffers (per-step H2D of the queries, scales,
lengths and block table, D2H of the rows), SM clocks sampled during the
timed region, and secondary lines for the gather/dequant, long-context and
multi-token workloads.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica
of the workload (independent requests, no collective on the data path), the
reported time is the max over ranks, and value counts all ranks' work.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexer decode (query,head,page) scores/s + top-16 rows/s; index-K GB/s vs HBM peak"
REPEATS = 5  # timed regions of K steps; the median is reported
UNIT = "scores/s"
PAGE_BYTES = 9216


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1946.9)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# Sources each kernel is built from (its own file and the headers it
# includes beyond the shared ones).
KERNEL_SOURCES = {
    "k_score_decode": ["idx_score_tc.cu", "idx_fused.cuh", "idx_select.cuh", "idx_internal.h"],
    "k_topk_rows": ["idx_topk.cu", "idx_select.cuh", "idx_internal.h"],
    "k_mtp_tc": ["idx_mtp_tc.cu", "idx_internal.h"],
    "k_dequant_nvfp4": ["idx_dequant.cu", "idx_internal.h"],
}
SHARED_SOURCES = ["idx_common.cuh", "idx_tc.cuh", "../../include/idx.h"]  # device code the kernels include


def _kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_nvfp4_gb300", "csrc")
    for n in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        with open(os.path.normpath(os.path.join(csrc, n)), "rb") as f:
            h.update(os.path.basename(n).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def _recorded_traffic(kernel: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/traffic.txt
    (lines "kernel bytes_per_launch source_hash"), valid only while the
    kernel's sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = _kernel_hash(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split("#")[0].split()
            if len(parts) >= 3 and parts[0] == kernel and parts[2] == cur:
                return float(parts[1])
    return None


# ---------------------------------------------------------------------------
# replicas across ranks
# ---------------------------------------------------------------------------

def replica_seed(rank: int) -> int:
    """Seed of rank's replica of the batched decode workload (rank 0: seed 2)."""
    return 2 + 1000 * rank


def max_over_ranks(dist, values, device):
    """Element-wise max of per-rank timings (every rank gets the result);
    identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * world / (ms_max / 1000.0)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"idx_clocks_{os.getpid()}.csv")

    def start(self):
        """Start sampling and return once the first sample is written, so the
        tool's own start-up does not overlap the timed region."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 10.0:
            self.f.flush()
            try:
                if os.path.getsize(self.path) > 0 and open(self.path).read().count("\n") >= 2:
                    break
            except OSError:
                pass
            time.sleep(0.05)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def decode_units(wl) -> dict:
    """Work of one decode step: (query, head, page) scores, rows, index-K pages."""
    from sparse_attention_indexer_nvfp4_gb300.workloads import PAGE_TOKENS

    q_len, width, mb = wl["query_len"], wl["width"], wl["max_blocks"]
    scores = rows = pages = stored = 0
    for s in wl["seq_lens"]:
        s = int(s)
        n = max(0, min((s - 1) // PAGE_TOKENS, mb, width))
        pages += n
        for i in range(q_len):
            own = (s - q_len + i) // PAGE_TOKENS
            k = max(0, min(own, n))
            scores += 4 * k
            stored += 4 * k
            rows += 4
    B = len(wl["seq_lens"])
    # scorer algorithmic bytes: index-K pages + block ids + score stores + queries, scales, lengths
    score_bytes = pages * (PAGE_BYTES + 4) + stored * 4 + B * (32 * 128 + 32 * 4 + 4)
    return dict(scores=scores, rows=rows, pages=pages, score_bytes=score_bytes)


class Timer:
    """CUDA-event timing on the launching stream."""

    def __init__(self, torch, stream):
        self.torch, self.stream = torch, stream

    def run(self, fn, iters: int) -> float:
        t = self.torch
        start = t.cuda.Event(enable_timing=True)
        end = t.cuda.Event(enable_timing=True)
        t.cuda.synchronize()
        start.record(self.stream)
        for _ in range(iters):
            fn()
        end.record(self.stream)
        t.cuda.synchronize()
        return start.elapsed_time(end) / iters  # ms

    def graph_median(self, fn, per_graph: int = 50, replays: int = 15) -> float:
        """Median over `replays` replays of a CUDA graph of `per_graph` calls of
        fn, in ms per call (for launches too short to time one by one)."""
        t = self.torch
        fn()
        t.cuda.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g):
            for _ in range(per_graph):
                fn()
        g.replay()
        t.cuda.synchronize()
        stream = t.cuda.current_stream()
        vals = []
        for _ in range(replays):
            start = t.cuda.Event(enable_timing=True)
            end = t.cuda.Event(enable_timing=True)
            start.record(stream)
            g.replay()
            end.record(stream)
            t.cuda.synchronize()
            vals.append(start.elapsed_time(end) / per_graph)
        return statistics.median(vals)

    def run_graph(self, fn, iters: int, per_graph: int = 20) -> float:
        """Like run(), for sequences of short kernels whose host-side launch
        cost would otherwise show up as idle gaps: `per_graph` calls of fn are
        captured into one CUDA graph, which is replayed."""
        t = self.torch
        fn()
        t.cuda.synchronize()
        g = t.cuda.CUDAGraph()
        with t.cuda.graph(g):
            for _ in range(per_graph):
                fn()
        g.replay()
        t.cuda.synchronize()
        reps = max(1, iters // per_graph)
        start = t.cuda.Event(enable_timing=True)
        end = t.cuda.Event(enable_timing=True)
        stream = t.cuda.current_stream()
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
        t.cuda.synchronize()
        return start.elapsed_time(end) / (reps * per_graph)  # ms


# ---------------------------------------------------------------------------
# CPU oracle baseline
# ---------------------------------------------------------------------------

def cpu_baseline_samples(wl, seconds: float, repeats: int = 3):
    """The oracle as it stands, timed on every host core: a pool of worker
    processes (one per core of this process's affinity set) scores random
    8-page runs of the workload's requests (dequantise each page, score it
    for all 32 rows), `repeats` samples of about `seconds` each.  Returns
    (median scores/s, cores, pages per sample, seconds per sample)."""
    from oracle.pool import DecodeSampler

    sampler = DecodeSampler(wl, query_len=wl["query_len"])
    try:
        runs = [sampler.rate(seconds, seed=k) for k in range(repeats)]
    finally:
        sampler.close()
    rates = sorted(r for r, _, _ in runs)
    return rates[len(rates) // 2], sampler.cores, runs[0][1], statistics.median(dt for _, _, dt in runs)


def run_reference(args, wl, rank: int):
    """The reference arm: the CPU oracle (there is no other implementation
    of this path to install), on all host cores, one bounded sample of the
    workload per step; the rate is the median over the timed steps and
    ms_per_step the time the oracle would take for one whole step at that
    rate."""
    if rank != 0:
        return
    from oracle.pool import DecodeSampler

    budget = 6.0 if args.quick else 20.0
    per = max(0.5, budget / max(1, args.steps + args.warmup))
    sampler = DecodeSampler(wl, query_len=wl["query_len"])
    try:
        runs = [sampler.rate(per, seed=s) for s in range(args.warmup + args.steps)][args.warmup:]
    finally:
        sampler.close()
    rate = statistics.median(r for r, _, _ in runs)
    units = decode_units(wl)
    ms = 1000.0 * units["scores"] / rate
    pages = sum(p for _, p, _ in runs)
    sample = (f"{pages} random pages in 8-page runs over {len(runs)} timed samples of {per:.1f} s "
              f"(dequant + 32-row scores each), {sampler.cores} worker processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64/f64 exact (oracle)", "data": "synthetic",
        "config": {"workload": "batched decode: 64 requests, seq_len U[8K,168K], 8 slots x 4 heads x 128, "
                               "1,344-column rows, 1% duplicated pages", "seed": 2,
                   "timing": "ms_per_step = one whole step's scores at the median sampled rate; "
                             f"each step samples {per:.1f} s"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": sampler.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args, wl, rank: int, world: int, dist):
    import torch

    import sparse_attention_indexer_nvfp4_gb300 as idx
    from sparse_attention_indexer_nvfp4_gb300 import workloads as W

    idx.load_library()
    dev_idx = torch.cuda.current_device()
    stream = torch.cuda.current_stream()
    timer = Timer(torch, stream)
    hbm_peak, bf16_peak, peak_kind = _peaks()

    def to_dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    q, qs, kv, bt, sl = (to_dev(wl[k]) for k in ("q", "q_scale", "kv", "bt", "seq_lens"))
    B = len(wl["seq_lens"])
    width, qlen = wl["width"], wl["query_len"]
    scores = torch.empty((B, 32, width), dtype=torch.float32, device="cuda")
    out = torch.empty((B, qlen, 4, 16), dtype=torch.int32, device="cuda")
    ws_bytes = idx.idx_decode_workspace_bytes(B, qlen, width)
    ws = torch.empty(max(8, ws_bytes) // 8, dtype=torch.int64, device="cuda") if ws_bytes else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    units = decode_units(wl)
    launches_per_step = 2 + (1 if ws_bytes > 0 else 0)  # scorer, selector (+ split-row merge)

    def step():
        idx.idx_decode_step(q, qs, kv, bt, sl, qlen, scores, out, ws, status)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    def timed(fn):
        """REPEATS timed regions of exactly K steps, each bracketed by a
        barrier and a synchronize; the median region's ms per step."""
        vals = []
        for _ in range(REPEATS):
            if dist is not None:
                dist.barrier()
            torch.cuda.synchronize()
            vals.append(timer.run(fn, args.steps))
        return statistics.median(vals), vals

    sampler = ClockSampler(dev_idx)
    sampler.start()
    ms, ms_repeats = timed(step)
    # dominant kernel: the decode scorer, timed alone over the same inputs
    ms_score, _ = timed(lambda: idx.idx_score_pages(q, qs, kv, bt, sl, qlen, scores, status))
    clocks = sampler.stop()

    # End to end through the C ABI with host buffers: every step copies its
    # inputs (q, q_scale, block table, seq_lens, packed into one pinned
    # buffer) host -> device and its rows device -> host.  The copies run on
    # two copy streams and the buffers are double-buffered, so step k+1's
    # inputs and step k-1's rows move while step k computes, as a serving
    # loop would run it.
    def packed_inputs(device):
        parts, off = [], 0
        for name in ("q", "q_scale", "bt", "seq_lens"):
            a = np.ascontiguousarray(wl[name])
            parts.append((name, a, off))
            off += -(-a.nbytes // 256) * 256
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if device == "cpu":
            buf = buf.pin_memory()
        views = {}
        for name, a, o in parts:
            v = buf[o:o + a.nbytes].view(getattr(torch, str(a.dtype))).view(a.shape)
            if device == "cpu":
                v.copy_(torch.from_numpy(a))
            views[name] = v
        return buf, views

    nslot = 2
    h_in = [packed_inputs("cpu") for _ in range(nslot)]
    d_in = [packed_inputs("cuda") for _ in range(nslot)]
    d_out = [torch.empty_like(out) for _ in range(nslot)]
    h_out = [torch.empty(tuple(out.shape), dtype=torch.int32).pin_memory() for _ in range(nslot)]
    h2d = h_in[0][0].numel()
    d2h = h_out[0].numel() * h_out[0].element_size()
    comp = torch.cuda.current_stream()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nslot)]
    ev_comp = [torch.cuda.Event() for _ in range(nslot)]
    ev_out = [torch.cuda.Event() for _ in range(nslot)]
    e2e_count = [0]

    def e2e_step():
        k = e2e_count[0]
        e2e_count[0] += 1
        sl_ = k % nslot
        with torch.cuda.stream(s_h2d):
            if k >= nslot:
                s_h2d.wait_event(ev_comp[sl_])  # step k - 2 has read this slot's inputs
            d_in[sl_][0].copy_(h_in[sl_][0], non_blocking=True)
            ev_in[sl_].record(s_h2d)
        comp.wait_event(ev_in[sl_])
        if k >= nslot:
            comp.wait_event(ev_out[sl_])  # step k - 2's rows have left this slot's output
        v = d_in[sl_][1]
        idx.idx_decode_step(v["q"], v["q_scale"], kv, v["bt"], v["seq_lens"], qlen, scores, d_out[sl_], ws, status)
        ev_comp[sl_].record(comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_comp[sl_])
            h_out[sl_].copy_(d_out[sl_], non_blocking=True)
            ev_out[sl_].record(s_d2h)

    def e2e_run(iters):
        for _ in range(iters):
            e2e_step()
        for e in ev_out:
            comp.wait_event(e)  # the last rows are on the host before the clock stops

    e2e_run(2)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(comp)
    e2e_run(args.steps)
    t_end.record(comp)
    torch.cuda.synchronize()
    ms_e2e = t_start.elapsed_time(t_end) / args.steps
    assert all(torch.equal(h, out.cpu()) for h in h_out)
    # the job's time is the slowest rank's
    ms, ms_e2e = max_over_ranks(dist, [ms, ms_e2e], "cuda")

    extra = {}
    if args.legs and rank == 0:
        extra = secondary(args, torch, idx, W, timer, hbm_peak, dict(q=q, qs=qs, kv=kv, bt=bt, sl=sl, wl=wl))

    total_scores = units["scores"] * world
    value = whole_job_rate(units["scores"], world, ms)
    achieved = units["score_bytes"] / (ms_score / 1000.0) / 1e9
    traffic = _recorded_traffic("k_score_decode")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic",
        "config": {
            "workload": "batched decode: 64 requests, seq_len U[8K,168K], 8 slots x 4 heads x 128, "
                        "1,344-column rows, 1% duplicated pages (seed 2)",
            "requests_per_gpu": B, "pages_per_step": units["pages"], "scores_per_step": units["scores"],
            "index_k_bytes_per_step": units["pages"] * PAGE_BYTES,
            "l2": "not flushed: the index-K pool (%.0f MB) exceeds the 129 MB L2" % (wl["kv"].nbytes / 1e6),
            "parallelism": f"replicas x{world}",
            "timing": f"median of {REPEATS} timed regions of {args.steps} steps (CUDA events on the launching "
                      "stream, barrier + synchronize around each)",
            "ms_per_step_repeats": ms_repeats,
        },
        "rows_per_s": units["rows"] * world / (ms / 1000.0),
        "index_k_gbs": units["pages"] * PAGE_BYTES * world / (ms / 1000.0) / 1e9,
        "index_k_frac_of_hbm": units["pages"] * PAGE_BYTES / (ms / 1000.0) / 1e9 / hbm_peak,
        "roofline": {
            "kernel": "k_score_decode", "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": traffic, "peak_kind": peak_kind,
            "ms_per_launch": ms_score, "algorithmic_bytes_per_launch": units["score_bytes"],
        },
        "e2e": {"value": total_scores / (ms_e2e / 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "note": "index-K cache resident in HBM (decode state); every step copies its packed inputs "
                        "from pinned host memory and its rows back, on two copy streams, double-buffered so "
                        "the copies overlap the neighbouring steps' compute"},
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "extra": extra,
    }
    if rank == 0 and world == 1:
        seconds = 2.0 if args.quick else 5.0
        rate, cores, pages, dt = cpu_baseline_samples(wl, seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"median of 3 samples of {dt:.1f} s, each ~{pages} random pages of the "
                                          f"same workload in 8-page runs (dequant + 32-row scores), {cores} worker "
                                          "processes (all cores of the affinity set)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def secondary(args, torch, idx, W, timer, hbm_peak, main) -> dict:
    """Other workloads of the path, each timed with CUDA events."""
    res = {}
    iters = max(3, args.steps // 4)

    def to_dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    fp8_peak = None
    if "fp8" in args.legs:
        # dense FP8 tensor-core rate (tcgen05.mma kind::f8f6f4, M=128 x N=256 x K=32, one CTA per SM), the
        # denominator of the multi-token and prefill scorers' tensor figures; median of 5 launches of ~3 ms
        chk = torch.zeros(1, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        n_it = 10000
        flops = idx.idx_fp8_mma_probe(n_it, chk, st)
        torch.cuda.synchronize()
        assert float(chk.item()) == 32.0 * n_it and int(st.item()) == 0
        vals = [timer.run(lambda: idx.idx_fp8_mma_probe(n_it, None, st), 1) for _ in range(5)]
        fp8_peak = flops / (statistics.median(vals) / 1e3) / 1e12
        res["fp8_dense_peak"] = {"tflops": fp8_peak, "ms_per_launch": statistics.median(vals),
                                 "method": "idx_fp8_mma_probe: one CTA per SM issues 4 x 10,000 tcgen05.mma "
                                           "kind::f8f6f4 M=128 x N=256 x K=32 (E4M3, fp32 accumulation in TMEM) "
                                           "back to back; CUDA events, median of 5 launches",
                                 "frac_of_nominal_4500": fp8_peak / 4500.0}

    if "tiny" in args.legs:
        # tiny decode: 1 request x 4,096 tokens, 31 pages scored
        t = W.tiny_decode(0)
        q, qs, kv, bt, sl = (to_dev(t[k]) for k in ("q", "q_scale", "kv", "bt", "seq_lens"))
        sc = torch.empty((1, 32, t["width"]), dtype=torch.float32, device="cuda")
        out = torch.empty((1, 8, 4, 16), dtype=torch.int32, device="cuda")
        ms = timer.graph_median(lambda: idx.idx_decode_step(q, qs, kv, bt, sl, 8, sc, out), 50, 15)
        u = decode_units(t)
        res["tiny_decode"] = {"workload": "1 request x 4,096 tokens (31 pages scored), 8 slots x 4 heads",
                              "us_per_step": ms * 1e3, "scores_per_s": u["scores"] / (ms / 1e3),
                              "timing": "CUDA graph of 50 steps, median of 15 replays", "launches": 2}

    if "qlen1" in args.legs:
        # query_len 1 (4 live rows per request) on the batched workload: the
        # decode step and its scorer (the tensor-core kernel at every query_len)
        m = main
        B = len(m["wl"]["seq_lens"])
        sc = torch.empty((B, 32, m["wl"]["width"]), dtype=torch.float32, device="cuda")
        out1 = torch.empty((B, 1, 4, 16), dtype=torch.int32, device="cuda")
        score = timer.run(lambda: idx.idx_score_pages(m["q"], m["qs"], m["kv"], m["bt"], m["sl"], 1, sc), iters)
        step1 = timer.run(lambda: idx.idx_decode_step(m["q"], m["qs"], m["kv"], m["bt"], m["sl"], 1, sc, out1), iters)
        u1 = decode_units(dict(m["wl"], query_len=1))
        res["query_len_1"] = {"workload": "batched decode, query_len 1 (4 live rows per request)",
                              "ms_step": step1, "ms_scorer": score, "scores_per_s": u1["scores"] / (step1 / 1e3),
                              "index_k_gbs": u1["pages"] * PAGE_BYTES / (score / 1e3) / 1e9}

    if "fused" in args.legs:
        # the fused decode step (selection in the scorer's CTAs, one launch)
        # against the two-launch step, alternating, on the main workload and
        # the long-context one; rows must be identical
        res["fused"] = {}
        for name in ("batched", "long_context"):
            if name == "batched":
                wl, q, qs, kv, bt, sl = main["wl"], main["q"], main["qs"], main["kv"], main["bt"], main["sl"]
            else:
                wl = W.long_context()
                q, qs, kv, bt, sl = (to_dev(wl[k]) for k in ("q", "q_scale", "kv", "bt", "seq_lens"))
            B, width = len(wl["seq_lens"]), wl["width"]
            sc = torch.empty((B, 32, width), dtype=torch.float32, device="cuda")
            out_c = torch.empty((B, 8, 4, 16), dtype=torch.int32, device="cuda")
            out_f = torch.full_like(out_c, -7)
            wsb = idx.idx_decode_workspace_bytes(B, 8, width)
            ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
            wsf = torch.zeros(idx.idx_decode_fused_workspace_bytes(B) // 8, dtype=torch.int64, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            chain = lambda: idx.idx_decode_step(q, qs, kv, bt, sl, 8, sc, out_c, ws, st)
            fused = lambda: idx.idx_decode_step(q, qs, kv, bt, sl, 8, sc, out_f, wsf, st, flags=idx.FUSED_SELECT)
            chain()
            fused()
            torch.cuda.synchronize()
            same = bool(torch.equal(out_c, out_f)) and int(st.item()) == 0
            tc, tf = [], []
            for _ in range(3):
                tc.append(timer.run(chain, iters))
                tf.append(timer.run(fused, iters))
            same = same and bool(torch.equal(out_c, out_f)) and int(wsf[: (B + 1) // 2].abs().sum().item()) == 0
            u = decode_units(wl)
            mc, mf = statistics.median(tc), statistics.median(tf)
            res["fused"][name] = {"ms_two_launch": mc, "ms_fused": mf, "rows_identical": same,
                                  "fused_frac_of_hbm": u["pages"] * PAGE_BYTES / (mf / 1e3) / 1e9 / hbm_peak,
                                  "launches_fused": 1, "launches_two_launch": 2 + (1 if wsb else 0)}
            if name != "batched":
                del q, qs, kv, bt, sl
            del sc, out_c, out_f, ws, wsf, wl
            torch.cuda.empty_cache()

    if "p256" in args.legs:
        # the batched decode on P256 pages: 672-column rows, each page scored as two 128-key halves
        wl = W.batched_decode(page_tokens=256)
        q, qs, kv, bt, sl = (to_dev(wl[k]) for k in ("q", "q_scale", "kv", "bt", "seq_lens"))
        B = len(wl["seq_lens"])
        sc = torch.empty((B, 32, 2 * wl["width"]), dtype=torch.float32, device="cuda")
        out = torch.empty((B, 8, 4, 16), dtype=torch.int32, device="cuda")
        wsb = idx.idx_decode_workspace_bytes(B, 8, wl["width"])
        ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
        fn = lambda: idx.idx_decode_step(q, qs, kv, bt, sl, 8, sc, out, ws, flags=idx.PAGE_256)
        fn()
        ms = timer.run(fn, iters)
        units = sum(2 * max(0, min((int(s) - 1) // 256, wl["width"])) for s in wl["seq_lens"])
        pages = units // 2
        byts = units * PAGE_BYTES
        res["p256"] = {"workload": "batched decode on P256 pages: 64 requests, seq_len U[8K,168K], 672-column rows",
                       "ms": ms, "pages_per_step": pages, "scores_per_s": pages * 32 / (ms / 1e3),
                       "index_k_gbs": byts / (ms / 1e3) / 1e9, "frac_of_hbm": byts / (ms / 1e3) / 1e9 / hbm_peak,
                       "launches": 2 + (1 if wsb else 0)}
        del q, qs, kv, bt, sl, sc, out, ws, wl
        torch.cuda.empty_cache()

    if "sweep" in args.legs:
        # standalone top-16: 4,096 rows per width, 1% specials and ties, ragged valid counts
        out = torch.empty((4096, 16), dtype=torch.int32, device="cuda")
        widths = {}
        for w in W.SWEEP_WIDTHS:
            d = W.topk_rows(100 + w, 4096, w)
            x, vn = to_dev(d["scores"]), to_dev(d["valid_n"])
            wsb = idx.idx_workspace_bytes(4096, w)
            ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
            ms = timer.graph_median(lambda: idx.idx_topk16_select(x, out, valid_n=vn, workspace=ws), 20, 15)
            widths[str(w)] = {"us": ms * 1e3, "score_gbs": 4096 * w * 4 / (ms / 1e3) / 1e9,
                              "rows_per_s": 4096 / (ms / 1e3)}
            del x, vn, ws
        res["topk_sweep"] = {"workload": "4,096 rows per width, 1% +-inf/NaN/+-0/FLT_MAX and ties, valid counts "
                                         "0..width+8", "timing": "CUDA graph of 20 calls, median of 15 replays",
                             "widths": widths}

    if "mxfp8" in args.legs:
        # MXFP8 quantisation of bf16 rows: a decode batch (16 rows x 2,048) and a large block (16,384 x 2,048)
        rng = np.random.default_rng(5)
        mx = {}
        for rows in (16, 16384):
            x = torch.from_numpy(rng.standard_normal((rows, 2048)).astype(np.float32)).cuda().to(torch.bfloat16)
            o = torch.empty((rows, 2048), dtype=torch.uint8, device="cuda")
            sc = torch.empty((rows, 64), dtype=torch.uint8, device="cuda")
            ms = timer.graph_median(lambda: idx.idx_mxfp8_quantize(x, o, sc), 50 if rows == 16 else 10, 15)
            byts = rows * 2048 * (2 + 1) + rows * 64
            mx[str(rows)] = {"us": ms * 1e3, "gbs": byts / (ms / 1e3) / 1e9,
                             "frac_of_hbm": byts / (ms / 1e3) / 1e9 / hbm_peak}
        res["mxfp8"] = {"workload": "bf16 rows x 2,048 columns (32-element MX blocks)",
                        "timing": "CUDA graph of 50 (16 rows) / 10 (16,384 rows) calls, median of 15 replays",
                        "rows": mx}

    if "gather" in args.legs:
        # gather/dequant: 256 requests, num_pages U[1,1344], 200,000-page pool
        g = W.gather_workload(seed=1)
        kv, bt, npg, off = (to_dev(g[k]) for k in ("kv", "bt", "num_pages", "page_offsets"))
        out = torch.empty((g["out_pages"], 128, 128), dtype=torch.uint8, device="cuda")
        fn = lambda: idx.idx_dequant_nvfp4_pages(kv, bt, npg, off, g["max_num_pages"], out)
        fn()
        ms = timer.run(fn, iters)
        byts = g["out_pages"] * (PAGE_BYTES + 16384 + 4)
        res["gather_dequant"] = {"workload": "256 requests, num_pages U[1,1344], 200,000-page pool, 2% special scales",
                                 "ms": ms, "pages_per_s": g["out_pages"] / (ms / 1e3), "gbs": byts / (ms / 1e3) / 1e9,
                                 "frac_of_hbm": byts / (ms / 1e3) / 1e9 / hbm_peak, "launches": 1}
        del kv, bt, npg, off, out, g
        torch.cuda.empty_cache()

    if "long" in args.legs:
        # long context: 16 x 500,000 tokens
        wl = W.long_context()
        q, qs, kv, bt, sl = (to_dev(wl[k]) for k in ("q", "q_scale", "kv", "bt", "seq_lens"))
        scores = torch.empty((16, 32, wl["width"]), dtype=torch.float32, device="cuda")
        out = torch.empty((16, 8, 4, 16), dtype=torch.int32, device="cuda")
        wsb = idx.idx_decode_workspace_bytes(16, 8, wl["width"])
        ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None
        fn = lambda: idx.idx_decode_step(q, qs, kv, bt, sl, 8, scores, out, ws)
        fn()
        ms = timer.run(fn, iters)
        u = decode_units(wl)
        res["long_context"] = {"workload": "16 requests x 500,000 tokens (3,906 pages), split rows merged",
                               "ms": ms, "scores_per_s": u["scores"] / (ms / 1e3),
                               "index_k_gbs": u["pages"] * PAGE_BYTES / (ms / 1e3) / 1e9,
                               "frac_of_hbm": u["pages"] * PAGE_BYTES / (ms / 1e3) / 1e9 / hbm_peak,
                               "launches": 2 + (1 if wsb else 0)}
        del q, qs, kv, bt, sl, scores, out, ws, wl
        torch.cuda.empty_cache()

    if "mtp" in args.legs:
        # multi-token scorer + top-16 per token
        m = W.mtp_workload(seed=3)
        args_d = [to_dev(m[k]) for k in ("q", "q_scale", "k", "k_scale", "bt", "num_keys", "cu_tokens")]
        T = int(m["cu_tokens"][-1])
        o = torch.empty((T, m["max_keys"]), dtype=torch.float32, device="cuda")
        idx_out = torch.empty((T, 16), dtype=torch.int32, device="cuda")
        wsb = idx.idx_workspace_bytes(T, m["max_keys"])
        ws = torch.empty(max(8, wsb) // 8, dtype=torch.int64, device="cuda") if wsb else None

        def mtp():
            idx.idx_mtp_score_fp8(*args_d, m["max_keys"], o)
            idx.idx_topk16_select(o, idx_out, workspace=ws)

        mtp()
        ms = timer.run_graph(mtp, max(iters, 100))
        ms_s = timer.run_graph(lambda: idx.idx_mtp_score_fp8(*args_d, m["max_keys"], o), max(iters, 100))
        ms_t = timer.run_graph(lambda: idx.idx_topk16_select(o, idx_out, workspace=ws), max(iters, 100))
        keys = int(m["num_keys"].sum())
        flops = 2.0 * T // len(m["num_keys"]) * 64 * 128 * keys
        kbytes = keys * (128 + 4) + T * (64 * 128 + 64 * 4) + T * m["max_keys"] * 4
        res["mtp"] = {"workload": "32 requests x 2 tokens x 64 heads, 32,768 keys each; top-16 per token",
                      "ms": ms, "ms_scorer": ms_s, "ms_topk": ms_t, "timing": "CUDA graph of 20 calls, replayed",
                      "token_keys_per_s": T * m["max_keys"] / (ms / 1e3),
                      "scorer_tflops": flops / (ms_s / 1e3) / 1e12, "scorer_gbs": kbytes / (ms_s / 1e3) / 1e9,
                      "scorer_frac_of_hbm": kbytes / (ms_s / 1e3) / 1e9 / hbm_peak, "launches": 2 + (1 if wsb else 0)}
        if fp8_peak:
            res["mtp"]["scorer_frac_of_fp8_peak"] = flops / (ms_s / 1e3) / 1e12 / fp8_peak

    if "prefill" in args.legs:
        # Q8KV8 prefill chain: gather-dequant, causal relu-weighted scores, top-16 per token
        pw = W.prefill_workload()
        kv, bt, nk, cu, q, qs = (to_dev(pw[k]) for k in ("kv", "bt", "num_keys", "cu_tokens", "q", "q_scale"))
        T, mk = int(pw["cu_tokens"][-1]), pw["max_keys"]
        sc = torch.empty((T, mk), dtype=torch.float32, device="cuda")
        out = torch.empty((T, 16), dtype=torch.int32, device="cuda")
        ws = torch.empty(idx.idx_prefill_workspace_bytes(len(pw["num_keys"]), pw["bt"].shape[1], T, mk),
                         dtype=torch.uint8, device="cuda")
        fn = lambda: idx.idx_prefill_index_step(kv, bt, nk, cu, q, qs, mk, sc, out, ws)
        fn()
        ms = timer.run(fn, iters)
        tok_keys = sum(int(pw["cu_tokens"][r + 1] - pw["cu_tokens"][r]) * int(n) for r, n in enumerate(pw["num_keys"]))
        flops = 2.0 * pw["heads"] * 128 * tok_keys
        res["prefill"] = {"workload": "chunked prefill: 4 requests x 16,384 keys, 2,048 new tokens each, 64 heads; "
                                      "top-16 per token", "ms": ms, "token_keys_per_s": tok_keys / (ms / 1e3),
                          "tflops": flops / (ms / 1e3) / 1e12, "launches": 4 + (1 if idx.idx_workspace_bytes(T, mk)
                                                                                 else 0)}
        if fp8_peak:
            res["prefill"]["frac_of_fp8_peak"] = flops / (ms / 1e3) / 1e12 / fp8_peak
        del kv, bt, nk, cu, q, qs, sc, out, ws
        torch.cuda.empty_cache()

    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip secondary workloads; short CPU baseline")
    ap.add_argument("--legs", default="fp8,gather,long,mtp,prefill,p256,fused,tiny,qlen1,sweep,mxfp8",
                    help="secondary workloads to time (comma list of fp8, gather, long, mtp, prefill, p256, tiny, qlen1, "
                         "sweep, mxfp8; empty for none)")
    args = ap.parse_args()
    args.legs = set() if args.quick else {x for x in args.legs.split(",") if x}

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from sparse_attention_indexer_nvfp4_gb300 import workloads as W

    if args.impl == "reference":
        if rank == 0:
            wl = W.batched_decode()
            run_reference(args, wl, rank)
        return

    import torch

    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        torch.cuda.set_device(local)
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    # each rank runs its own replica (different seed, same shape)
    wl = W.batched_decode(seed=replica_seed(rank))
    run_native(args, wl, rank, world, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
