#!/usr/bin/env python
"""Throughput of the QSA indexer hot path on GB300: one step = K1a q-prep over
every row and K1b K-compress over every block (one fused pass over indexQk,
qsa_index_qk_prep), then K2 block scoring of every row (one-shot), on the B=8,
S=16384 bf16 scoring workload (indexQk ~ N(0,1), contextLengths = S).  The
separate K1a and K1b entry points are timed too.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain C restatement, on every host
core) over whole steps of the same workload and reports the same metric.
With N > 1 (torchrun) every rank runs its own replica of the workload: the rows
are independent, there is no exchange step (weak scaling); rank 0 prints
rows of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexer rows/s and achieved HBM GB/s (K1a, K1b) vs 8 TB/s at 1 GB300"
UNIT = "rows/s"
WORKLOAD = "qsa indexer prefill step (fused K1a+K1b, then K2), B={B} S=16384 bf16, ctx=S, N(0,1) indexQk"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- bookkeeping

def algorithmic_bytes(ctx: np.ndarray, B: int, S: int, NB: int) -> dict:
    """Bytes each kernel must move (T = 2 bytes), from the layouts on the
    "Qsa Indexer Kernels" page: per valid row or block, its reads and writes."""
    ctx = np.clip(ctx.astype(np.int64), 0, None)
    valid_rows = int(np.minimum(ctx, S).sum())
    pad_rows = B * S - valid_rows
    positions = int(min(S, ctx.max()))
    k1a = valid_rows * 2048 + pad_rows * 1024 + positions * 256
    valid_blocks = int(np.minimum(ctx // 4, NB).sum())
    k1b = valid_blocks * (1024 + 256) + (B * NB - valid_blocks) * 256 + int(min(NB, ctx.max() // 4)) * 256
    vis_blocks = int(np.minimum(ctx // 4, NB).sum())
    k2 = valid_rows * 1024 + vis_blocks * 256 + B * S * NB * 4
    # selection reads each valid row's visible logits and writes 2051 int32 per row
    vis_logits = 0
    for c in ctx:
        t = np.arange(int(min(c, S)))
        vis_logits += int(np.minimum((t + 1) // 4, NB).sum())
    select = vis_logits * 4 + B * S * 2051 * 4
    # scoring fused with selection: q and kbar read once, outIdx written; no logits
    fused_select = valid_rows * 1024 + vis_blocks * 256 + B * S * 2051 * 4
    # causal MMA work: row t of a sequence scores floor((t+1)/4) blocks x 4 heads x 128 dims
    flops = 0
    for c in ctx:
        t = np.arange(int(min(c, S)))
        flops += int(((t + 1) // 4).sum()) * 4 * 128 * 2
    return {"k1a": k1a, "k1b": k1b, "k2": k2, "select": select, "fused_select": fused_select,
            "k2_causal_flops": flops}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk.get("bf16_tflops", 1934.3)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.proc = None
        self.device_id = device_id

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        top = max(sm)
        loaded = [s for s, p in zip(sm, pw) if p >= 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_peak_seen": top, "power_w_max": max(pw)}


def smi_device_id(local: int) -> str:
    """nvidia-smi id of torch's device `local`: its UUID if nvidia-smi accepts it."""
    import torch
    try:
        cand = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
        r = subprocess.run(["nvidia-smi", "-i", cand, "--query-gpu=uuid", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
        if r.returncode == 0 and r.stdout.strip():
            return cand
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip()]
    return ids[local] if local < len(ids) else str(local)


def k2_profiled_traffic(batch: int):
    """DRAM bytes per K2 launch from the committed ncu summary, scaled to `batch`
    sequences; None if the kernel source changed since the capture."""
    import hashlib
    import re
    prof = os.path.join(ROOT, "profiles", "k2_scores_tc_B4_S16384.md")
    src = os.path.join(ROOT, "sparse_attention_indexer_qsa_gb300", "csrc", "k2_scores_tc.cu")
    try:
        text = open(prof).read()
        want = re.search(r"source_sha256_prefix: ([0-9a-f]+)", text).group(1)
        have = hashlib.sha256(open(src, "rb").read()).hexdigest()[:len(want)]
        if want != have:
            return None
        per_b8 = int(re.search(r"traffic_bytes_per_launch_B8: (\d+)", text).group(1))
        return per_b8 * batch / 8
    except Exception:
        return None


# ------------------------------------------------------------------ oracle leg

def oracle_sample(wl, budget_s: float = 12.0, seed: int = 0, threads: int | None = None) -> dict:
    """Time the CPU oracle (as it stands; its calls release the GIL, so `threads`
    host threads run it side by side on disjoint rows) on a bounded sample of the
    workload and extrapolate to one full step: K1a on whole rows, K1b on whole
    blocks, K2 on rows spread evenly over every position t (its cost grows with t)."""
    import concurrent.futures as cf
    import oracle
    B, S, NB = wl.B, wl.S, wl.num_blocks
    dtype = wl.dtype
    if threads is None:
        threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    threads = max(1, int(threads))
    pool = cf.ThreadPoolExecutor(max_workers=threads)
    # K1a: a slab of rows of sequence 0, one contiguous share a thread
    n1 = min(S, 512 * threads)
    cuts = np.linspace(0, n1, threads + 1).astype(int)

    def k1a_part(i):
        lo, hi = int(cuts[i]), int(cuts[i + 1])
        ctx = np.array([hi - lo], np.int32)
        oracle.q_prep(dtype, wl.index_qk[:1, lo:hi], wl.cos_sin[lo:], ctx, wl.w_q, wl.eps)

    t0 = time.perf_counter()
    list(pool.map(k1a_part, range(threads)))
    k1a_per_row = (time.perf_counter() - t0) / n1
    # K1b: the blocks of that slab, one contiguous share a thread
    bcuts = (cuts // 4) * 4

    def k1b_part(i):
        lo, hi = int(bcuts[i]), int(bcuts[i + 1])
        nb = (hi - lo) // 4
        if nb:
            oracle.k_compress(dtype, wl.index_qk[:1, lo:hi], wl.cos_sin[lo:], np.array([hi - lo], np.int32),
                              wl.w_k, wl.eps, nb, 0, nb, 0)

    t0 = time.perf_counter()
    list(pool.map(k1b_part, range(threads)))
    k1b_per_block = (time.perf_counter() - t0) / max(1, n1 // 4)
    # K2: rows at random positions of sequence 0 (oracle-made qNormed/kbar), each
    # thread takes every threads-th position of one permutation until the budget
    q0 = oracle.q_prep(dtype, wl.index_qk[:1], wl.cos_sin, wl.context_lengths[:1], wl.w_q, wl.eps)[0]
    kb0 = oracle.k_compress(dtype, wl.index_qk[:1], wl.cos_sin, wl.context_lengths[:1], wl.w_k, wl.eps,
                            NB, 0, NB, 0)[0]
    ctx0 = int(wl.context_lengths[0])
    order = np.random.default_rng(seed).permutation(S)
    t_start = time.perf_counter()

    def k2_part(i):
        done = 0
        for t in order[i::threads]:
            oracle.scores_row(dtype, q0[t], kb0, int(t), ctx0)
            done += 1
            if time.perf_counter() - t_start > budget_s and done >= 8:
                break
        return done

    rows_done = sum(pool.map(k2_part, range(threads)))
    k2_wall = time.perf_counter() - t_start
    pool.shutdown()
    # the sampled positions are uniform over t, so their mean cost is the step's mean row cost
    k2_per_row = k2_wall / rows_done
    rows = B * S
    step_s = k1a_per_row * rows + k1b_per_block * B * NB + k2_per_row * rows
    return {
        "value": rows / step_s,
        "unit": UNIT,
        "cores": threads,
        "kind": "oracle",
        "sample": (f"{threads} host threads on disjoint rows: K1a on {n1} rows, K1b on {n1 // 4} blocks, K2 on "
                   f"{rows_done} rows at random positions of sequence 0 (S={S}); wall time per row/block "
                   f"scaled to one full step of {rows} rows and {B * NB} blocks"),
        "est_step_s": step_s,
    }


# ------------------------------------------------------------------ main legs

def flush_l2(buf, clean: bool = False) -> None:
    """Evict L2 before a timed launch: write `buf` (2x L2), then, when `clean`, read it
    back.  After the write alone L2 holds the flush's dirty lines, and a timed launch
    that reads new data writes them back as it evicts them (K1b at B=8, 43 MB read,
    takes 15.0 us that way against 12.3 us after the read).  The read turns L2 into
    clean lines, so the timed launch pays only for its own traffic."""
    import torch
    buf.fill_(1)
    if clean:
        buf.view(torch.int64).sum()


def decode_leg(qsa, lib, stream, K, B=64, ctx_len=16384):
    """One decode step for B sequences of length ctx_len over a paged pool
    (pre-decode, paged scores, top-k + expand), timed with CUDA events per kernel.
    The pool's V-tails hold N(0,1) bf16 values; every sequence completes a block this
    step (ctx % 4 == 0), so the pre-decode compresses a block from three K-tails."""
    import torch
    sp = stream.cuda_stream
    gen = torch.Generator(device="cuda").manual_seed(6)
    pages = (ctx_len + 127) // 128
    num_pages = B * pages
    pool = torch.randn((2 * num_pages, 128, 2, 384), device="cuda", generator=gen).to(torch.bfloat16)
    table = torch.empty((B, 2, pages), dtype=torch.int32, device="cuda")
    ids = torch.arange(num_pages, dtype=torch.int32, device="cuda").view(B, pages)
    table[:, 0] = ids
    table[:, 1] = ids + num_pages
    state = qsa.pool_state(pool, table, num_pages)
    rows = torch.randn((B, 1, 640), device="cuda", generator=gen).to(torch.bfloat16)
    cs = torch.randn((ctx_len, 64), device="cuda", generator=gen)
    ctx = torch.full((B,), ctx_len, dtype=torch.int32, device="cuda")
    wq = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    wk = (torch.randn(128, device="cuda", generator=gen) * 0.1).to(torch.bfloat16)
    q = torch.empty((B, 1, 4, 128), dtype=torch.bfloat16, device="cuda")
    maxb = (ctx_len + 3) // 4
    logits = torch.empty((B, maxb), dtype=torch.float32, device="cuda")
    out = torch.empty((B, 2051), dtype=torch.int32, device="cuda")
    split = torch.zeros((B, 2), dtype=torch.int32, device="cuda")
    import ctypes
    st_ref = ctypes.byref(state)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        rc = lib.qsa_indexer_pre_decode(qsa.QSA_BF16, q.data_ptr(), rows.data_ptr(), cs.data_ptr(), ctx.data_ptr(),
                                        wq.data_ptr(), wk.data_ptr(), 1e-6, st_ref, B, sp)
        if ev is not None:
            ev[1].record(stream)
        rc |= lib.qsa_index_scores_decode(qsa.QSA_BF16, logits.data_ptr(), q.data_ptr(), ctx.data_ptr(), st_ref, B,
                                          maxb, sp)
        if ev is not None:
            ev[2].record(stream)
        rc |= lib.qsa_topk_expand_decode(out.data_ptr(), logits.data_ptr(), ctx.data_ptr(), split.data_ptr(), 2, B,
                                         maxb, sp)
        if ev is not None:
            ev[3].record(stream)
        if rc != 0:
            raise RuntimeError(qsa.qsa_last_error())

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    # a step touches 67 MB at B=64 (V-tails and logits), which L2 would keep from one
    # step to the next: every timed step runs after an L2 flush
    l2_flush = torch.empty(2 * torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size,
                           dtype=torch.uint8, device="cuda")
    n = max(20, K)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for i in range(n):
        flush_l2(l2_flush)
        step(evs[i])
    torch.cuda.synchronize()
    ms = {name: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n))
          for j, name in enumerate(("pre_decode", "scores_decode", "topk_expand_decode"))}
    step_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][3]) for i in range(n))

    def step_on(st):
        rc = lib.qsa_indexer_pre_decode(qsa.QSA_BF16, q.data_ptr(), rows.data_ptr(), cs.data_ptr(), ctx.data_ptr(),
                                        wq.data_ptr(), wk.data_ptr(), 1e-6, st_ref, B, st)
        rc |= lib.qsa_index_scores_decode(qsa.QSA_BF16, logits.data_ptr(), q.data_ptr(), ctx.data_ptr(), st_ref, B,
                                          maxb, st)
        rc |= lib.qsa_topk_expand_decode(out.data_ptr(), logits.data_ptr(), ctx.data_ptr(), split.data_ptr(), 2, B,
                                         maxb, st)
        return rc

    # a serving loop replays the step as a graph: one step per replay, L2 flushed before each
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            if step_on(gs.cuda_stream) != 0:
                raise RuntimeError("decode step failed during capture")
    torch.cuda.current_stream().wait_stream(gs)
    # CUDA events resolve about 1 us here: a step is the mean over many replays
    n_rep = max(200, K)
    gts = []
    for _ in range(n_rep):
        flush_l2(l2_flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        e1.synchronize()
        gts.append(e0.elapsed_time(e1))
    graph_step_ms = statistics.mean(gts)

    # the same step as one launch (qsa_indexer_decode_step), timed the same way
    def fused_on(st):
        return lib.qsa_indexer_decode_step(qsa.QSA_BF16, out.data_ptr(), logits.data_ptr(), q.data_ptr(),
                                           rows.data_ptr(), cs.data_ptr(), ctx.data_ptr(), wq.data_ptr(),
                                           wk.data_ptr(), 1e-6, st_ref, split.data_ptr(), 2, B, maxb, st)

    if fused_on(sp) != 0:
        raise RuntimeError(qsa.qsa_last_error())
    torch.cuda.synchronize()
    fs = torch.cuda.Stream()
    fs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(fs):
        fgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph, stream=fs):
            if fused_on(fs.cuda_stream) != 0:
                raise RuntimeError("fused decode step failed during capture")
    torch.cuda.current_stream().wait_stream(fs)
    fts = []
    for _ in range(n_rep):
        flush_l2(l2_flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fgraph.replay()
        e1.record()
        e1.synchronize()
        fts.append(e0.elapsed_time(e1))
    fused_step_ms = statistics.mean(fts)
    fused_step_median_ms = statistics.median(fts)
    # the same replays after a clean flush (written, then read), whose lines the step evicts
    # without writing them back
    fts_clean = []
    for _ in range(n_rep):
        flush_l2(l2_flush, clean=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fgraph.replay()
        e1.record()
        e1.synchronize()
        fts_clean.append(e0.elapsed_time(e1))
    nvis = ctx_len // 4
    alg = {"pre_decode": B * (1280 + 1024 + 3 * 256 + 256 + 2 * 256),
           "scores_decode": B * (nvis * 256 + 1024 + nvis * 4),
           "topk_expand_decode": B * (nvis * 4 + 2051 * 4)}
    # prefill persistence into the same pool: K1b with the V-tail write over every
    # sequence's ctx-1 tokens (4095 complete blocks each), then the 3 raw K-tails
    iq_full = torch.randn((B, ctx_len, 640), device="cuda", generator=gen).to(torch.bfloat16)
    kb_dense = torch.empty((B, maxb, 128), dtype=torch.bfloat16, device="cuda")
    pctx = torch.full((B,), ctx_len - 1, dtype=torch.int32, device="cuda")
    cs_full = torch.randn((ctx_len, 64), device="cuda", generator=gen)

    def compress_paged(st):
        return lib.qsa_index_k_compress_paged(qsa.QSA_BF16, kb_dense.data_ptr(), iq_full.data_ptr(),
                                              cs_full.data_ptr(), pctx.data_ptr(), wk.data_ptr(), 1e-6, st_ref,
                                              B, ctx_len, maxb, 0, maxb, 0, st)

    def raw_tails(st):
        return lib.qsa_raw_k_tail_write_prefill(qsa.QSA_BF16, iq_full.data_ptr(), pctx.data_ptr(), st_ref, B,
                                                ctx_len, st)

    for name, fn in (("k_compress_paged", compress_paged), ("raw_k_tail_write_prefill", raw_tails)):
        for _ in range(3):
            if fn(sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())
        pts = []
        for _ in range(20):
            flush_l2(l2_flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(sp)
            e1.record(stream)
            e1.synchronize()
            pts.append(e0.elapsed_time(e1))
        ms[name] = statistics.median(pts)
    # the same-size yardstick of the paged scores: a plain gathering kernel reading the
    # same V-tails (256 B each at the pool's 6 KB block pitch; the V pages are consecutive
    # here) and writing 4 B a block, timed like the kernels above
    if ctx_len % 128 == 0:
        blk_pitch = 4 * 2 * 384 * 2
        v_first = num_pages * 128 * 2 * 384 * 2 + 256 * 2
        y_out = torch.empty(B * nvis, dtype=torch.int32, device="cuda")

        def yard(st):
            return lib.qsa_testing_gather_yardstick(y_out.data_ptr(), pool.data_ptr(), B * nvis, blk_pitch, v_first,
                                                    256, st)

        for _ in range(3):
            if yard(sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())
        yts = []
        for _ in range(n):
            flush_l2(l2_flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            yard(sp)
            e1.record(stream)
            e1.synchronize()
            yts.append(e0.elapsed_time(e1))
        ms["yardstick_scores_decode"] = statistics.mean(yts)
        alg["yardstick_scores_decode"] = B * nvis * (256 + 4)
        del y_out
    valid_blocks = B * ((ctx_len - 1) // 4)
    alg["k_compress_paged"] = valid_blocks * (1024 + 256 + 256) + ((ctx_len - 1) // 4) * 256
    alg["raw_k_tail_write_prefill"] = B * ((ctx_len - 1) % 4) * 512
    del iq_full, kb_dense, l2_flush
    hbm_peak, _, _ = load_peaks()
    kernels = {k: {"ms": ms[k], "alg_bytes": alg[k], "gbs": alg[k] / (ms[k] * 1e-3) / 1e9,
                   "frac_of_measured_hbm": alg[k] / (ms[k] * 1e-3) / 1e9 / hbm_peak} for k in ms}
    if "yardstick_scores_decode" in kernels:
        kernels["scores_decode"]["frac_of_yardstick"] = (kernels["scores_decode"]["gbs"] /
                                                         kernels["yardstick_scores_decode"]["gbs"])
    del pool
    torch.cuda.empty_cache()
    return {"workload": f"decode step, B={B} sequences at ctx={ctx_len}, paged pool (128-token pages), bf16",
            "ms_per_step": fused_step_ms, "ms_per_step_median": fused_step_median_ms,
            "ms_per_step_after_clean_flush": statistics.mean(fts_clean),
            "tokens_per_s": B / (fused_step_ms * 1e-3),
            "ms_per_step_three_launches": graph_step_ms, "ms_per_step_eager": step_ms, "kernels": kernels,
            "timed": ("step: qsa_indexer_decode_step (one launch) as a CUDA graph replayed after an L2 flush "
                      "(a 2x-L2 buffer written; ms_per_step_after_clean_flush: written, then read, so that "
                      "the step evicts clean lines), "
                      f"mean of {n_rep} replays (CUDA events resolve about 1 us; ms_per_step_median: their median); "
                      "ms_per_step_three_launches: the three separate launches timed the same way; "
                      "kernels: CUDA events "
                      "per kernel over eagerly launched steps, each after an L2 flush; k_compress_paged and "
                      "raw_k_tail_write_prefill: the prefill persistence of the same B sequences (ctx-1 tokens "
                      "each) into the pool, one launch after an L2 flush, median; yardstick_scores_decode: "
                      "qsa_testing_gather_yardstick reading the same V-tails and writing 4 B a block, timed "
                      "like scores_decode")}


def _graph_ms(torch, launches, reps: int = 10) -> float:
    """Median over `reps` replays of a CUDA graph holding `launches` (callables taking a
    stream handle), divided by the number of launches: per-launch device time."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for f in launches[:2]:                # first-call set-up outside the capture
            if f(s.cuda_stream) != 0:
                raise RuntimeError("launch failed before capture")
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for f in launches:
                if f(s.cuda_stream) != 0:
                    raise RuntimeError("launch failed during capture")
    torch.cuda.current_stream().wait_stream(s)
    times = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times) / len(launches)


def _k1_launchers(qsa, lib, dt, bufs, ctx, cs, wq, wk, eps, B, S, NB):
    """(K1a, K1b, fused K1) launchers over buffer set i: (iq, qn, kb) views."""
    def k1a(i):
        iq, qn, _ = bufs(i)
        return lambda st: lib.qsa_index_q_prep(dt, qn, iq, cs, ctx, wq, eps, B, S, st)

    def k1b(i):
        iq, _, kb = bufs(i)
        return lambda st: lib.qsa_index_k_compress(dt, kb, iq, cs, ctx, wk, eps, B, S, NB, 0, NB, 0, st)

    def fused(i):
        iq, qn, kb = bufs(i)
        return lambda st: lib.qsa_index_qk_prep(dt, qn, kb, iq, cs, ctx, wq, wk, eps, B, S, NB, st)
    return {"k1a": k1a, "k1b": k1b, "k1_fused": fused}


def _k1_touched(B: int, S: int, NB: int) -> dict:
    """Bytes each K1 kernel touches (the cache-line footprint that L2 could keep between
    launches): K1a the q part of every row and qNormed, K1b the 256-byte K slices and
    kbar, the fused pass whole rows, qNormed and kbar."""
    return {"k1a": B * S * 2048 + S * 256, "k1b": B * S * 256 + B * NB * 256 + S * 64,
            "k1_fused": B * S * 2304 + B * NB * 256 + S * 256}


K1_MAX_COPIES = 2048


def k1_configs_leg(qsa, lib, hbm_peak: float, names=None, sweep: bool = True) -> dict:
    """K1a, K1b and the fused K1 on the small configurations (tiny, batched bf16/fp16,
    long, decode-parity full compress) and a size sweep of B*S from 2^16 to 2^22 rows.
    Each timed launch of a kernel uses its own copy of the inputs and outputs, cycling
    through enough copies that the kernel's footprint over a cycle exceeds twice the L2
    size (at most K1_MAX_COPIES: the tiny configuration stays partly L2-warm); the
    launches run back to back from a CUDA graph, median of 10 replays."""
    import torch
    import workloads
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size

    def copies(touched: int) -> int:
        return int(min(K1_MAX_COPIES, max(1, -(-2 * l2 // touched))))

    def measure(B, S, NB, dt, ctx_np, make_sets, cs, wq, wk, eps):
        touched = _k1_touched(B, S, NB)
        n_sets = {k: copies(v) for k, v in touched.items()}
        bufs = make_sets(max(n_sets.values()))
        ctx = torch.from_numpy(np.ascontiguousarray(ctx_np, np.int32)).cuda()
        L = _k1_launchers(qsa, lib, dt, bufs, ctx.data_ptr(), cs.data_ptr(), wq.data_ptr(), wk.data_ptr(), eps,
                          B, S, NB)
        ab = algorithmic_bytes(ctx_np, B, S, NB)
        ab["k1_fused"] = ab["k1a"] + ab["k1b"]
        # the same-size yardstick: a plain streaming kernel moving each K1 kernel's byte pattern
        # (K1a: 1024 B in and out per row; K1b: 4 x 256 B in at a 1280 B pitch, 256 B out per
        # block) over every row / block, through the same copies and the same graph harness
        units_a, units_b = B * S, B * (S // 4)

        def yard(kind):
            def mk(i):
                iq, qn, kb = bufs(i)
                if kind == "k1a":
                    return lambda st: lib.qsa_testing_stream_yardstick(qn, iq, units_a, 1, 1280, 1280, 0, 1024, st)
                return lambda st: lib.qsa_testing_stream_yardstick(kb, iq, units_b, 4, 1280, 5120, 1024, 256, st)
            return mk
        L["yardstick_k1a"], L["yardstick_k1b"] = yard("k1a"), yard("k1b")
        n_sets["yardstick_k1a"], n_sets["yardstick_k1b"] = n_sets["k1a"], n_sets["k1b"]
        touched["yardstick_k1a"], touched["yardstick_k1b"] = touched["k1a"], touched["k1b"]
        ab["yardstick_k1a"], ab["yardstick_k1b"] = units_a * 2048, units_b * (1024 + 256)
        out = {}
        for name, mk in L.items():
            launches = [mk(i) for i in range(n_sets[name])]
            if len(launches) == 1:
                launches = launches * 2  # footprint above 2x L2: the second launch is cold too
            ms = _graph_ms(torch, launches)
            gbs = ab[name] / (ms * 1e-3) / 1e9
            out[name] = {"us": ms * 1e3, "alg_bytes": ab[name], "gbs": gbs, "frac_of_measured_hbm": gbs / hbm_peak,
                         "copies": n_sets[name], "touched_bytes": touched[name]}
        for name in ("k1a", "k1b"):
            out[name]["frac_of_yardstick"] = out[name]["gbs"] / out["yardstick_" + name]["gbs"]
            # the yardstick's time over the kernel's.  The yardstick moves every row's / block's
            # q or K bytes, more than the kernel where rows or blocks lie past the context, and
            # reads no rope rows: where contexts are short the GB/s ratio above understates the
            # kernel, and this one is the fairer
            out[name]["time_vs_yardstick"] = out["yardstick_" + name]["us"] / out[name]["us"]
        del bufs
        return out

    res = {"configs": {}, "sweep": []}
    cfgs = {"tiny": lambda: workloads.tiny(), "batched_bf16": lambda: workloads.batched("bf16"),
            "batched_fp16": lambda: workloads.batched("fp16"), "long": lambda: workloads.long_prefill(),
            "decode_parity_full_compress": lambda: workloads.decode_parity()}
    for name, make_wl in cfgs.items():
        if names is not None and name not in names:
            continue
        wl = make_wl()
        B, S, NB = wl.B, wl.S, wl.num_blocks
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                         else np.ascontiguousarray(a)).cuda()

        def make(n, wl=wl, B=B, S=S, NB=NB):
            iq0 = torch.from_numpy(np.ascontiguousarray(wl.index_qk).view(np.int16)).cuda()
            iq = iq0.unsqueeze(0).repeat(n, 1, 1, 1).contiguous()
            qn = torch.empty((n, B, S, 512), dtype=torch.int16, device="cuda")
            kb = torch.empty((n, B, NB, 128), dtype=torch.int16, device="cuda")
            return lambda i: (iq[i].data_ptr(), qn[i].data_ptr(), kb[i].data_ptr())
        dt = qsa.QSA_BF16 if wl.dtype == "bf16" else qsa.QSA_F16
        r = measure(B, S, NB, dt, wl.context_lengths, make, dev(wl.cos_sin), dev(wl.w_q), dev(wl.w_k), wl.eps)
        r["shape"] = {"B": B, "S": S, "num_blocks": NB, "dtype": wl.dtype}
        res["configs"][name] = r
        torch.cuda.empty_cache()
    if not sweep:
        return res
    # sweep: S = 16384, ctx = S, B = 4 .. 256; inputs drawn on the device (seeded), bf16
    S = 16384
    NB = S // 4
    cs = torch.from_numpy(workloads.cos_sin_table(S)).cuda()
    rng = np.random.default_rng(5)
    wq = torch.from_numpy(workloads.gamma(rng, "bf16").view(np.int16)).cuda()
    wk = torch.from_numpy(workloads.gamma(rng, "bf16").view(np.int16)).cuda()
    gen = torch.Generator(device="cuda").manual_seed(5)
    for B in (4, 8, 16, 32, 64, 128, 256):
        def make(n, B=B):
            iq = torch.empty((n, B, S, 640), dtype=torch.int16, device="cuda")
            for i in range(n):
                iq[i].copy_(torch.randn((B, S, 640), generator=gen, device="cuda").to(torch.bfloat16)
                            .view(torch.int16))
            qn = torch.empty((n, B, S, 512), dtype=torch.int16, device="cuda")
            kb = torch.empty((n, B, NB, 128), dtype=torch.int16, device="cuda")
            return lambda i: (iq[i].data_ptr(), qn[i].data_ptr(), kb[i].data_ptr())
        r = measure(B, S, NB, qsa.QSA_BF16, np.full(B, S, np.int32), make, cs, wq, wk, 1e-6)
        row = {"rows": B * S, "B": B, "S": S}
        for name in ("k1a", "k1b", "k1_fused", "yardstick_k1a", "yardstick_k1b"):
            row[name + "_gbs"] = r[name]["gbs"]
            row[name + "_us"] = r[name]["us"]
            row[name + "_copies"] = r[name]["copies"]
        res["sweep"].append(row)
        torch.cuda.empty_cache()
    res["how"] = ("per-launch device time from a CUDA graph of back-to-back launches (median of 10 replays); each "
                  "kernel cycles through copies of its inputs and outputs whose footprint exceeds 2x L2 (at most "
                  f"{K1_MAX_COPIES} copies); the sweep's inputs are drawn on the device (torch generator, seed 5), "
                  "S=16384, ctx=S, bf16; yardstick_k1a / yardstick_k1b: qsa_testing_stream_yardstick moving "
                  "the K1a / K1b byte pattern over every row / block in the same harness")
    res["l2_bytes"] = l2
    return res


def prefill_select_leg(qsa, lib, stream, K, B=8):
    """The prefill selection of the scoring workload (B sequences of 16384 tokens, ctx = S)
    both ways: qsa_index_scores + qsa_index_topk_expand, and the fused
    qsa_index_scores_topk_expand; K launches of each after 3 warm-up launches."""
    import torch
    wl = rank_workload(B, 0)
    S, NB = wl.S, wl.num_blocks
    rows = B * S
    host = PrefillStepGpu.host
    iq = host(wl.index_qk).cuda().view(torch.bfloat16)
    cs, ctx = host(wl.cos_sin).cuda(), host(wl.context_lengths).cuda()
    wq, wk = host(wl.w_q).cuda().view(torch.bfloat16), host(wl.w_k).cuda().view(torch.bfloat16)
    qn = torch.empty((B, S, 4, 128), dtype=torch.bfloat16, device="cuda")
    kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
    sp = stream.cuda_stream
    qsa.qsa_index_qk_prep(qn, kb, iq, cs, ctx, wq, wk, wl.eps, B, S, NB, stream=sp)
    logits = torch.empty((rows, NB), dtype=torch.float32, device="cuda")
    out2 = torch.empty((rows, 2051), dtype=torch.int32, device="cuda")
    out1 = torch.empty_like(out2)

    def two():
        qsa.qsa_index_scores(logits, qn, kb, ctx, B, S, NB, 0, rows, stream=sp)
        qsa.qsa_index_topk_expand(out2, logits, ctx, B, S, NB, 0, rows, stream=sp)

    def fused():
        qsa.qsa_index_scores_topk_expand(out1, qn, kb, ctx, B, S, NB, 0, rows, stream=sp)

    def ms(fn):
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / K

    res = {"B": B, "S": S, "num_blocks": NB, "fused_ms": ms(fused), "two_calls_ms": ms(two)}
    torch.cuda.synchronize()
    res["outidx_equal"] = bool(torch.equal(out1, out2))
    res["device_fault_flags"] = qsa.qsa_device_fault_flags()
    return res


# ----------------------------------------------------------------- ranks (N > 1)

def rank_barrier(world: int) -> None:
    """All ranks meet (gloo; no data-path collective exists: rows are independent)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_of(x: float, world: int) -> float:
    """The slowest rank's time: whole-job time of N replicas run side by side."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rows_per_s(rows_per_rank: int, ms_max: float, world: int) -> float:
    """Weak scaling: every rank processed its own rows_per_rank in at most ms_max."""
    return world * rows_per_rank / (ms_max * 1e-3)


def rank_seed(rank: int) -> int:
    """Each rank draws its own replica of the scoring workload: seed 4 on rank 0."""
    return 4 + rank


def rank_workload(batch: int, rank: int):
    import workloads
    return workloads.scoring("bf16", seed=rank_seed(rank), B=batch, full_context=True)


L2_NOTE = ("inputs larger than L2 (indexQk 168 MB, qNormed 134 MB) and each step writes "
           "2.15 GB of logits, which evicts L2 between steps")


def step_config(B: int, S: int, NB: int) -> dict:
    """The workload both arms run, printed identically by both."""
    return {"workload": WORKLOAD.format(B=B), "B": B, "S": S, "num_blocks": NB, "rows_per_step": B * S,
            "k2_row_chunk": B * S, "l2": L2_NOTE}


def base_line(args, world: int, wl, ms_step: float) -> dict:
    rows = wl.B * wl.S
    return {"metric": METRIC, "value": whole_job_rows_per_s(rows, ms_step, world), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": step_config(wl.B, wl.S, wl.num_blocks)}


def run_steps(args, rank: int, world: int, make_impl):
    """One rank of a bench run: this rank's seeded workload, W warm-up steps, K timed
    steps between barriers on the impl's own clock, the slowest rank's time, and ONE
    JSON line printed by rank 0 (returned there; None on the other ranks).

    make_impl(args, wl, rank, world) supplies the step: PrefillStepGpu for the GPU
    arm.  It provides step(), sync(), check(), sampler() (a context whose value has
    summary()), time_steps(K) -> ms for K steps, after_timed(args, world) (work that
    runs inside the clock sampling) and report(...) -> the line's other keys."""
    wl = rank_workload(args.batch, rank)
    impl = make_impl(args, wl, rank, world)
    for _ in range(args.warmup):
        impl.step()
    impl.sync()
    impl.check()
    with impl.sampler() as clk:
        rank_barrier(world)
        impl.sync()
        ms_total = impl.time_steps(args.steps)
        impl.sync()
        rank_barrier(world)
        after = impl.after_timed(args, world)
    ms_step = max_over_ranks_of(ms_total / args.steps, world)
    extra = impl.report(args, world, ms_step, after, clk.summary())
    if rank != 0:
        return None
    line = base_line(args, world, wl, ms_step)
    line.update(extra)
    print(json.dumps(line), flush=True)
    return line


def oracle_full_step(wl, pool, threads: int, logits: np.ndarray, piece: int = 256) -> None:
    """One whole step of the CPU oracle on `threads` host threads: K1a over every row,
    K1b over every block (both in 512-row slabs of each sequence), then K2 over every
    row in `piece`-row pieces into `logits` [B*S, NB].  Its C calls release the GIL."""
    import oracle
    B, S, NB = wl.B, wl.S, wl.num_blocks
    dtype = wl.dtype
    qn = np.empty((B, S, 4, 128), np.uint16)
    kb = np.zeros((B, NB, 128), np.uint16)
    slab = 512

    def k1(job):
        b, lo = job
        hi = min(S, lo + slab)
        c = np.array([min(max(int(wl.context_lengths[b]) - lo, 0), hi - lo)], np.int32)
        iq = wl.index_qk[b:b + 1, lo:hi]
        qn[b, lo:hi] = oracle.q_prep(dtype, iq, wl.cos_sin[lo:], c, wl.w_q, wl.eps)[0]
        nb = (hi - lo) // 4
        kb[b, lo // 4:lo // 4 + nb] = oracle.k_compress(dtype, iq, wl.cos_sin[lo:], c, wl.w_k, wl.eps,
                                                        nb, 0, nb, 0)[0]

    list(pool.map(k1, [(b, lo) for b in range(B) for lo in range(0, S, slab)]))
    rows = B * S

    def k2(r0):
        n = min(piece, rows - r0)
        logits[r0:r0 + n] = oracle.scores(dtype, qn, kb, wl.context_lengths, r0, n)

    list(pool.map(k2, range(0, rows, piece)))


def run_reference(args, rank: int) -> None:
    """The reference arm: the CPU oracle as it stands, on all host cores, timed over
    whole steps of the workload when W + K of them fit the time budget, otherwise on a
    bounded sample of each step scaled to a full step (the line then says so)."""
    if rank != 0:
        return
    import concurrent.futures as cf
    wl = rank_workload(args.batch, 0)
    B, S, NB = wl.B, wl.S, wl.num_blocks
    rows = B * S
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    budget_s = 300.0
    probe = oracle_sample(wl, budget_s=2.0, seed=0, threads=threads)
    whole = probe["est_step_s"] * (args.steps + args.warmup) <= budget_s
    vals = []
    res = None
    if whole:
        pool = cf.ThreadPoolExecutor(max_workers=threads)
        logits = np.empty((rows, NB), np.float32)
        for _ in range(args.warmup):
            oracle_full_step(wl, pool, threads, logits)
        for _ in range(args.steps):
            a = time.perf_counter()
            oracle_full_step(wl, pool, threads, logits)
            vals.append(rows / (time.perf_counter() - a))
        pool.shutdown()
        sample = (f"whole steps: K1a over all {rows} rows, K1b over all {B * NB} blocks and K2 over all "
                  f"{rows} rows, on {threads} host threads (disjoint rows); the median of {args.steps} "
                  f"timed steps after {args.warmup} warm-up steps")
    else:
        budget = max(1.0, budget_s / max(1, args.steps + args.warmup))
        for i in range(args.warmup):
            oracle_sample(wl, budget_s=budget, seed=i, threads=threads)
        for i in range(args.steps):
            res = oracle_sample(wl, budget_s=budget, seed=1000 + i, threads=threads)
            vals.append(res["value"])
        sample = res["sample"]
    value = statistics.median(vals)
    line = base_line(args, 1, wl, 1000.0 * rows / value)
    line.update({
        "impl": "reference", "n_gpus": args.gpus, "dtype": "f32",
        "extrapolated": not whole,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    })
    print(json.dumps(line), flush=True)


class PrefillStepGpu:
    """The GPU arm's step for run_steps: fused K1 (qsa_index_qk_prep), then K2 over every
    row, on this rank's workload resident in HBM; plus the legs reported beside it."""

    def __init__(self, args, wl, rank: int, world: int):
        import torch
        import sparse_attention_indexer_qsa_gb300 as qsa
        self.torch, self.qsa, self.wl, self.rank = torch, qsa, wl, rank
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(self.local)
        B, S, NB = wl.B, wl.S, wl.num_blocks
        self.B, self.S, self.NB, self.rows = B, S, NB, B * S
        dev = lambda a: self.host(a).cuda()
        self.iq = dev(wl.index_qk).view(torch.bfloat16)
        self.cs, self.ctx = dev(wl.cos_sin), dev(wl.context_lengths)
        self.wq, self.wk = dev(wl.w_q).view(torch.bfloat16), dev(wl.w_k).view(torch.bfloat16)
        self.qn = torch.empty((B, S, 4, 128), dtype=torch.bfloat16, device="cuda")
        self.kb = torch.empty((B, NB, 128), dtype=torch.bfloat16, device="cuda")
        self.logits = torch.empty((self.rows, NB), dtype=torch.float32, device="cuda")
        self.stream = torch.cuda.current_stream()
        self.sp = self.stream.cuda_stream
        self.lib = qsa.load()
        self.eps = wl.eps
        self.evs = []

    @staticmethod
    def host(a):
        import torch
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)

    def step(self, ev=None):
        # K1a + K1b (prefill range) in one pass over indexQk, then K2 over every row
        lib, qsa, stream = self.lib, self.qsa, self.stream
        if ev is not None:
            ev[0].record(stream)
        st = lib.qsa_index_qk_prep(qsa.QSA_BF16, self.qn.data_ptr(), self.kb.data_ptr(), self.iq.data_ptr(),
                                   self.cs.data_ptr(), self.ctx.data_ptr(), self.wq.data_ptr(), self.wk.data_ptr(),
                                   self.eps, self.B, self.S, self.NB, self.sp)
        if ev is not None:
            ev[1].record(stream)
        st |= lib.qsa_index_scores(qsa.QSA_BF16, self.logits.data_ptr(), self.qn.data_ptr(), self.kb.data_ptr(),
                                   self.ctx.data_ptr(), self.B, self.S, self.NB, 0, self.rows, self.sp)
        if ev is not None:
            ev[2].record(stream)
        if st != 0:
            raise RuntimeError(qsa.qsa_last_error())

    def sync(self):
        self.torch.cuda.synchronize()

    def check(self):
        assert self.qsa.qsa_device_fault_flags() == 0

    def sampler(self):
        return ClockSampler(smi_device_id(self.local))

    def time_steps(self, K: int) -> float:
        """K steps on the device clock (CUDA events on the launching stream), then K more
        with per-kernel events inside each step.  An event between K1 and K2 makes K2
        wait for it instead of launching as K1's programmatic dependent (about 9 us a
        step), so the K timed steps carry no event between their kernels; the per-kernel
        times come from the second pass, which runs right after them."""
        torch = self.torch
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(K):
            self.step()
        end.record(self.stream)
        end.synchronize()
        self.evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for i in range(K):
            self.step(self.evs[i])
        self.evs[-1][-1].synchronize()
        return start.elapsed_time(end)

    def after_timed(self, args, world: int) -> dict:
        """End-to-end through the public API with host buffers: every step copies its
        inputs in from pinned memory and its logits out to pinned memory.  The copies
        run on their own streams and overlap compute: step n+1's inputs go in while
        step n's logits come out, and K2 runs in row chunks whose logits are copied out
        as soon as each chunk is done (logits double-buffered)."""
        torch, qsa, wl = self.torch, self.qsa, self.wl
        B, S, NB, rows, stream, sp, eps = self.B, self.S, self.NB, self.rows, self.stream, self.sp, self.eps
        qn, kb = self.qn, self.kb
        K_e2e = 0 if args.no_e2e else max(3, min(args.steps, 20))
        host = self.host
        h_in = [host(wl.index_qk).pin_memory(), host(wl.cos_sin).pin_memory(),
                host(wl.context_lengths).pin_memory(), host(wl.w_q).pin_memory(), host(wl.w_k).pin_memory()]
        d_in = [torch.empty_like(h, device="cuda") for h in h_in]
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        n_chunks = B
        chunk = rows // n_chunks
        h_logits = [torch.empty((rows, NB), dtype=torch.float32).pin_memory() for _ in range(2)] if K_e2e else []
        d_logits = [self.logits, torch.empty_like(self.logits)] if K_e2e else [self.logits]
        d2h = rows * NB * 4
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        state = {"ev_k1": None}
        ev_out = {}

        def e2e_step(n):
            d_iq, d_cs, d_ctx, d_wq, d_wk = d_in
            with torch.cuda.stream(s_in):
                if state["ev_k1"] is not None:
                    s_in.wait_event(state["ev_k1"])   # the previous step has consumed the inputs
                for h, d in zip(h_in, d_in):
                    d.copy_(h, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            qsa.qsa_index_qk_prep(qn, kb, d_iq, d_cs, d_ctx, d_wq, d_wk, eps, B, S, NB, stream=sp, dtype="bf16")
            state["ev_k1"] = torch.cuda.Event()
            state["ev_k1"].record(stream)
            buf = d_logits[n % 2]
            for c in range(n_chunks):
                prev = ev_out.get((n - 2, c))
                if prev is not None:
                    stream.wait_event(prev)           # this logits chunk has been copied out
                qsa.qsa_index_scores(buf[c * chunk:(c + 1) * chunk], qn, kb, d_ctx, B, S, NB, c * chunk, chunk,
                                     stream=sp, dtype="bf16")
                ev_c = torch.cuda.Event()
                ev_c.record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_c)
                    h_logits[n % 2][c * chunk:(c + 1) * chunk].copy_(buf[c * chunk:(c + 1) * chunk],
                                                                     non_blocking=True)
                    ev_o = torch.cuda.Event()
                    ev_o.record(s_out)
                    ev_out[(n, c)] = ev_o

        if K_e2e:
            e2e_step(-2)
            torch.cuda.synchronize()
        # three timed blocks of K_e2e steps; the median block is reported (the host link is
        # shared with the rest of the machine, and one disturbed block should not decide)
        blocks = []
        for _ in range(3 if K_e2e else 0):
            ev_out.clear()
            state["ev_k1"] = None
            rank_barrier(world)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for n in range(K_e2e):
                e2e_step(n)
            stream.wait_stream(s_out)
            e1.record(stream)
            e1.synchronize()
            rank_barrier(world)
            blocks.append(e0.elapsed_time(e1) / K_e2e)
        ms_e2e = sorted(blocks)[1] if K_e2e else float("nan")
        return {"ms_e2e": ms_e2e, "K_e2e": K_e2e, "blocks": blocks, "h2d": h2d, "d2h": d2h}

    def report(self, args, world: int, ms_step: float, after: dict, clocks: dict) -> dict:
        torch, qsa, lib, wl = self.torch, self.qsa, self.lib, self.wl
        B, S, NB, rows, stream, sp, eps = self.B, self.S, self.NB, self.rows, self.stream, self.sp, self.eps
        qn, kb, iq, cs, ctx, wq, wk, logits = (self.qn, self.kb, self.iq, self.cs, self.ctx, self.wq, self.wk,
                                               self.logits)
        K = args.steps
        torch.cuda.synchronize()

        def k1a_only():
            if lib.qsa_index_q_prep(qsa.QSA_BF16, qn.data_ptr(), iq.data_ptr(), cs.data_ptr(), ctx.data_ptr(),
                                    wq.data_ptr(), eps, B, S, sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())

        def k1b_only():
            if lib.qsa_index_k_compress(qsa.QSA_BF16, kb.data_ptr(), iq.data_ptr(), cs.data_ptr(), ctx.data_ptr(),
                                        wk.data_ptr(), eps, B, S, NB, 0, NB, 0, sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())

        def loop_ms(fn, n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            for _ in range(3):
                fn()
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / n

        # the separate K1a and K1b entry points, each back to back over the same workload.
        # K1b alone touches 42 MB (the K slices and kbar), which L2 would keep across
        # back-to-back launches: each standalone launch runs after an L2 flush instead
        l2_flush = torch.empty(2 * torch.cuda.get_device_properties(self.local).L2_cache_size, dtype=torch.uint8,
                               device="cuda")

        def cold_ms(fn, n, clean=False):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(n):
                flush_l2(l2_flush, clean)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            return statistics.median(ts)

        ms_k1a = cold_ms(k1a_only, max(K // 4, 20))
        ms_k1b = cold_ms(k1b_only, max(K // 4, 20))
        ms_k1a_clean = cold_ms(k1a_only, max(K // 4, 20), clean=True)
        ms_k1b_clean = cold_ms(k1b_only, max(K // 4, 20), clean=True)
        # prefill selection on the step's logits (top-512 blocks per row -> 2051 token ids)
        out_idx = torch.empty((rows, 2051), dtype=torch.int32, device="cuda")

        def select_only():
            if lib.qsa_index_topk_expand(out_idx.data_ptr(), logits.data_ptr(), ctx.data_ptr(), B, S, NB, 0, rows,
                                         sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())

        ms_sel = loop_ms(select_only, max(10, K // 10))

        # K2 over the same rows in 8192-row chunks (rowStart, numRows), as a caller that bounds
        # its logits buffer would call it: all chunks back to back, per step
        chunk_rows = 8192

        def k2_chunked():
            for r0 in range(0, rows, chunk_rows):
                n = min(chunk_rows, rows - r0)
                if lib.qsa_index_scores(qsa.QSA_BF16, logits.data_ptr() + r0 * NB * 4, qn.data_ptr(), kb.data_ptr(),
                                        ctx.data_ptr(), B, S, NB, r0, n, sp) != 0:
                    raise RuntimeError(qsa.qsa_last_error())

        ms_k2_chunked = loop_ms(k2_chunked, max(10, K // 10))

        # the whole prefill indexer pipeline a caller runs: K1 (one pass), K2, then the top-512
        # selection with expand, back to back on the stream
        def pipeline():
            self.step()
            select_only()

        ms_pipeline = loop_ms(pipeline, max(10, K // 10))

        # K2 fused with the selection (no logits written): alone, and as the pipeline
        # K1 (one pass) then the fused call; its outIdx must equal the two calls'
        out_fused = torch.empty_like(out_idx)

        def fused_only():
            if lib.qsa_index_scores_topk_expand(qsa.QSA_BF16, out_fused.data_ptr(), qn.data_ptr(), kb.data_ptr(),
                                                ctx.data_ptr(), B, S, NB, 0, rows, sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())

        def pipeline_fused():
            if lib.qsa_index_qk_prep(qsa.QSA_BF16, qn.data_ptr(), kb.data_ptr(), iq.data_ptr(), cs.data_ptr(),
                                     ctx.data_ptr(), wq.data_ptr(), wk.data_ptr(), eps, B, S, NB, sp) != 0:
                raise RuntimeError(qsa.qsa_last_error())
            fused_only()

        ms_fused = loop_ms(fused_only, max(10, K // 10))
        ms_pipeline_fused = loop_ms(pipeline_fused, max(10, K // 10))
        pipeline()
        torch.cuda.synchronize()
        fused_equal = bool(torch.equal(out_fused, out_idx))
        decode = None if args.no_decode else decode_leg(qsa, lib, stream, K, B=args.decode_batch)
        k1_small = None if args.no_sweep or self.rank != 0 else k1_configs_leg(qsa, lib, load_peaks()[0])
        torch.cuda.synchronize()
        faults = qsa.qsa_device_fault_flags()

        ms_e2e = max_over_ranks_of(after["ms_e2e"], world)
        evs = self.evs
        per_kernel = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                      for j, n in enumerate(("k1_fused", "k2"))}
        per_kernel["k1a"] = ms_k1a
        per_kernel["k1b"] = ms_k1b
        per_kernel["select"] = ms_sel
        if self.rank != 0:
            return {}

        hbm_peak, tf_peak, peak_src = load_peaks()
        ab = algorithmic_bytes(wl.context_lengths, B, S, NB)
        ab["k1_fused"] = ab["k1a"] + ab["k1b"]
        kernels = {}
        for n in ("k1_fused", "k2", "k1a", "k1b", "select"):
            gbs = ab[n] / (per_kernel[n] * 1e-3) / 1e9
            kernels[n] = {"ms": per_kernel[n], "alg_bytes": ab[n], "gbs": gbs,
                          "frac_of_measured_hbm": gbs / hbm_peak, "frac_of_8tbs": gbs / NOMINAL_HBM_GBS}
        kernels["k1_fused"]["rows_per_s"] = rows / (per_kernel["k1_fused"] * 1e-3)
        kernels["k1_fused"]["timed"] = ("inside the step (CUDA events around the launch, over a second pass of "
                                         "the timed steps run right after them)")
        kernels["k2"]["timed"] = ("inside the step (CUDA events around the launch, over a second pass of the "
                                  "timed steps run right after them: an event between K1 and K2 keeps K2 from "
                                  "launching during K1's tail, so the timed steps carry none)")
        for n, ms_clean in (("k1a", ms_k1a_clean), ("k1b", ms_k1b_clean)):
            kernels[n]["timed"] = ("separate entry point after the step loop; each launch after an L2 flush (a "
                                   "2x-L2 buffer written), median; ms_after_clean_flush / gbs_after_clean_flush: "
                                   "after the buffer is written, then read, so that the launch evicts clean lines "
                                   "instead of writing the flush's dirty ones back")
            kernels[n]["ms_after_clean_flush"] = ms_clean
            kernels[n]["gbs_after_clean_flush"] = ab[n] / (ms_clean * 1e-3) / 1e9
        kernels["select"]["timed"] = ("separate entry point, back-to-back launches after the step loop "
                                      "(1 GB of logits)")
        kernels["select"]["rows_per_s"] = rows / (per_kernel["select"] * 1e-3)
        kernels["k1a"]["rows_per_s"] = rows / (per_kernel["k1a"] * 1e-3)
        kernels["k1b"]["blocks_per_s"] = B * NB / (per_kernel["k1b"] * 1e-3)
        kernels["k1b"]["token_rows_per_s"] = 4 * B * NB / (per_kernel["k1b"] * 1e-3)
        kernels["k2"]["rows_per_s"] = rows / (per_kernel["k2"] * 1e-3)
        kernels["k2"]["causal_tflops"] = ab["k2_causal_flops"] / (per_kernel["k2"] * 1e-3) / 1e12
        kernels["k2"]["frac_of_measured_bf16_peak"] = kernels["k2"]["causal_tflops"] / tf_peak
        kernels["prefill_pipeline"] = {
            "ms": ms_pipeline, "rows_per_s": rows / (ms_pipeline * 1e-3),
            "timed": "qsa_index_qk_prep, qsa_index_scores and qsa_index_topk_expand back to back, per step"}
        kernels["fused_select"] = {
            "ms": ms_fused, "alg_bytes": ab["fused_select"], "gbs": ab["fused_select"] / (ms_fused * 1e-3) / 1e9,
            "frac_of_measured_hbm": ab["fused_select"] / (ms_fused * 1e-3) / 1e9 / hbm_peak,
            "rows_per_s": rows / (ms_fused * 1e-3), "outidx_equals_two_calls": fused_equal,
            "timed": "qsa_index_scores_topk_expand over every row, back to back after the step loop"}
        kernels["prefill_pipeline_fused"] = {
            "ms": ms_pipeline_fused, "rows_per_s": rows / (ms_pipeline_fused * 1e-3),
            "timed": "qsa_index_qk_prep then qsa_index_scores_topk_expand, back to back, per step"}
        kernels["k2_chunked_8192"] = {
            "ms": ms_k2_chunked, "chunks": (rows + chunk_rows - 1) // chunk_rows,
            "gbs": ab["k2"] / (ms_k2_chunked * 1e-3) / 1e9,
            "frac_of_measured_hbm": ab["k2"] / (ms_k2_chunked * 1e-3) / 1e9 / hbm_peak,
            "timed": "K2 over the same rows as consecutive 8192-row calls, back to back after the step loop"}
        step_bytes = ab["k1_fused"] + ab["k2"]
        step_gbs = step_bytes / (ms_step * 1e-3) / 1e9
        kernels["step"] = {
            "ms": ms_step, "alg_bytes": step_bytes, "gbs": step_gbs, "frac_of_measured_hbm": step_gbs / hbm_peak,
            "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
            "timed": "the whole step (fused K1, then K2): ms_per_step of this line"}

        traffic = k2_profiled_traffic(B)
        k2_gbs = kernels["k2"]["gbs"]
        extra = {
            "roofline": {"bound": "hbm", "kernel": "k2_scores_tc", "achieved": k2_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": k2_gbs / hbm_peak, "traffic": traffic,
                         "peak_source": f"{peak_src} hbm_gbs"},
            "kernels": kernels,
            "e2e": {"value": whole_job_rows_per_s(rows, ms_e2e, world), "unit": UNIT,
                    "h2d_bytes_per_step": after["h2d"], "d2h_bytes_per_step": after["d2h"], "ms_per_step": ms_e2e,
                    "steps": after["K_e2e"], "block_ms_per_step": [round(x, 4) for x in after["blocks"]],
                    "how": "Python API, pinned host buffers; copies overlap compute across streams; "
                           "K2 in per-sequence row chunks; the median of three timed blocks of `steps` steps"},
            "gpu_launches": 2 * K,
            "clocks": clocks,
            "device_fault_flags": faults,
        }
        if decode is not None:
            extra["decode"] = decode
        if k1_small is not None:
            extra["k1_small_configs"] = k1_small
        if world == 1 and not args.no_cpu_baseline:
            extra["cpu_baseline"] = oracle_sample(wl)
        return extra


def run_ours(args, rank: int, world: int) -> None:
    run_steps(args, rank, world, PrefillStepGpu)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-decode", action="store_true", help="skip the paged decode-step leg")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip K1 on the small configurations and the B*S size sweep")
    ap.add_argument("--decode-batch", type=int, default=64, help="sequences in the decode-step leg")
    ap.add_argument("--only-decode", action="store_true",
                    help="run only the decode-step leg (for profiler captures)")
    ap.add_argument("--only-prefill-select", action="store_true",
                    help="run only the prefill selection of --batch sequences, fused and as two calls "
                         "(for profiler captures)")
    ap.add_argument("--only-k1-configs", nargs="?", const="all", default=None, metavar="NAMES",
                    help="run only K1 on the small configurations and the size sweep, or on the named "
                         "configurations (comma-separated) without the sweep; for profiler captures")
    ap.add_argument("--batch", type=int, default=8,
                    help="sequences per step (8 is the scoring workload; smaller for profiler captures)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank)
        elif args.only_decode:
            if rank == 0:
                import torch
                import sparse_attention_indexer_qsa_gb300 as qsa
                torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
                leg = decode_leg(qsa, qsa.load(), torch.cuda.current_stream(), args.steps, B=args.decode_batch)
                print(json.dumps({"decode": leg}), flush=True)
        elif args.only_prefill_select:
            if rank == 0:
                import torch
                import sparse_attention_indexer_qsa_gb300 as qsa
                torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
                leg = prefill_select_leg(qsa, qsa.load(), torch.cuda.current_stream(), args.steps, B=args.batch)
                print(json.dumps({"prefill_select": leg}), flush=True)
        elif args.only_k1_configs:
            if rank == 0:
                import torch
                import sparse_attention_indexer_qsa_gb300 as qsa
                torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
                names = None if args.only_k1_configs == "all" else args.only_k1_configs.split(",")
                leg = k1_configs_leg(qsa, qsa.load(), load_peaks()[0], names=names, sweep=names is None)
                print(json.dumps({"k1_small_configs": leg}), flush=True)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
