"""Benchmark of the packed index step (score + block top-k) on GB300.

One step = one idx_score_topk call (score kernel + top-k kernel) over the whole
synthetic batch of the workload, with the batch resident in HBM.  Prints ONE
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The headline workload is timed first; the other decode workloads
(EXTRA_WORKLOADS) follow in the same process and are reported under "extra".
--impl reference times the CPU oracle (the plain fp64 restatement of the
method) over the whole step of the same workload on this host's cores; it is
the reference arm (the pages' own kernels are not available to run).
Multi-GPU runs (torchrun) are independent replicas: each rank scores its own
copy of the workload (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "index-step µs/layer and achieved HBM GB/s (score+top-k), 16 req × 131K bf16"
DEFAULT_WORKLOAD = "bf16_16x131k"
PUBLISHED_US = {"bf16_16x131k": 119.1, "fp8_16x131k": 87.4}   # packed kernel, one GB300 rank
# decode workloads timed after the headline in the same run (spec configs)
EXTRA_WORKLOADS = ["fp8_32x524k", "fp8_16x131k", "nvfp4_64x150k"]
BYTES_PER_TOKEN = {"bf16": 256, "fp8_e4m3": 132, "nvfp4": 72}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
L2_BYTES = 129 * 1024 * 1024
L2_FLUSH_BYTES = 256 * 1024 * 1024
SCORE_SOURCES = ["idx_score.cu", "idx_ptx.cuh", "idx_internal.cuh"]
WIDE_SOURCES = ["idx_wide.cu", "idx_tc.cuh", "idx_ptx.cuh", "idx_internal.cuh"]
STORE_SOURCES = ["idx_store.cu", "idx_internal.cuh"]


def is_wide(spec) -> bool:
    """More than 16 packed rows: the 128-row tensor-core tiles."""
    return spec.packed_queries * spec.gqa > 16


def code_only(text: str) -> str:
    """C/C++ source without its comments and with every run of blank space
    outside string and character literals made one space: what the compiler
    sees, so an edit of comments or layout keeps a kernel's hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):            # a comment counts as blank space
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":                       # a literal is kept as written
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif c.isspace():
            out.append(" ")
            i += 1
        else:
            out.append(c)
            i += 1
        if len(out) > 1 and out[-1] == " " and out[-2] == " ":
            out.pop()
    return "".join(out).strip()


def kernel_sha(wide: bool = False, sources=None) -> str:
    """Hash of the kernel sources as the compiler sees them (comments and
    layout left out); `profiles/traffic.json` holds DRAM counters per hash."""
    h = hashlib.sha256()
    for f in (sources or (WIDE_SOURCES if wide else SCORE_SOURCES)):
        with open(os.path.join(ROOT, "sparse_attention_indexer_packed_gb300", "csrc", f),
                  encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return 6800.0, "fallback 6.8 TB/s"


def measured_tensor_peak(k_dtype: str):
    """Dense tensor-core peak in TFLOP/s for the MMA's input type: the measured
    cuBLAS bf16 burst figure (f16 runs at the bf16 rate; e4m3 at twice it, the
    nominal 4.5 / 2.25 PFLOP/s ratio)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            bf16 = float(json.load(fh)["bf16_tflops"])
        src = "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS bf16 burst)"
    except Exception:
        bf16, src = 1900.0, "fallback 1.9 PFLOP/s bf16"
    if k_dtype == "fp8_e4m3":
        return 2.0 * bf16, src + " x 2 (e4m3 / bf16 nominal ratio)"
    return bf16, src + (" (f16 operands: same rate)" if k_dtype == "nvfp4" else "")


def algorithmic_bytes(batch) -> dict:
    """Bytes the score kernel must move at minimum: each request's keys read once
    up to its longest row, plus q, the page-table entries and slot/length
    metadata, plus the block-max writes; the top-k reads the block maxima back
    and writes the outputs."""
    s = batch.spec
    lens = batch.group_lens()
    k_bytes = sum(lens) * BYTES_PER_TOKEN[s.k_dtype]
    q_bytes = batch.q.numel() * batch.q.element_size() + (0 if batch.q_scale is None else batch.q_scale.numel() * 4)
    pages = sum((L + 63) // 64 for L in lens)
    meta = pages * 4 + batch.R * 4 + batch.row_lens.numel() * 4
    bm = 0
    for r in range(batch.R):
        if lens[r] == 0:
            continue
        for j in range(s.packed_queries):
            L = int(batch.row_lens[r, j])
            bm += s.gqa * max(0, (L + 127) // 128) * 4
    out = batch.R * batch.M * s.topk * 8
    # useful multiply-adds: every row against every key inside its own length
    flops = 0
    for r in range(batch.R):
        if lens[r] == 0:
            continue
        for j in range(s.packed_queries):
            flops += s.gqa * max(0, int(batch.row_lens[r, j])) * 128 * 2
    # per request the tensor-core path re-reads the keys once per 128-row tile
    tiles = -(-batch.M // 128) if batch.M > 16 else 1
    return {"score": k_bytes + q_bytes + meta + bm, "keys": k_bytes, "topk": bm + out,
            "flops": flops, "key_reads_per_request": tiles}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.dev = device_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_spec(spec, rank: int, world_size: int):
    """The workload a rank scores: replicas draw their own inputs (seed offset by
    rank) with the same shapes, so per-GPU work is fixed as N grows."""
    if world_size <= 1:
        return spec
    return workloads.Spec(**{**spec.__dict__, "seed": spec.seed + 100 * rank})


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, dev) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flush_l2(buf: torch.Tensor) -> None:
    """Evict L2 before a timed step: write a buffer twice the size of L2, then
    read it back, so the dirty lines of the write are written back to HBM here
    and not during the step that follows."""
    buf.fill_(1)
    buf.view(torch.int32).max()


def metric_name(args) -> str:
    """The headline metric on the default workload with the block-max score;
    any other workload or block score is named in the metric itself."""
    if args.workload == DEFAULT_WORKLOAD and args.block_score == "max":
        return METRIC
    suffix = "" if args.block_score == "max" else f", {args.block_score} block score"
    return f"index-step µs/layer ({args.workload}{suffix})"


def workload_config(s, R, args, ws_n, workload=None) -> dict:
    """The workload's own keys in the JSON line's config (the same on both arms)."""
    return {
        "workload": workload or args.workload, "requests": R, "packed_queries": s.packed_queries,
        "gqa": s.gqa, "k_dtype": s.k_dtype, "q_dtype": s.q_dtype,
        "context": (f"U[{s.len_range[0]},{s.len_range[1]}]" if s.len_range else "explicit"),
        "topk": s.topk, "init_blocks": s.init_blocks, "local_blocks": s.local_blocks,
        "block_score": args.block_score,
        "block": 128, "page": 64, "parallelism": f"replicas x{ws_n}",
    }


def score_fn(idx, args):
    return idx.idx_score_topk_lse if args.block_score == "lse" else idx.idx_score_topk


def percentile(xs, q):
    """The q-quantile of xs (linear interpolation between order statistics)."""
    ys = sorted(xs)
    if not ys:
        return float("nan")
    pos = (len(ys) - 1) * q
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (pos - lo)


class Resident:
    """One workload's batch resident in HBM with its outputs and workspace."""

    def __init__(self, idx, spec, dev):
        self.batch = batch = workloads.make_batch(spec)
        s = self.spec = batch.spec
        self.payload = batch.payload.to(dev)
        self.scale = None if batch.scale is None else batch.scale.to(dev)
        if s.k_dtype == "nvfp4":
            idx.idx_store_nvfp4(batch.staging.to(dev), batch.slot_mapping.to(dev),
                                (self.payload, self.scale))
        self.q = batch.q.to(dev)
        self.q_scale = None if batch.q_scale is None else batch.q_scale.to(dev)
        self.pt = batch.page_table.to(dev)
        self.slots = batch.slot_ids.to(dev)
        self.lens = batch.row_lens.to(dev)
        R, M = batch.R, batch.M
        self.out_ids = torch.empty((R, M, s.topk), dtype=torch.int32, device=dev)
        self.out_sc = torch.empty((R, M, s.topk), dtype=torch.float32, device=dev)
        self.wsp = idx.alloc_workspace(R, s.packed_queries, s.gqa, batch.max_pages, device=dev)
        self.in_bytes = (self.payload.numel() + (0 if self.scale is None else self.scale.numel()) +
                         self.q.numel() * self.q.element_size())

    def call(self, fn, dev, events=None):
        """One step on whatever stream is current (the caller's or a capture's)."""
        import sparse_attention_indexer_packed_gb300 as idx
        s = self.spec
        if events is not None:
            idx.idx_set_kernel_events(*events)
        fn(self.q, self.q_scale, self.payload, self.scale, s.k_dtype, self.pt, self.slots,
           self.lens, s.packed_queries, s.gqa, s.init_blocks, s.local_blocks, s.topk,
           self.out_ids, self.out_sc, self.wsp, torch.cuda.current_stream(dev))


def time_step(idx, res, fn, dev, stream, args, ws_n, min_seconds):
    """Time the step of a resident workload.

    A sample is K = args.steps steps replayed from CUDA graphs between two CUDA
    events (workloads whose inputs fit in L2 get it flushed before every step,
    outside the step's events).  Samples are repeated back to back until they
    span min_seconds and number at least 100 steps; value is the median per-step
    time over samples, max over ranks.  A second pass replays the same steps with
    the library's events around each kernel (external event nodes of a second
    graph) for the per-kernel durations."""
    K = args.steps
    n_per = max(d for d in range(1, min(K, 25) + 1) if K % d == 0)
    reps = K // n_per
    flush_buf = (torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
                 if res.in_bytes < 2 * L2_BYTES else None)
    for _ in range(args.warmup):
        res.call(fn, dev)
    torch.cuda.synchronize(dev)
    flags = idx.idx_workspace_errors(res.wsp)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during warm-up")
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain):
        for _ in range(1 if flush_buf is not None else n_per):
            res.call(fn, dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_per)]
    for trio in evs:            # torch creates an event's CUDA handle on its first record()
        for e in trio:
            e.record(stream)
    g_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ev):
        for k in range(n_per):
            if flush_buf is not None:
                flush_l2(flush_buf)
            res.call(fn, dev, evs[k])
    for _ in range(2):
        g_plain.replay()
        g_ev.replay()
    torch.cuda.synchronize(dev)
    flags = idx.idx_workspace_errors(res.wsp)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in the graph replays")

    def sample(pairs):
        """Record one sample of K steps; returns its event pairs."""
        out = []
        if flush_buf is None:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g_plain.replay()
            b.record(stream)
            out.append((a, b))
        else:
            for _ in range(K):
                flush_l2(flush_buf)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g_plain.replay()
                b.record(stream)
                out.append((a, b))
        pairs.append(out)

    def elapsed(p):
        return sum(a.elapsed_time(b) for a, b in p)

    # one sample sets the count; then all samples run back to back, one sync
    probe = []
    sample(probe)
    torch.cuda.synchronize(dev)
    per_sample_ms = max(1e-3, elapsed(probe[0]))
    n_samples = max(5, -(-100 // K), int(math.ceil(min_seconds * 1e3 / per_sample_ms)))
    n_samples = min(n_samples, 20000)
    barrier(ws_n)
    torch.cuda.synchronize(dev)
    samples = []
    for _ in range(n_samples):
        sample(samples)
    torch.cuda.synchronize(dev)
    barrier(ws_n)
    step_us = [elapsed(p) * 1e3 / K for p in samples]
    med = statistics.median(step_us)
    value = max_over_ranks(med, ws_n, dev)

    # per-kernel durations: at least 100 steps with the library's events
    n_ev = max(reps, -(-100 // n_per))
    score_ms, topk_ms, step_ms = [], [], []
    for _ in range(n_ev):
        g_ev.replay()
        torch.cuda.synchronize(dev)
        score_ms += [e[0].elapsed_time(e[1]) for e in evs]
        topk_ms += [e[1].elapsed_time(e[2]) for e in evs]
        step_ms += [e[0].elapsed_time(e[2]) for e in evs]
    # isolated calls, the do_bench way: per rep the L2 flushed, then CUDA events
    # around one step replayed from a one-step graph, so nothing of the step
    # overlaps the one before it
    iso_buf = (flush_buf if flush_buf is not None else
               torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev))
    if flush_buf is None:
        g_one = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_one):
            res.call(fn, dev)
        g_one.replay()
        torch.cuda.synchronize(dev)
    else:
        g_one = g_plain
    iso_pairs = []
    for _ in range(max(100, K)):
        flush_l2(iso_buf)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g_one.replay()
        b.record(stream)
        iso_pairs.append((a, b))
    torch.cuda.synchronize(dev)
    iso_us = [a.elapsed_time(b) * 1e3 for a, b in iso_pairs]
    del iso_buf
    return {
        "isolated": {"median_us": round(max_over_ranks(statistics.median(iso_us), ws_n, dev), 3),
                     "p10_us": round(percentile(iso_us, 0.1), 3),
                     "p90_us": round(percentile(iso_us, 0.9), 3), "reps": len(iso_us),
                     "how": "per rep: L2 flushed (256 MB written then read), then CUDA events "
                            "around one step (score + top-k) replayed from a one-step CUDA "
                            "graph; no overlap with the step before"},
        "value_us": value, "median_us": med, "p10_us": percentile(step_us, 0.1),
        "p90_us": percentile(step_us, 0.9), "samples": n_samples, "steps_per_sample": K,
        "timed_steps": n_samples * K, "timed_s": sum(elapsed(p) for p in samples) / 1e3,
        "steps_per_graph": 1 if flush_buf is not None else n_per,
        "l2": (f"inputs larger than L2 ({res.in_bytes / 1e6:.0f} MB per step), no flush"
               if flush_buf is None else
               f"L2 flushed before every step ({L2_FLUSH_BYTES >> 20} MB written then read, "
               f"outside the step's events)"),
        "score_us": statistics.fmean(score_ms) * 1e3, "topk_us": statistics.fmean(topk_ms) * 1e3,
        "score_us_median": statistics.median(score_ms) * 1e3,
        "evented_step_us": statistics.fmean(step_ms) * 1e3, "evented_steps": len(step_ms),
        "flush_buf": flush_buf,
    }


def roofline(res, t, workload) -> dict:
    """The dominant (score) kernel against its bound: algorithmic bytes at the
    measured copy peak, or useful flops at the measured tensor peak, whichever
    ideal time is longer."""
    s = res.spec
    ab = algorithmic_bytes(res.batch)
    wide = is_wide(s)
    score_s = t["score_us"] * 1e-6
    achieved = ab["score"] / score_s / 1e9
    peak, peak_src = measured_peak()
    tflops = ab["flops"] / score_s / 1e12
    tpeak, tpeak_src = measured_tensor_peak(s.k_dtype)
    tensor_bound = ab["flops"] / (tpeak * 1e12) > ab["score"] / (peak * 1e9)
    traffic = None
    try:
        with open(TRAFFIC_FILE) as fh:
            tr = json.load(fh).get(workload)
        if tr and tr.get("kernel_sha") == kernel_sha(wide):
            traffic = tr["dram_bytes_per_launch"]
    except Exception:
        pass
    out = ({"bound": "tensor", "kernel": "wide_kernel", "achieved": round(tflops, 1),
            "peak": tpeak, "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
            "peak_source": tpeak_src, "traffic": traffic,
            "hbm_GBps": round(achieved, 1), "hbm_frac": round(achieved / peak, 4)}
           if tensor_bound else
           {"bound": "hbm", "kernel": "wide_kernel" if wide else "score_kernel",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": traffic,
            "tensor_TFLOPs": round(tflops, 1), "tensor_frac": round(tflops / tpeak, 4)})
    out.update({
        "algorithmic_bytes_per_launch": ab["score"],
        "algorithmic_flops_per_launch": ab["flops"],
        "key_reads_per_request": ab["key_reads_per_request"],
        "score_us": round(t["score_us"], 3), "score_us_median": round(t["score_us_median"], 3),
        "topk_us": round(t["topk_us"], 3),
        "frac_of_8TBps": round(achieved / 8000.0, 4),
        "step_us_with_kernel_events": round(t["evented_step_us"], 3),
        "evented_steps": t["evented_steps"],
    })
    return out


def time_store(idx, res, dev, stream, reps=20) -> dict:
    """The NVFP4 quantize-store of the batch's keys (the write path, outside the
    index step), timed on its own: every staged key quantised and written into
    the pool planes.  Inputs are far larger than L2, so no flush."""
    b = res.batch
    src = b.staging.to(dev)
    smap = b.slot_mapping.to(dev)
    pool = (res.payload, res.scale)
    for _ in range(3):
        idx.idx_store_nvfp4(src, smap, pool, stream)
    torch.cuda.synchronize(dev)
    pairs = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        idx.idx_store_nvfp4(src, smap, pool, stream)
        e.record(stream)
        pairs.append((a, e))
    torch.cuda.synchronize(dev)
    us = [a.elapsed_time(e) * 1e3 for a, e in pairs]
    keys = int(smap.numel())
    live = int((smap >= 0).sum().item())
    # per key: its 8-byte slot read; per stored key: 256 B of bf16 read, 64 B of
    # codes and 8 B of scales written
    nbytes = 8 * keys + live * (256 + 64 + 8)
    med = statistics.median(us)
    peak, peak_src = measured_peak()
    del src, smap
    achieved = nbytes / (med * 1e-6) / 1e9
    traffic = None
    try:
        with open(TRAFFIC_FILE) as fh:
            tr = json.load(fh).get(res.spec.name + ":store")
        if tr and tr.get("kernel_sha") == kernel_sha(sources=STORE_SOURCES):
            traffic = tr["dram_bytes_per_launch"]
    except Exception:
        pass
    return {"kernel": "store_nvfp4_kernel", "keys": keys, "us": round(med, 3), "traffic": traffic,
            "p10_us": round(percentile(us, 0.1), 3), "p90_us": round(percentile(us, 0.9), 3),
            "reps": reps, "algorithmic_bytes": nbytes, "bound": "hbm",
            "achieved": round(achieved, 1), "unit": "GB/s", "peak": peak,
            "frac": round(achieved / peak, 4), "peak_source": peak_src}


def timing_record(t) -> dict:
    return {"median_us": round(t["median_us"], 3), "p10_us": round(t["p10_us"], 3),
            "p90_us": round(t["p90_us"], 3), "samples": t["samples"],
            "steps_per_sample": t["steps_per_sample"], "timed_steps": t["timed_steps"],
            "timed_s": round(t["timed_s"], 3), "steps_per_graph": t["steps_per_graph"],
            "l2": t["l2"], "isolated": t["isolated"],
            "how": "value = median over samples of K steps each (CUDA graph replays between "
                   "two CUDA events, samples back to back); score_us / topk_us: CUDA events "
                   "the library records around each kernel (external event nodes of a "
                   "second graph), averaged over its evented_steps"}


def run_ablation(idx, res, dev, stream, flush_buf, n_ab):
    """The same step with every draft row scored on its own (per-row kernel)."""
    s = res.spec

    def perrow(events=None):
        if events is not None:
            idx.idx_set_kernel_events(*events)
        idx.idx_score_topk_perrow(res.q, res.q_scale, res.payload, res.scale, s.k_dtype, res.pt,
                                  res.slots, res.lens, s.packed_queries, s.gqa, s.init_blocks,
                                  s.local_blocks, s.topk, res.out_ids, res.out_sc, res.wsp,
                                  torch.cuda.current_stream(dev))

    for _ in range(3):
        perrow()
    abev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in abev:
        e.record(stream)
    g_ab = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ab):
        perrow()
    g_abev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_abev):
        perrow(abev)
    g_ab.replay()
    torch.cuda.synchronize(dev)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(n_ab):
        if flush_buf is not None:
            flush_l2(flush_buf)
        g_ab.replay()
    a1.record(stream)
    torch.cuda.synchronize(dev)
    ab_score = ab_step = 0.0
    for _ in range(n_ab):
        if flush_buf is not None:
            flush_l2(flush_buf)
        g_abev.replay()
        torch.cuda.synchronize(dev)
        ab_score += abev[0].elapsed_time(abev[1])
        ab_step += abev[0].elapsed_time(abev[2])
    # with the L2 flush the back-to-back pass also holds the flushes: use the
    # evented steps then
    ab_us = (a0.elapsed_time(a1) * 1e3 / n_ab) if flush_buf is None else ab_step / n_ab * 1e3
    return {"variant": "per-row (each draft row its own decode row, keys read P times)",
            "us_per_step": round(ab_us, 3), "score_us": round(ab_score / n_ab * 1e3, 3),
            "steps": n_ab}


def measure_extra(idx, name, args, dev, stream, ws_n, rank):
    """Another decode workload in the same run: value, per-kernel times,
    roofline and end-to-end step, without the ablation or the CPU baseline."""
    spec = replica_spec(workloads.WORKLOADS[name], rank, ws_n)
    res = Resident(idx, spec, dev)
    fn = score_fn(idx, args)
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.2)
    t = time_step(idx, res, fn, dev, stream, args, ws_n, min_seconds=0.3)
    clocks = sampler.stop()
    e2e = run_e2e(idx, res.batch, res.payload, res.scale, dev, stream, args, ws_n)
    store = time_store(idx, res, dev, stream) if res.spec.k_dtype == "nvfp4" else None
    out = {"workload": name, "value": round(t["value_us"], 3), "unit": "us",
           "config": workload_config(res.spec, res.batch.R, args, ws_n, workload=name),
           "timing": timing_record(t), "roofline": roofline(res, t, name), "e2e": e2e,
           "clocks": clocks, "gpu_launches": 2 * t["timed_steps"]}
    if store is not None:
        out["store"] = store
    del res, t
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import sparse_attention_indexer_packed_gb300 as idx
    from sparse_attention_indexer_packed_gb300.build import build_library

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build_library()

    spec = replica_spec(workloads.WORKLOADS[args.workload], rank, ws_n)
    res = Resident(idx, spec, dev)
    s, batch = res.spec, res.batch
    stream = torch.cuda.current_stream(dev)
    fn = score_fn(idx, args)

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    t = time_step(idx, res, fn, dev, stream, args, ws_n, min_seconds=args.min_seconds)
    clocks = sampler.stop()
    gpu_ids = res.out_ids.cpu().numpy()

    ablation = None
    if not args.no_ablation:
        ablation = run_ablation(idx, res, dev, stream, t["flush_buf"],
                                max(10, min(args.steps, 100)))
        ablation["slowdown_vs_packed"] = round(ablation["us_per_step"] / t["value_us"], 3)

    # ---- end to end through the public API with host buffers ------------------
    e2e = run_e2e(idx, batch, res.payload, res.scale, dev, stream, args, ws_n)
    store = time_store(idx, res, dev, stream) if s.k_dtype == "nvfp4" else None
    rl = roofline(res, t, args.workload)
    ab = algorithmic_bytes(batch)
    value = t["value_us"]   # µs per step on each rank (replicas run concurrently)
    line = {
        "metric": metric_name(args),
        "value": round(value, 3),
        "unit": "us",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": (round(value / PUBLISHED_US[args.workload], 4)
                        if args.workload in PUBLISHED_US else None),
        "dtype": {"bf16": "bf16", "fp8_e4m3": "e4m3", "nvfp4": "e2m1xe4m3/bf16"}[s.k_dtype],
        "data": "synthetic",
        "config": workload_config(s, batch.R, args, ws_n),
        "timing": dict(timing_record(t),
                       aggregate_GBps=round(ws_n * ab["score"] / (value * 1e-6) / 1e9, 1)),
        "roofline": rl,
        "e2e": e2e,
        "ablation": ablation,
        "gpu_launches": 2 * t["timed_steps"],
        "clocks": clocks,
    }
    if store is not None:
        line["store"] = store
    del t["flush_buf"]
    if not args.no_extra:
        extras = [w for w in EXTRA_WORKLOADS if w != args.workload]
        if extras:
            del res
            torch.cuda.empty_cache()
            line["extra"] = [measure_extra(idx, w, args, dev, stream, ws_n, rank) for w in extras]
    if rank == 0:
        line["cpu_baseline"] = (cpu_baseline(batch, args, gpu_ids)
                                if ws_n == 1 and not args.no_cpu_baseline else None)
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _layout(tensors):
    """Byte offsets of `tensors` laid back to back at 256-byte aligned offsets."""
    offs, off = [], 0
    for t in tensors:
        off = (off + 255) // 256 * 256
        nb = t.numel() * t.element_size()
        offs.append((off, nb))
        off += nb
    return offs, (off + 255) // 256 * 256


def _views(buf, tensors, offs):
    return [buf[o:o + nb].view(t.dtype).view(t.shape) for t, (o, nb) in zip(tensors, offs)]


def run_e2e(idx, batch, payload, scale, dev, stream, args, ws_n=1):
    """Same step through the public API, inputs copied from pinned host memory
    and outputs read back, all inside the timed region.  As a serving loop would
    stage them: a step's inputs sit back to back in one pinned buffer (one copy
    in), its outputs in one device buffer (one copy out), and the copies run on a
    copy stream with two device buffer sets, so step k + 1's inputs are copied in
    and step k's outputs copied out while the next step's kernels run; the
    copies' events are waited for at the previous step's top-k launch.  Keys that
    fit in L2 are rotated over enough identical copies of the pool (at least
    twice L2 in all) that no step finds its keys in L2 from an earlier one."""
    s = batch.spec
    kbytes = payload.numel() + (0 if scale is None else scale.numel())
    npool = max(1, -(-2 * L2_BYTES // kbytes)) if kbytes < 2 * L2_BYTES else 1
    pools = [(payload, scale)] + [(payload.clone(), None if scale is None else scale.clone())
                                  for _ in range(npool - 1)]
    R, M, topk = batch.R, batch.M, s.topk
    ins = [batch.q, batch.page_table, batch.slot_ids, batch.row_lens]
    if batch.q_scale is not None:
        ins.append(batch.q_scale)
    outs = [torch.empty((R, M, topk), dtype=torch.int32), torch.empty((R, M, topk), dtype=torch.float32)]
    ioffs, itotal = _layout(ins)
    ooffs, ototal = _layout(outs)
    h_in = torch.empty(itotal, dtype=torch.uint8).pin_memory()
    for h, t in zip(_views(h_in, ins, ioffs), ins):
        h.copy_(t)
    d_in = [torch.empty(itotal, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(ototal, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_out = [torch.empty(ototal, dtype=torch.uint8).pin_memory() for _ in range(2)]
    vin = [_views(b, ins, ioffs) for b in d_in]
    vout = [_views(b, outs, ooffs) for b in d_out]
    wsp = idx.alloc_workspace(R, s.packed_queries, s.gqa, batch.max_pages, device=dev)
    fn = score_fn(idx, args)
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the set copied in
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the step on the set has run
    ev_out = [torch.cuda.Event() for _ in range(2)]   # its outputs copied out

    def copy_in(k):
        i = k % 2
        with torch.cuda.stream(cs):
            if k >= 2:
                cs.wait_event(ev_used[i])      # step k - 2 has read this set
            d_in[i].copy_(h_in, non_blocking=True)
            ev_in[i].record(cs)

    def compute(k, st, last):
        # The step's dependencies on the copy stream are hung on the previous
        # step's top-k launch (idx_set_kernel_waits), not on this step's score
        # launch, so the score kernel keeps its programmatic overlap with the
        # step before it: step k + 1's inputs (copied after step k - 1's outputs
        # on the copy stream) are waited for before step k's top-k; the first
        # step of a run waits before its score kernel.
        i = k % 2
        q, pt, sl, ln = vin[i][:4]
        qs = vin[i][4] if batch.q_scale is not None else None
        kp, ks = pools[k % npool]
        idx.idx_set_kernel_waits(ev_in[i] if k == 0 else None,
                                 None if last else ev_in[(k + 1) % 2])
        fn(q, qs, kp, ks, s.k_dtype, pt, sl, ln, s.packed_queries, s.gqa,
           s.init_blocks, s.local_blocks, topk, vout[i][0], vout[i][1], wsp, st)
        ev_used[i].record(st)

    def copy_out(k):
        i = k % 2
        with torch.cuda.stream(cs):
            cs.wait_event(ev_used[i])
            h_out[i].copy_(d_out[i], non_blocking=True)
            ev_out[i].record(cs)

    def run(n):
        # on the current stream (the caller's, or a graph's capture stream)
        st = torch.cuda.current_stream(dev)
        start = torch.cuda.Event()
        start.record(st)
        cs.wait_event(start)
        copy_in(0)
        for k in range(n):
            if k + 1 < n:
                copy_in(k + 1)
            compute(k, st, k + 1 == n)
            copy_out(k)
        st.wait_event(ev_out[(n - 1) % 2])

    run(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    # a serving loop replays the captured steps: G steps (a multiple of the
    # buffer sets and of the pool copies) per graph
    G = 2 * npool // math.gcd(2, npool)
    while G < 64:
        G *= 2
    # each replay of G steps is timed on its own; the value is the median over
    # replays (at least nine, so neither p10 nor p90 is an extreme), and one
    # disturbed window (the host's copy path is shared) does not set it
    reps = max(9, -(-max(10, min(args.steps, 200)) // G))
    n = reps * G
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    mode = "graph"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run(G)
        graph.replay()
        torch.cuda.synchronize(dev)
        evs[0].record(stream)
        for r in range(reps):
            graph.replay()
            evs[r + 1].record(stream)
    except RuntimeError as e:   # capture refused: time the same pipeline eagerly
        torch.cuda.synchronize(dev)
        mode = "eager (graph capture failed: %s)" % str(e).splitlines()[0][:100]
        evs[0].record(stream)
        for r in range(reps):
            run(G)
            evs[r + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(evs[r].elapsed_time(evs[r + 1]) * 1e3 / G for r in range(reps))
    # replicas run concurrently: the job's step is the slowest rank's
    us = max_over_ranks(statistics.median(per), ws_n, dev)
    p10 = max_over_ranks(per[int(0.1 * (reps - 1))], ws_n, dev)
    p90 = max_over_ranks(per[int(round(0.9 * (reps - 1)))], ws_n, dev)
    # the staged buffers must give what the same call on separate device tensors gives
    ref_ids = torch.empty((R, M, topk), dtype=torch.int32, device=dev)
    ref_sc = torch.empty((R, M, topk), dtype=torch.float32, device=dev)
    fn(batch.q.to(dev), None if batch.q_scale is None else batch.q_scale.to(dev), payload, scale,
       s.k_dtype, batch.page_table.to(dev), batch.slot_ids.to(dev), batch.row_lens.to(dev),
       s.packed_queries, s.gqa, s.init_blocks, s.local_blocks, topk, ref_ids, ref_sc, wsp, stream)
    torch.cuda.synchronize(dev)
    got = _views(h_out[(G - 1) % 2], outs, ooffs)
    if not (torch.equal(got[0], ref_ids.cpu()) and
            torch.equal(got[1].view(torch.int32), ref_sc.cpu().view(torch.int32))):
        raise RuntimeError("staged end-to-end outputs differ from the device-resident call")
    return {"value": round(us, 3), "unit": "us", "h2d_bytes_per_step": int(itotal),
            "d2h_bytes_per_step": int(ototal), "steps": n, "key_pool_copies": npool,
            "replays": reps, "p10": round(p10, 3), "p90": round(p90, 3),
            "note": "keys stay resident in the pool (a layer's index-K cache); q, page table, "
                    "slot ids and row lengths are copied in (one pinned staging buffer, one "
                    "copy), ids and scores copied out (one copy), on a copy stream that "
                    "overlaps them with the neighbouring steps' kernels (step k + 1's input "
                    "copy is waited for at step k's top-k launch, idx_set_kernel_waits); the "
                    "steps replayed from a CUDA graph of steps_per_graph steps, each replay "
                    "timed, the median per step reported",
            "steps_per_graph": G, "mode": mode}


def _oracle_pool(batch, block_score):
    """The oracle's step arguments for the batch and a process pool running it on
    every host core (oracle.pool)."""
    import oracle.inputs
    import oracle.pool
    kw = dict(oracle.inputs.step_kwargs(batch), block_score=block_score)
    return oracle.pool.OraclePool(kw)


def _tokens_rows(batch, requests) -> int:
    """Token-rows the oracle scores for these requests (rows x their lengths)."""
    lens = batch.group_lens()
    return int(sum(batch.row_lens[r].clamp_min(0).sum() for r in requests if lens[r] > 0)) * \
        batch.spec.gqa


def cpu_baseline(batch, args, gpu_ids=None) -> dict:
    """The oracle (as it stands) timed on this host's cores over the whole step:
    every request and packed row, requests handed to single-threaded worker
    processes.  One untimed step starts the workers; then steps are timed until
    about 10 s of wall time (at least 2).  The untimed step's ids are compared
    with the GPU's, row by row, as a full-size cross-check."""
    import oracle.pool
    with _oracle_pool(batch, args.block_score) as p:
        ids, _ = p.step()
        times = []
        t_end = time.perf_counter() + 10.0
        while len(times) < 2 or (time.perf_counter() < t_end and len(times) < 20):
            t0 = time.perf_counter()
            p.step()
            times.append(time.perf_counter() - t0)
        workers, nreq = p.workers, len(p.requests)
    out = {"value": round(statistics.median(times) * 1e6, 1), "unit": "us", "cores": workers,
           "kind": "oracle", "cpu_model": oracle.pool.cpu_model(),
           "sample": (f"the whole step: all {nreq} requests with keys x {batch.M} packed rows "
                      f"({_tokens_rows(batch, range(batch.R))} token-rows), {len(times)} timed "
                      f"steps after one untimed one, median; {workers} single-threaded worker "
                      f"processes, one request per task")}
    if gpu_ids is not None:
        same = sum(set(ids[r, i][ids[r, i] >= 0].tolist()) ==
                   set(gpu_ids[r, i][gpu_ids[r, i] >= 0].tolist())
                   for r in range(batch.R) for i in range(batch.M))
        out["ids_equal_to_gpu_rows"] = f"{same}/{batch.R * batch.M}"
    return out


def run_reference(args):
    """The reference arm: the oracle timed on this host's cores, W untimed and K
    timed steps of the whole workload (every request and row), on the same
    config, metric and unit as our arm.  Should the second warm-up step run past
    6 s, each step is a bounded sample instead: the longest requests that fit
    3 s, scaled by token-rows to the whole step (said in the line)."""
    import oracle.pool
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    spec = workloads.WORKLOADS[args.workload]
    batch = workloads.make_batch(spec)
    with _oracle_pool(batch, args.block_score) as p:
        todo = list(p.requests)
        p.step(todo)                       # first warm-up step (starts the workers)
        t0 = time.perf_counter()
        p.step(todo)                       # second warm-up step sizes the sample
        second = time.perf_counter() - t0
        scale = 1.0
        if second > 6.0:
            per_tok = second / max(1, _tokens_rows(batch, todo))
            keep, acc = [], 0
            for r in todo:
                if keep and (acc + _tokens_rows(batch, [r])) * per_tok > 3.0:
                    break
                keep.append(r)
                acc += _tokens_rows(batch, [r])
            scale = _tokens_rows(batch, todo) / max(1, acc)
            todo = keep
        for _ in range(max(0, args.warmup - 2)):
            p.step(todo)
        times = []
        for _ in range(args.steps):
            t1 = time.perf_counter()
            p.step(todo)
            times.append((time.perf_counter() - t1) * scale)
        workers = p.workers
    us = statistics.median(times) * 1e6
    if scale == 1.0:
        sample = (f"each step the whole workload: {len(todo)} requests with keys x {batch.M} "
                  f"packed rows; median of {args.steps} steps after {args.warmup} untimed; "
                  f"{workers} single-threaded worker processes, one request per task")
    else:
        sample = (f"each step {len(todo)} of the requests (the longest), scaled by token-rows "
                  f"(x{scale:.2f}) to the whole step; median of {args.steps} steps")
    line = {
        "impl": "reference",
        "metric": metric_name(args),
        "value": round(us, 1), "unit": "us", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, batch.R, args, ws_n),
        "cpu_baseline": {"value": round(us, 1), "unit": "us", "cores": workers, "kind": "oracle",
                         "cpu_model": oracle.pool.cpu_model(), "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--block-score", default="max", choices=["max", "lse"],
                    help="block score the selection ranks by (max: the headline step)")
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="timed samples of K steps are repeated until they span this long")
    ap.add_argument("--no-ablation", action="store_true", help="skip the per-row ablation timing")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle's CPU timing (profiling runs)")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --workload (not the other decode workloads as well)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
