"""Benchmark of the packed index step (score + block top-k) on GB300.

One step = one idx_score_topk call (score kernel + top-k kernel) over the whole
synthetic batch of the workload, with the batch resident in HBM.  Prints ONE
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 restatement of the
method) on a bounded sample of the same workload, on this host's cores; it is
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
BYTES_PER_TOKEN = {"bf16": 256, "fp8_e4m3": 132, "nvfp4": 72}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
L2_BYTES = 129 * 1024 * 1024
L2_FLUSH_BYTES = 256 * 1024 * 1024
SCORE_SOURCES = ["idx_score.cu", "idx_ptx.cuh", "idx_internal.cuh"]
WIDE_SOURCES = ["idx_wide.cu", "idx_tc.cuh", "idx_ptx.cuh", "idx_internal.cuh"]


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


def kernel_sha(wide: bool = False) -> str:
    """Hash of the kernel sources as the compiler sees them (comments and
    layout left out); `profiles/traffic.json` holds DRAM counters per hash."""
    h = hashlib.sha256()
    for f in (WIDE_SOURCES if wide else SCORE_SOURCES):
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


def workload_config(s, R, args, ws_n) -> dict:
    """The workload's own keys in the JSON line's config (both arms)."""
    return {
        "workload": args.workload, "requests": R, "packed_queries": s.packed_queries,
        "gqa": s.gqa, "k_dtype": s.k_dtype, "q_dtype": s.q_dtype,
        "context": (f"U[{s.len_range[0]},{s.len_range[1]}]" if s.len_range else "explicit"),
        "topk": s.topk, "init_blocks": s.init_blocks, "local_blocks": s.local_blocks,
        "block_score": args.block_score,
        "block": 128, "page": 64, "parallelism": f"replicas x{ws_n}",
    }


def score_fn(idx, args):
    return idx.idx_score_topk_lse if args.block_score == "lse" else idx.idx_score_topk


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
    batch = workloads.make_batch(spec)
    s = batch.spec
    payload = batch.payload.to(dev)
    scale = None if batch.scale is None else batch.scale.to(dev)
    if s.k_dtype == "nvfp4":
        idx.idx_store_nvfp4(batch.staging.to(dev), batch.slot_mapping.to(dev), (payload, scale))
        batch.staging = None
    q = batch.q.to(dev)
    q_scale = None if batch.q_scale is None else batch.q_scale.to(dev)
    pt = batch.page_table.to(dev)
    slots = batch.slot_ids.to(dev)
    lens = batch.row_lens.to(dev)
    R, M, topk = batch.R, batch.M, s.topk
    out_ids = torch.empty((R, M, topk), dtype=torch.int32, device=dev)
    out_sc = torch.empty((R, M, topk), dtype=torch.float32, device=dev)
    wsp = idx.alloc_workspace(R, s.packed_queries, s.gqa, batch.max_pages, device=dev)
    stream = torch.cuda.current_stream(dev)

    fn = score_fn(idx, args)

    def step(events=None):
        # on whatever stream is current: the caller's, or a graph's capture stream
        if events is not None:
            idx.idx_set_kernel_events(*events)
        fn(q, q_scale, payload, scale, s.k_dtype, pt, slots, lens,
           s.packed_queries, s.gqa, s.init_blocks, s.local_blocks, topk,
           out_ids, out_sc, wsp, torch.cuda.current_stream(dev))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    flags = idx.idx_workspace_errors(wsp)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during warm-up")

    # ---- CUDA graphs: a serving loop captures the step once and replays it, so
    # the timed steps carry no per-call host cost.  A graph holds n_per steps
    # (n_per divides K) and is replayed K / n_per times.
    n_per = max(d for d in range(1, min(args.steps, 25) + 1) if args.steps % d == 0)
    reps = args.steps // n_per
    # inputs that fit in L2 (129 MB) get it flushed before every step (a 256 MB
    # write and read, outside the step's own pair of events); larger inputs
    # stream through it anyway and run back to back
    in_bytes = (payload.numel() + (0 if scale is None else scale.numel()) +
                q.numel() * q.element_size())
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) \
        if in_bytes < 2 * L2_BYTES else None
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain):
        for _ in range(1 if flush_buf is not None else n_per):
            step()
    # per-kernel events recorded by the library inside the graph (external nodes)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_per)]
    for trio in evs:            # torch creates an event's CUDA handle on its first record()
        for e in trio:
            e.record(stream)
    g_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_ev):
        for k in range(n_per):
            if flush_buf is not None:
                flush_l2(flush_buf)
            step(evs[k])
    for _ in range(2):
        g_plain.replay()
        g_ev.replay()
    torch.cuda.synchronize(dev)
    flags = idx.idx_workspace_errors(wsp)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} in the graph replays")

    # ---- timed region 1: K steps back to back (graph replays) ------------------
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    barrier(ws_n)
    torch.cuda.synchronize(dev)
    if flush_buf is None:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            g_plain.replay()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        run_ms = t0.elapsed_time(t1)
    else:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a_ev, b_ev in pairs:
            flush_l2(flush_buf)
            a_ev.record(stream)
            g_plain.replay()
            b_ev.record(stream)
        torch.cuda.synchronize(dev)
        run_ms = sum(a_ev.elapsed_time(b_ev) for a_ev, b_ev in pairs)
    barrier(ws_n)
    total_ms = max_over_ranks(run_ms, ws_n, dev)

    # ---- timed region 2: the same K steps with the library's events around each
    # kernel (per-kernel durations on the launching stream)
    barrier(ws_n)
    torch.cuda.synchronize(dev)
    score_ms, topk_ms, step_ms = [], [], []
    for _ in range(reps):
        g_ev.replay()
        torch.cuda.synchronize(dev)
        score_ms += [e[0].elapsed_time(e[1]) for e in evs]
        topk_ms += [e[1].elapsed_time(e[2]) for e in evs]
        step_ms += [e[0].elapsed_time(e[2]) for e in evs]
    barrier(ws_n)
    clocks = sampler.stop()
    evented_ms = max_over_ranks(sum(step_ms), ws_n, dev)

    # ---- ablation: the same step with every draft row scored on its own -------
    ablation = None
    if not args.no_ablation:
        n_ab = max(10, min(args.steps, 100))

        def perrow(events=None):
            if events is not None:
                idx.idx_set_kernel_events(*events)
            idx.idx_score_topk_perrow(q, q_scale, payload, scale, s.k_dtype, pt, slots, lens,
                                      s.packed_queries, s.gqa, s.init_blocks, s.local_blocks,
                                      topk, out_ids, out_sc, wsp, torch.cuda.current_stream(dev))

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
        ab_score = 0.0
        ab_step = 0.0
        for _ in range(n_ab):
            if flush_buf is not None:
                flush_l2(flush_buf)
            g_abev.replay()
            torch.cuda.synchronize(dev)
            ab_score += abev[0].elapsed_time(abev[1])
            ab_step += abev[0].elapsed_time(abev[2])
        ab_score = ab_score / n_ab * 1e3
        # with the L2 flush the back-to-back pass also holds the flushes: use the
        # evented steps then
        ab_us = (a0.elapsed_time(a1) * 1e3 / n_ab) if flush_buf is None else ab_step / n_ab * 1e3
        ablation = {"variant": "per-row (each draft row its own decode row, keys read P times)",
                    "us_per_step": round(ab_us, 3), "score_us": round(ab_score, 3),
                    "slowdown_vs_packed": round(ab_us / (total_ms / args.steps * 1e3), 3),
                    "steps": n_ab}

    # ---- end to end through the public API with host buffers ------------------
    e2e = run_e2e(idx, batch, payload, scale, dev, stream, args)

    ab = algorithmic_bytes(batch)
    score_avg_ms = sum(score_ms) / len(score_ms)
    wide = is_wide(s)
    achieved = ab["score"] / (score_avg_ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    tflops = ab["flops"] / (score_avg_ms * 1e-3) / 1e12
    tpeak, tpeak_src = measured_tensor_peak(s.k_dtype)
    # the bound is whichever ideal time is longer: bytes at the copy peak or
    # useful flops at the tensor peak
    tensor_bound = ab["flops"] / (tpeak * 1e12) > ab["score"] / (peak * 1e9)
    traffic = None
    try:
        with open(TRAFFIC_FILE) as fh:
            tr = json.load(fh).get(args.workload)
        if tr and tr.get("kernel_sha") == kernel_sha(wide):
            traffic = tr["dram_bytes_per_launch"]
    except Exception:
        pass
    ms_per_step = total_ms / args.steps
    value = ms_per_step * 1e3 / 1.0   # µs per step on each rank (replicas run concurrently)
    line = {
        "metric": metric_name(args),
        "value": round(value, 3),
        "unit": "us",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": (round(value / PUBLISHED_US[args.workload], 4)
                        if args.workload in PUBLISHED_US else None),
        "dtype": {"bf16": "bf16", "fp8_e4m3": "e4m3", "nvfp4": "e2m1xe4m3/bf16"}[s.k_dtype],
        "data": "synthetic",
        "config": {
            **workload_config(s, R, args, ws_n),
            "l2": (f"inputs larger than L2 ({ab['keys'] / 1e6:.0f} MB of keys read per step), no flush"
                   if flush_buf is None else
                   f"L2 flushed before every step ({L2_FLUSH_BYTES >> 20} MB written then read, "
                   f"outside the step's events; {ab['keys'] / 1e6:.1f} MB of keys per step)"),
            "aggregate_GBps": round(ws_n * ab["score"] / (ms_per_step * 1e-3) / 1e9, 1),
        },
        "roofline": {
            **({"bound": "tensor", "kernel": "wide_kernel", "achieved": round(tflops, 1),
                "peak": tpeak, "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
                "peak_source": tpeak_src, "traffic": traffic,
                "hbm_GBps": round(achieved, 1), "hbm_frac": round(achieved / peak, 4)}
               if tensor_bound else
               {"bound": "hbm", "kernel": "wide_kernel" if wide else "score_kernel",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src, "traffic": traffic,
                "tensor_TFLOPs": round(tflops, 1), "tensor_frac": round(tflops / tpeak, 4)}),
            "algorithmic_bytes_per_launch": ab["score"],
            "algorithmic_flops_per_launch": ab["flops"],
            "key_reads_per_request": ab["key_reads_per_request"],
            "score_us": round(score_avg_ms * 1e3, 3), "topk_us": round(sum(topk_ms) / len(topk_ms) * 1e3, 3),
            "frac_of_8TBps": round(achieved / 8000.0, 4),
            "timing": "value: K steps replayed from CUDA graphs (n_per steps per graph), no "
                      "events between the kernels; score_us, topk_us and achieved: CUDA "
                      "events the library records around each kernel (external event "
                      "nodes of a second graph) in a second pass of K steps",
            "steps_per_graph": n_per,
            "step_us_with_kernel_events": round(evented_ms / args.steps * 1e3, 3),
        },
        "e2e": e2e,
        "ablation": ablation,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if rank == 0:
        line["cpu_baseline"] = (cpu_baseline(batch, args)
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


def run_e2e(idx, batch, payload, scale, dev, stream, args):
    """Same step through the public API, inputs copied from pinned host memory
    and outputs read back, all inside the timed region.  As a serving loop would
    stage them: a step's inputs sit back to back in one pinned buffer (one copy
    in), its outputs in one device buffer (one copy out), and the copies run on a
    copy stream with two device buffer sets, so step k + 1's inputs are copied in
    and step k's outputs copied out while the next step's kernels run.  Keys that
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

    def compute(k, st):
        i = k % 2
        st.wait_event(ev_in[i])
        if k >= 2:
            st.wait_event(ev_out[i])           # step k - 2's outputs are out
        q, pt, sl, ln = vin[i][:4]
        qs = vin[i][4] if batch.q_scale is not None else None
        kp, ks = pools[k % npool]
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
            compute(k, st)
            copy_out(k)
        st.wait_event(ev_out[(n - 1) % 2])

    run(max(3, args.warmup))
    torch.cuda.synchronize(dev)
    # a serving loop replays the captured steps: G steps (a multiple of the
    # buffer sets and of the pool copies) per graph
    G = 2 * npool // math.gcd(2, npool)
    while G < 64:
        G *= 2
    reps = max(2, -(-max(10, min(args.steps, 200)) // G))
    n = reps * G
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    mode = "graph"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run(G)
        graph.replay()
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
    except RuntimeError as e:   # capture refused: time the same pipeline eagerly
        torch.cuda.synchronize(dev)
        mode = "eager (graph capture failed: %s)" % str(e).splitlines()[0][:100]
        t0.record(stream)
        for _ in range(reps):
            run(G)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    us = t0.elapsed_time(t1) * 1e3 / n
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
            "note": "keys stay resident in the pool (a layer's index-K cache); q, page table, "
                    "slot ids and row lengths are copied in (one pinned staging buffer, one "
                    "copy), ids and scores copied out (one copy), on a copy stream that "
                    "overlaps them with the neighbouring steps' kernels; the steps replayed "
                    "from a CUDA graph of steps_per_graph steps",
            "steps_per_graph": G, "mode": mode}


def _oracle_sample(batch, budget_s: float, block_score: str = "max"):
    """Time the oracle on request 0 with its rows cut to n tokens; returns
    (seconds per token-row, n, cores)."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from _util import oracle_kwargs
    s = batch.spec
    kw = dict(oracle_kwargs(batch), block_score=block_score)
    r0 = next(r for r in range(batch.R) if batch.group_lens()[r] > 0)
    n = 4096
    while True:
        lens = np.minimum(kw["row_lens"][r0:r0 + 1], n)
        kw1 = dict(kw, q=kw["q"][r0:r0 + 1], q_scale=None if kw["q_scale"] is None else kw["q_scale"][r0:r0 + 1],
                   slot_ids=kw["slot_ids"][r0:r0 + 1], row_lens=lens)
        t = time.perf_counter()
        oracle.index.index_step(**kw1)
        dt = time.perf_counter() - t
        tokens = int(lens.sum()) * s.gqa
        if dt > budget_s / 4 or n >= int(kw["row_lens"][r0].max()):
            return dt / tokens, n, dt
        n *= 2


def _cores() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(batch, args) -> dict:
    per_tok, n, dt = _oracle_sample(batch, budget_s=20.0, block_score=args.block_score)
    total_rows = int(sum(batch.row_lens[r].clamp_min(0).sum() for r in range(batch.R)
                         if batch.group_lens()[r] > 0)) * batch.spec.gqa
    us = per_tok * total_rows * 1e6
    return {"value": round(us, 1), "unit": "us", "cores": _cores(), "kind": "oracle",
            "sample": f"request 0, all {batch.M} packed rows cut to {n} tokens "
                      f"({dt:.2f} s), scaled by token-rows to the whole step"}


def run_reference(args):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    spec = workloads.WORKLOADS[args.workload]
    batch = workloads.make_batch(spec)
    budget = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    per_tok, n, dt = _oracle_sample(batch, budget_s=budget * 4, block_score=args.block_score)
    total_rows = int(sum(batch.row_lens[r].clamp_min(0).sum() for r in range(batch.R)
                         if batch.group_lens()[r] > 0)) * spec.gqa
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from _util import oracle_kwargs
    kw = dict(oracle_kwargs(batch), block_score=args.block_score)
    r0 = next(r for r in range(batch.R) if batch.group_lens()[r] > 0)
    lens = np.minimum(kw["row_lens"][r0:r0 + 1], n)
    kw1 = dict(kw, q=kw["q"][r0:r0 + 1], q_scale=None if kw["q_scale"] is None else kw["q_scale"][r0:r0 + 1],
               slot_ids=kw["slot_ids"][r0:r0 + 1], row_lens=lens)
    for _ in range(args.warmup):
        oracle.index.index_step(**kw1)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.index.index_step(**kw1)
    el = time.perf_counter() - t
    tokens = int(lens.sum()) * spec.gqa
    us = el / args.steps / tokens * total_rows * 1e6
    cores = _cores()
    sample = (f"per step: request 0, all {batch.M} packed rows cut to {n} tokens; "
              f"scaled by token-rows to the whole step")
    line = {
        "impl": "reference",
        "metric": metric_name(args),
        "value": round(us, 1), "unit": "us", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, batch.R, args, ws_n),
        "cpu_baseline": {"value": round(us, 1), "unit": "us", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--block-score", default="max", choices=["max", "lse"],
                    help="block score the selection ranks by (max: the headline step)")
    ap.add_argument("--no-ablation", action="store_true", help="skip the per-row ablation timing")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle's CPU timing (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
