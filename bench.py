#!/usr/bin/env python3
"""Benchmark of the W4A16 GEMM hot path on GB300.

A step is one pass of the hot path over one batch of synthetic input: for the
default workload (the decode square projection: K = N = 4096, group 128) one
W4A16 GEMM call for each M in {1, 2, 4, 8, 16}.  Every call in the timed
region uses a distinct copy of the quantized weight (enough copies to exceed
three times the L2 size), so the weight stream always comes from HBM.  The
timed region is one replay of a CUDA graph holding exactly --steps steps,
bracketed by CUDA events on the capture stream.

Printed: one JSON line (rank 0).  `value` is the weight-stream bandwidth of
the whole job (packed words + scales + zeros of every call, all ranks) over the
timed region; per-M microseconds per call (CUDA graph, and eager launches one
by one), GB/s in three conventions (packed + scales + zeros; packed words
only; every algorithmic byte), roofline fractions, a cuBLAS fp16 reference
(torch.matmul on the dequantized weight, same rotation) and the fp64 oracle on
the host cores (`cpu_baseline`) ride along.

--impl reference times the fp64 CPU oracle instead (the reference arm).
Multi-GPU (torchrun): every rank runs the same step on its own GPU with its own
weights (replicas, weak scaling); timings are max-reduced over ranks.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("W4A16 µs/call and weight-stream HBM GB/s (% of GB300 roofline), M=1..16")
GROUP = 128

# workload name -> shapes (K, N), Ms, outliers, experts
WORKLOADS = {
    "decode_square": dict(shapes=[(4096, 4096)], Ms=[1, 2, 4, 8, 16], outliers=False, experts=1,
                          config=1),
    "decode_ffn": dict(shapes=[(4096, 14336), (14336, 4096)], Ms=[1, 2, 4, 8, 16], outliers=True,
                       experts=1, config=2),
    "moe_experts": dict(shapes=[(2048, 768), (768, 2048)], Ms=[1, 2, 4, 8, 16], outliers=False,
                        experts=64, config=3),
    "prefill_sweep": dict(shapes=[(4096, 14336), (8192, 28672)],
                          Ms=[16, 32, 64, 128, 256, 1024, 4096], outliers=False, experts=1,
                          config=4),
}


def weight_bytes(K, N, group=GROUP):
    return K * N // 2 + 2 * 2 * (K // group) * N


def total_bytes(M, K, N, group=GROUP):
    return weight_bytes(K, N, group) + 2 * M * K + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


# The sources each workload's kernels are built from: a committed ncu summary
# is used only while these are unchanged.
KERNEL_SOURCES = {
    "decode": ["api.cu", "common.cuh", "decode.cu", "decode_math.cuh", "decode_tma.cu",
               "sm100_ptx.cuh", "tmap.cu", "tmap.cuh"],
    "prefill": ["api.cu", "common.cuh", "prefill.cu", "prefill_tile.cuh",
                "sm100_ptx.cuh", "tcgen05.cuh", "tmap.cu", "tmap.cuh"],
}


def workload_kind(workload):
    return "prefill" if workload.startswith("prefill") else "decode"


def source_sha(kind):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_codes_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kind]):
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """Per-launch DRAM bytes of the workload's kernels from the committed ncu
    summary, or None when absent or taken on a different kernel source."""
    kind = workload_kind(workload)
    path = os.path.join(ROOT, "profiles", "%s_kernel_%s.txt" % (kind, workload))
    if not os.path.exists(path):
        return None
    kv = {}
    for ln in open(path):
        if ":" in ln and not ln.startswith(" "):
            k, v = ln.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha") != source_sha(kind):
        return None
    try:
        return float(kv["dram_bytes_per_launch_mean"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples; only those that arrive
    inside the timed region [mark_start, mark_end] are reported."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        inside = [ln for t, ln in self.lines if self.t0 is not None and self.t0 <= t <= self.t1]
        used = inside if inside else [ln for _, ln in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in used:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "samples_in_timed_region": len(inside)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("W4A16_BENCH_BACKEND") != "gloo"
                                else "gloo")
        pg = dist
    return rank, local, world, pg


def reduce_max(pg, value, device):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg):
    if pg is not None:
        pg.barrier()


# --------------------------------------------------------------- CPU oracle
def oracle_calls(wl, cols, rows=None):
    """Inputs of one sampled step for the fp64 oracle: the first `cols` columns
    of every weight (quantized once, offline) and the step's activations (their
    first `rows` rows when given)."""
    import oracle
    from weight_only_int4_codes_gb300 import synth
    calls = []
    for si, (K, N) in enumerate(wl["shapes"]):
        n = min(cols, N)
        W = synth.weight(K, n, seed=synth.weight_seed(wl["config"], shape_index=si),
                         outliers=wl["outliers"])
        qw = oracle.quantize_pack(W, GROUP)
        for M in wl["Ms"]:
            x = synth.activations(M, K, seed=synth.x_seed(wl["config"], M, shape_index=si))
            if rows is not None:
                x = x[:rows]
            calls.append((x, qw, weight_bytes(K, n)))
    return calls


def oracle_step(wl, calls):
    import oracle
    for _ in range(wl["experts"]):
        for x, qw, _b in calls:
            oracle.gemm(x, *qw, group=GROUP)


def oracle_sample(wl, cols, reps_min_s):
    """Time the fp64 oracle on a column sample of every call of one step,
    repeated for at least `reps_min_s` seconds.  Returns (median seconds per
    sampled step, weight bytes per sampled step, threads used)."""
    import oracle
    calls = oracle_calls(wl, cols)
    per_step_bytes = sum(c[2] for c in calls) * wl["experts"]
    oracle_step(wl, calls)                       # warm (library load, page faults)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle_step(wl, calls)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= reps_min_s:
            break
    return statistics.median(times), per_step_bytes, oracle.num_threads()


def run_reference(args, rank, world, pg):
    """Reference arm: the fp64 CPU oracle, rank 0 only."""
    wl = WORKLOADS[args.workload]
    if rank != 0:
        return
    import oracle
    # The sample of a step: the first `cols` columns of every weight (and, if
    # that is not enough, the first `rows` rows of every x), shrunk after a
    # trial step until the whole run (warm-up and timed steps) fits the time
    # budget (two minutes by default).  The trial step is the first warm-up
    # step.  A step has a floor (one column, one row of x), so very many steps
    # can still overrun the budget.
    budget_s = args.ref_seconds
    cols, rows = args.ref_cols, None
    for _ in range(8):
        calls = oracle_calls(wl, cols, rows)
        t0 = time.perf_counter()
        oracle_step(wl, calls)
        projected = (time.perf_counter() - t0) * (args.steps + args.warmup)
        if projected <= budget_s:
            break
        f = budget_s / projected
        if cols > 1:
            cols = max(1, int(cols * f))
        elif rows != 1:
            rows = max(1, int((rows or max(wl["Ms"])) * f))
        else:
            break
    bytes_step = sum(c[2] for c in calls) * wl["experts"]
    threads = oracle.num_threads()
    for _ in range(max(args.warmup, 3) - 1):      # the other untimed warm-up steps
        oracle_step(wl, calls)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, calls)
    elapsed = time.perf_counter() - t0
    gbs = bytes_step * args.steps / elapsed / 1e9
    sample = ("%d of each weight's columns (all K rows, %s of x, M in %s) per call, fp64 oracle "
              "(quantize once, then dequantize + fp64 matmul per call)"
              % (cols, "all rows" if rows is None else "the first %d rows" % rows, wl["Ms"]))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4),
        "unit": "GB/s (weight stream)", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * elapsed / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64; x~N(0,1), W~N(0,0.02) fp16)",
        "config": {"workload": args.workload, "group": GROUP,
                   "shapes": wl["shapes"], "Ms": wl["Ms"], "experts": wl["experts"]},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s (weight stream)",
                         "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s (weight stream)",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- GPU
def timed_replays(graph, stream, reps, calls_per_replay):
    """Microseconds per call of `reps` replays of a graph holding
    `calls_per_replay` calls, each replay bracketed by events on `stream`
    (replay() launches on the current stream, so `stream` is made current)."""
    import torch
    out = []
    with torch.cuda.stream(stream):
        graph.replay()                       # upload + warm
        stream.synchronize()
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b) * 1e3 / calls_per_replay)
    return out


def timed_eager(calls, stream, reps):
    """Microseconds per call of `reps` rounds of the `calls` issued one by one
    (no graph), each round bracketed by events on `stream`."""
    import torch
    out = []
    with torch.cuda.stream(stream):
        for c in calls:                      # warm
            c()
        stream.synchronize()
        for _ in range(reps):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for c in calls:
                c()
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b) * 1e3 / len(calls))
    return out


def run_ours(args, rank, local, world, pg):
    import numpy as np
    import torch

    import weight_only_int4_codes_gb300 as w4
    from weight_only_int4_codes_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w4.load_library()
    wl = WORKLOADS[args.workload]
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    stream = torch.cuda.Stream(device=dev)
    gemm_cfg = dict(pdl=not args.no_pdl)
    if args.variant != "auto":
        gemm_cfg.update(path="decode", variant=args.variant)
    # MoE workloads: by default one grouped launch per (shape, M) covers all
    # experts (w4a16_gemm_grouped); --no-grouped issues one call per expert
    E = wl["experts"]
    grouped = E > 1 and not args.no_grouped
    group_cfg = dict(pdl=not args.no_pdl)

    # weights: quantize once per shape on the GPU (offline step), then R
    # byte-identical copies at distinct addresses per shape so that the
    # rotation's footprint exceeds 3x L2.
    shapes = []
    for si, (K, N) in enumerate(wl["shapes"]):
        W = synth.weight(K, N, seed=synth.weight_seed(wl["config"], shape_index=si) + 7919 * rank,
                         outliers=wl["outliers"])
        Wd = torch.from_numpy(W).to(dev)
        base = w4.quantize_pack(Wd, GROUP)
        wdq = w4.dequantize(*base, group=GROUP) if args.cublas else None
        del Wd
        per_copy = weight_bytes(K, N)
        R = max(2, math.ceil(3 * l2 / per_copy) + 1)
        copies = [tuple(t.clone() for t in base) for _ in range(R)]
        dq_copies = None
        if wdq is not None:
            Rq = max(2, math.ceil(3 * l2 / (2 * K * N)) + 1)
            dq_copies = [wdq.clone() for _ in range(Rq)]
        xs = {}
        outs = {}
        xg, og = {}, {}
        for M in wl["Ms"]:
            x = synth.activations(M, K, seed=synth.x_seed(wl["config"], M, shape_index=si))
            xs[M] = torch.from_numpy(x).to(dev)
            outs[M] = torch.empty((M, N), dtype=torch.float16, device=dev)
            if grouped:
                # distinct activations per expert, stacked [E, M, K]
                xg[M] = torch.from_numpy(np.stack([
                    synth.activations(M, K, seed=synth.x_seed(wl["config"], M, expert=e,
                                                              shape_index=si))
                    for e in range(E)])).to(dev)
                og[M] = torch.empty((E, M, N), dtype=torch.float16, device=dev)
        shapes.append(dict(K=K, N=N, copies=copies, dq=dq_copies, xs=xs, outs=outs, xg=xg,
                           og=og))
    torch.cuda.synchronize(dev)

    if grouped:
        calls_per_step = [(s, M) for s in shapes for M in wl["Ms"]]
        per_call = E                   # GEMMs (experts) per launch
    else:
        calls_per_step = [(s, M) for s in shapes for M in wl["Ms"]] * E
        per_call = 1
    step_weight_bytes = per_call * sum(weight_bytes(s["K"], s["N"]) for s, _ in calls_per_step)
    step_total_bytes = per_call * sum(total_bytes(M, s["K"], s["N"]) for s, M in calls_per_step)
    counters = {id(s): 0 for s in shapes}

    def grouped_call(s, M, api=False):
        """One launch over E experts, each reading the next distinct weight copy."""
        R = len(s["copies"])
        i = counters[id(s)]
        counters[id(s)] = (i + E) % R
        ws = [s["copies"][(i + e) % R] for e in range(E)]
        w4.gemm_grouped(s["xg"][M], [w[0] for w in ws], [w[1] for w in ws], [w[2] for w in ws],
                        group=GROUP, out=s["og"][M], config=None if api else group_cfg)

    def one_step():
        for s, M in calls_per_step:
            if grouped:
                grouped_call(s, M)
                continue
            i = counters[id(s)]
            counters[id(s)] = (i + 1) % len(s["copies"])
            w4.gemm_ex(s["xs"][M], *s["copies"][i], group=GROUP, out=s["outs"][M],
                       config=gemm_cfg)

    # warm-up (eager, also loads the kernels and fills the plan cache)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize(dev)

    # capture exactly `steps` steps in one graph
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(args.steps):
            one_step()
    with torch.cuda.stream(stream):
        graph.replay()                 # untimed replay (graph upload)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(pg)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if clocks:
        clocks.mark_start()
    with torch.cuda.stream(stream):          # replay() launches on the current stream
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.mark_end()
    barrier(pg)
    clock_rec = clocks.stop() if clocks else None
    ms = ev0.elapsed_time(ev1)
    ms = reduce_max(pg, ms, dev)
    ms_step = ms / args.steps
    gbs = world * step_weight_bytes * args.steps / (ms * 1e-3) / 1e9

    # ---- per-M microseconds per call (graphs of R rotating calls), and cuBLAS
    per_m = {}
    for si, s in enumerate(shapes):
        for M in wl["Ms"]:
            R = len(s["copies"])
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(R):
                    w4.gemm_ex(s["xs"][M], *s["copies"][i], group=GROUP, out=s["outs"][M],
                               config=gemm_cfg)
            ts = timed_replays(g, stream, args.reps, R)
            us = statistics.median(ts)
            K, N = s["K"], s["N"]
            calls = [lambda i=i: w4.gemm_ex(s["xs"][M], *s["copies"][i], group=GROUP,
                                            out=s["outs"][M], config=gemm_cfg)
                     for i in range(R)]
            us_eager = statistics.median(timed_eager(calls, stream, args.reps))
            rec = {"us_per_call": round(us, 3),
                   "us_per_call_eager": round(us_eager, 3),
                   "weight_GBs": round(weight_bytes(K, N) / us / 1e3, 1),
                   "packed_GBs": round(K * N // 2 / us / 1e3, 1),
                   "total_GBs": round(total_bytes(M, K, N) / us / 1e3, 1),
                   "roofline_frac": round(max(total_bytes(M, K, N) / (peaks["hbm_gbs"] * 1e9),
                                              2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12))
                                          / (us * 1e-6), 4)}
            if s["dq"] is not None:
                Rq = len(s["dq"])
                with torch.cuda.stream(stream):       # cuBLAS handle/workspace outside capture
                    torch.matmul(s["xs"][M], s["dq"][0], out=s["outs"][M])
                torch.cuda.synchronize(dev)
                gq = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gq, stream=stream):
                    for i in range(Rq):
                        torch.matmul(s["xs"][M], s["dq"][i], out=s["outs"][M])
                tq = timed_replays(gq, stream, args.reps, Rq)
                rec["cublas_fp16_us_per_call"] = round(statistics.median(tq), 3)
                rec["speedup_vs_cublas"] = round(rec["cublas_fp16_us_per_call"] / us, 3)
            if grouped:
                # one grouped launch per E experts (all distinct weight copies)
                nG = max(1, R // E)
                gg = torch.cuda.CUDAGraph()
                counters[id(s)] = 0
                with torch.cuda.graph(gg, stream=stream):
                    for _ in range(nG):
                        grouped_call(s, M)
                tg = statistics.median(timed_replays(gg, stream, args.reps, nG))
                rec["grouped_us_per_%d_experts" % E] = round(tg, 3)
                rec["grouped_weight_GBs"] = round(E * weight_bytes(K, N) / tg / 1e3, 1)
                rec["grouped_roofline_frac"] = round(
                    E * total_bytes(M, K, N) / (peaks["hbm_gbs"] * 1e9) / (tg * 1e-6), 4)
                rec["grouped_speedup_vs_%d_calls" % E] = round(E * us / tg, 2)
            key = "M=%d" % M if len(shapes) == 1 else "K=%d,N=%d,M=%d" % (K, N, M)
            per_m[key] = rec

    # ---- end to end through the public API: x from pinned host memory and
    # the result back to pinned host memory every call; weights resident.
    h2d = per_call * sum(2 * M * s["K"] for s, M in calls_per_step)
    d2h = per_call * sum(2 * M * s["N"] for s, M in calls_per_step)
    xkey, okey = ("xg", "og") if grouped else ("xs", "outs")
    host_x = {(id(s), M): s[xkey][M].cpu().pin_memory() for s in shapes for M in wl["Ms"]}
    host_o = {(id(s), M): torch.empty_like(s[okey][M], device="cpu").pin_memory()
              for s in shapes for M in wl["Ms"]}
    e2e_steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        def e2e_step():
            for s, M in calls_per_step:
                s[xkey][M].copy_(host_x[(id(s), M)], non_blocking=True)
                if grouped:
                    grouped_call(s, M, api=True)
                else:
                    i = counters[id(s)]
                    counters[id(s)] = (i + 1) % len(s["copies"])
                    w4.gemm(s["xs"][M], *s["copies"][i], group=GROUP, out=s["outs"][M])
                host_o[(id(s), M)].copy_(s[okey][M], non_blocking=True)
            stream.synchronize()
        e2e_step()
        barrier(pg)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(pg, e2e_s, dev)
    e2e_gbs = world * step_weight_bytes * e2e_steps / e2e_s / 1e9

    # ---- roofline of the dominant kernel, from the timed region: every launch
    # in it is one of the workload's GEMM kernels.  Decode shapes are bound by
    # HBM (algorithmic bytes per launch / mean launch time); the prefill sweep
    # by the fp16 tensor cores (fp16 and bf16 dense rates are equal on GB300).
    launches = len(calls_per_step) * args.steps
    mean_launch_s = ms * 1e-3 / launches
    if workload_kind(args.workload) == "prefill":
        step_flops = sum(2.0 * M * s["K"] * s["N"] for s, M in calls_per_step)
        achieved = step_flops / len(calls_per_step) / mean_launch_s / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "traffic": ncu_traffic(args.workload),
                    "peak_source": (peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops_sustained: "
                                    "a seconds-long step)") if peaks["source"] == "measured"
                    else "fallback 1700 TFLOP/s sustained"}
    else:
        alg_bytes_launch = step_total_bytes / len(calls_per_step)
        achieved = alg_bytes_launch / mean_launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": ncu_traffic(args.workload),
                    "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                    if peaks["source"] == "measured" else "fallback 6800 GB/s"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        sec, b, threads = oracle_sample(wl, args.ref_cols, args.cpu_seconds)
        cpu = {"value": round(b / sec / 1e9, 4), "unit": "GB/s (weight stream)",
               "cores": threads, "kind": "oracle",
               "sample": "%d of each weight's columns, every call of one step, repeated for "
                         ">= %.0f s (median step)" % (args.ref_cols, args.cpu_seconds)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s (weight stream)",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
            "data": "synthetic (seeded numpy PCG64; x~N(0,1), W~N(0,0.02) fp16, "
                    "quantized on the GPU)",
            "config": {"workload": args.workload, "group": GROUP, "shapes": wl["shapes"],
                       "Ms": wl["Ms"], "experts": wl["experts"],
                       "l2": "inputs larger than L2: every call reads a distinct weight copy "
                             "(rotation footprint >= 3x L2)",
                       "timing": "one CUDA-graph replay of exactly `steps` steps, CUDA events",
                       "pdl": not args.no_pdl, "variant": args.variant,
                       "launch": ("grouped: one launch per (shape, M) over %d experts" % E)
                       if grouped else "one call per GEMM",
                       "parallelism": "replicas" if world > 1 else "1gpu"},
            "us_per_call": per_m,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s (weight stream)",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "public API call per GEMM, x copied from pinned host memory and out "
                            "copied back every call, weights resident in HBM"},
            "gpu_launches": launches,
            "clocks": clock_rec,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode_square")
    ap.add_argument("--reps", type=int, default=20, help="repeats of the per-M timing graphs")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-grouped", action="store_true",
                    help="MoE workload: one call per expert instead of one grouped launch")
    ap.add_argument("--variant", choices=["auto", "tma", "registers"], default="auto",
                    help="decode kernel variant (auto = the library's dispatch)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cublas", action=argparse.BooleanOptionalAction, default=True)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only-shape", type=int, default=None,
                    help="profiling aid: keep only this shape index of the workload")
    ap.add_argument("--only-m", type=int, default=None,
                    help="profiling aid: keep only this M of the workload")
    ap.add_argument("--ref-cols", type=int, default=256)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: time budget of the whole run (the sample shrinks to fit)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    if args.only_shape is not None or args.only_m is not None:
        wl = dict(WORKLOADS[args.workload])
        if args.only_shape is not None:
            wl["shapes"] = [wl["shapes"][args.only_shape]]
        if args.only_m is not None:
            wl["Ms"] = [args.only_m]
        WORKLOADS[args.workload] = wl
    rank, local, world, pg = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world, pg)
    else:
        run_ours(args, rank, local, world, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
