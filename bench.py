#!/usr/bin/env python3
"""Benchmark of the W4A16 GEMM hot path on GB300.

A step is one pass of the hot path over one batch of synthetic input.  The
default workload, `decode`, covers every decode configuration: the square
projection (K = N = 4096), the FFN projections (4096 x 14336 and 14336 x 4096,
with outliers) and the MoE expert shapes (2048 x 768 and 768 x 2048, 64 expert
weight sets called back to back on one stream), each at M = 1, 2, 4, 8, 16,
group 128: one W4A16 GEMM call per (shape, M, expert).  Every call reads a
distinct copy of its weights (the rotation of copies exceeds three times the
L2), so the weight stream always comes from HBM.  The timed region is the
requested number of steps, run as replays of one CUDA graph per configuration
(programmatic dependent launch inside), every replay bracketed by CUDA events
on the capture stream; per-configuration times come from the same events.

Printed: one JSON line (rank 0).  `value` is the weight-stream bandwidth of the
whole job (packed words + scales + zeros of every call, all ranks) over the
timed region.  Beside it: per-shape microseconds per call (CUDA graph and eager
launches), GB/s and roofline fractions, a cuBLAS fp16 reference (torch.matmul on
the dequantized weight), the same GEMMs in bfloat16, with groups of 64 and 256
rows (M = 1), and on the repacked weight layout, the 64 experts of a MoE shape in
one grouped launch (natural and repacked weights),
the streaming-read ceiling of a launch of the same size in the same launch
chain, the fp64 oracle on the host cores (`cpu_baseline`), and `e2e`: the step
through the public API (prepared calls) with all of its activations copied
from pinned host memory in one transfer and all results copied back in one.

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
DECODE_MS = [1, 2, 4, 8, 16]
PREFILL_MS = [16, 32, 64, 128, 256, 1024, 4096]

# configuration -> its shapes; si = index of the shape within the configuration
# (it picks the seeds of that shape's weights and activations)
CONFIGS = {
    "decode_square": [dict(K=4096, N=4096, config=1, si=0, outliers=False, experts=1)],
    "decode_ffn": [dict(K=4096, N=14336, config=2, si=0, outliers=True, experts=1),
                   dict(K=14336, N=4096, config=2, si=1, outliers=True, experts=1)],
    "moe_experts": [dict(K=2048, N=768, config=3, si=0, outliers=False, experts=64),
                    dict(K=768, N=2048, config=3, si=1, outliers=False, experts=64)],
    "prefill_sweep": [dict(K=4096, N=14336, config=4, si=0, outliers=False, experts=1),
                      dict(K=8192, N=28672, config=4, si=1, outliers=False, experts=1)],
}
# workload -> the configurations its step runs, and the batch rows
WORKLOADS = {
    "decode": dict(configs=["decode_square", "decode_ffn", "moe_experts"], Ms=DECODE_MS),
    "decode_square": dict(configs=["decode_square"], Ms=DECODE_MS),
    "decode_ffn": dict(configs=["decode_ffn"], Ms=DECODE_MS),
    "moe_experts": dict(configs=["moe_experts"], Ms=DECODE_MS),
    "prefill_sweep": dict(configs=["prefill_sweep"], Ms=PREFILL_MS),
}


def shapes_of(wl):
    return [dict(sh, cfg=c) for c in wl["configs"] for sh in CONFIGS[c]]


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


# The sources each kind of workload's kernels are built from: a committed ncu
# summary is used only while these are unchanged.
KERNEL_SOURCES = {
    "decode": ["api.cu", "common.cuh", "decode.cu", "decode_math.cuh", "decode_tma.cu",
               "decode_warp.cu", "sm100_ptx.cuh", "tmap.cu", "tmap.cuh"],
    "prefill": ["api.cu", "common.cuh", "prefill.cu", "prefill_tile.cuh", "sm100_ptx.cuh",
                "tcgen05.cuh", "tmap.cu", "tmap.cuh"],
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


def ncu_traffic(name):
    """Per-launch DRAM bytes of a configuration's kernels from the committed ncu
    summary, or None when absent or taken on a different kernel source."""
    kind = workload_kind(name)
    path = os.path.join(ROOT, "profiles", "%s_kernel_%s.txt" % (kind, name))
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
    first `rows` rows when given); each entry runs once per expert."""
    import oracle
    from weight_only_int4_codes_gb300 import synth
    calls = []
    for sh in shapes_of(wl):
        K, N = sh["K"], sh["N"]
        n = min(cols, N)
        W = synth.weight(K, n, seed=synth.weight_seed(sh["config"], shape_index=sh["si"]),
                         outliers=sh["outliers"])
        qw = oracle.quantize_pack(W, GROUP)
        for M in wl["Ms"]:
            x = synth.activations(M, K, seed=synth.x_seed(sh["config"], M, shape_index=sh["si"]))
            if rows is not None:
                x = x[:rows]
            calls.append((x, qw, weight_bytes(K, n), sh["experts"]))
    return calls


def oracle_step(calls):
    import oracle
    for x, qw, _b, experts in calls:
        for _ in range(experts):
            oracle.gemm(x, *qw, group=GROUP)


def step_bytes(calls):
    return sum(b * e for _x, _q, b, e in calls)


def oracle_sample(wl, cols, reps_min_s):
    """Time the fp64 oracle on a column sample of every call of one step,
    repeated for at least `reps_min_s` seconds.  Returns (median seconds per
    sampled step, weight bytes per sampled step, threads used)."""
    import oracle
    calls = oracle_calls(wl, cols)
    oracle_step(calls)                           # warm (library load, page faults)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle_step(calls)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= reps_min_s:
            break
    return statistics.median(times), step_bytes(calls), oracle.num_threads()


def config_obj(args, world):
    """The `config` object both arms print (the same keys and values)."""
    wl = WORKLOADS[args.workload]
    return {"workload": args.workload, "group": GROUP,
            "shapes": [[sh["K"], sh["N"]] for sh in shapes_of(wl)],
            "experts": [sh["experts"] for sh in shapes_of(wl)], "Ms": wl["Ms"],
            "l2": "inputs larger than L2: every call reads a distinct weight copy (rotation "
                  "footprint >= 3x L2)",
            "timing": "replays of one CUDA graph per configuration, each bracketed by CUDA "
                      "events; value over the sum",
            "pdl": not args.no_pdl,
            "launch": "one call per GEMM (MoE: 64 expert calls back to back per shape and M)",
            "parallelism": "replicas" if world > 1 else "1gpu"}


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
        oracle_step(calls)
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
    bytes_step = step_bytes(calls)
    threads = oracle.num_threads()
    for _ in range(max(args.warmup, 3) - 1):      # the other untimed warm-up steps
        oracle_step(calls)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(calls)
    elapsed = time.perf_counter() - t0
    gbs = bytes_step * args.steps / elapsed / 1e9
    sample = ("%d of each weight's columns (all K rows, %s of x, M in %s) per call, every call "
              "of the step, fp64 oracle (quantize once, then dequantize + fp64 matmul per call)"
              % (cols, "all rows" if rows is None else "the first %d rows" % rows, wl["Ms"]))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4),
        "unit": "GB/s (weight stream)", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * elapsed / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64; x~N(0,1), W~N(0,0.02) fp16)",
        "config": config_obj(args, world),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s (weight stream)",
                         "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s (weight stream)",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- GPU
def graph_of(fns, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in fns:
            f()
    return g


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


def steps_per_replay(steps, calls_per_step, max_nodes=8000, min_replays=20):
    """Steps per graph replay: the largest divisor of `steps` that leaves at
    least `min_replays` replays and at most `max_nodes` launches per graph."""
    best = 1
    for d in range(1, steps + 1):
        if steps % d == 0 and steps // d >= min(min_replays, steps) and \
                d * calls_per_step <= max_nodes:
            best = d
    return best


def run_ours(args, rank, local, world, pg):
    import numpy as np
    import torch

    import weight_only_int4_codes_gb300 as w4
    from weight_only_int4_codes_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w4.load_library()
    wl = WORKLOADS[args.workload]
    Ms = wl["Ms"]
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.Stream(device=dev)
    gemm_cfg = dict(pdl=not args.no_pdl)
    if args.variant != "auto":
        gemm_cfg.update(path="decode", variant=args.variant)
    decode = workload_kind(args.workload) == "decode"

    # weights: quantize once per shape on the GPU (offline step), then R
    # byte-identical copies at distinct addresses per shape so that the
    # rotation's footprint exceeds 3x L2; the same for the repacked layout
    shapes = []
    for sh in shapes_of(wl):
        K, N, E = sh["K"], sh["N"], sh["experts"]
        W = synth.weight(K, N, seed=synth.weight_seed(sh["config"], shape_index=sh["si"]) +
                         7919 * rank, outliers=sh["outliers"])
        Wd = torch.from_numpy(W).to(dev)
        base = w4.quantize_pack(Wd, GROUP)
        wdq = w4.dequantize(*base, group=GROUP) if args.cublas else None
        R = max(2, math.ceil(3 * l2 / weight_bytes(K, N)) + 1)
        copies = [tuple(t.clone() for t in base) for _ in range(R)]
        # extras: the same weight quantized in bfloat16, and (decode) with
        # groups of 64 and 256 rows, R copies each
        bf16_copies, group_copies = None, {}
        if not args.no_extras:
            base_b = w4.quantize_pack_bf16(Wd.bfloat16(), GROUP)
            bf16_copies = [tuple(t.clone() for t in base_b) for _ in range(R)]
            if workload_kind(args.workload) == "decode":
                for gsz in (64, 256):
                    bg = w4.quantize_pack(Wd, gsz)
                    group_copies[gsz] = [tuple(t.clone() for t in bg) for _ in range(R)]
        del Wd
        rep_ok = decode and w4.repacked_bytes(K, N, GROUP) > 0 and not args.no_extras
        repacked = [w4.repack(*c, group=GROUP) for c in copies] if rep_ok else None
        dq = None
        if wdq is not None:
            Rq = max(2, math.ceil(3 * l2 / (2 * K * N)) + 1)
            dq = [wdq.clone() for _ in range(Rq)]
        xs, outs = {}, {}
        for M in Ms:
            # distinct activations per expert, stacked [E, M, K]
            xs[M] = torch.from_numpy(np.stack([
                synth.activations(M, K, seed=synth.x_seed(sh["config"], M, expert=e,
                                                          shape_index=sh["si"]))
                for e in range(E)])).to(dev)
            outs[M] = torch.empty((E, M, N), dtype=torch.float16, device=dev)
        shapes.append(dict(sh, copies=copies, repacked=repacked, dq=dq, xs=xs, outs=outs,
                           bf16_copies=bf16_copies, group_copies=group_copies))
    # the activations and outputs of every (shape, M) live in two flat arenas,
    # so that the end-to-end step moves all of its inputs with one
    # host->device copy and all of its results with one device->host copy
    x_arena = torch.empty(sum(v.numel() for s in shapes for v in s["xs"].values()),
                          dtype=torch.float16, device=dev)
    o_arena = torch.empty(sum(v.numel() for s in shapes for v in s["outs"].values()),
                          dtype=torch.float16, device=dev)
    xo = oo = 0
    for s in shapes:
        for M in Ms:
            n = s["xs"][M].numel()
            assert n % 8 == 0 and s["outs"][M].numel() % 8 == 0   # 16-byte aligned views
            v = x_arena[xo:xo + n].view(s["xs"][M].shape)
            v.copy_(s["xs"][M])
            s["xs"][M] = v
            xo += n
            n = s["outs"][M].numel()
            s["outs"][M] = o_arena[oo:oo + n].view(s["outs"][M].shape)
            oo += n
    torch.cuda.synchronize(dev)

    counters = {}

    def call_fns(s, M, api=False, cfg=None):
        """The step's calls of one (shape, M): one per expert, each reading the
        next distinct weight copy."""
        fns = []
        for e in range(s["experts"]):
            R = len(s["copies"])
            i = counters.get(id(s), 0)
            counters[id(s)] = (i + 1) % R
            w = s["copies"][i]
            x, o = s["xs"][M][e], s["outs"][M][e]
            if api:
                # the public API's reusable call (arguments marshalled once),
                # with the timed region's configuration
                fns.append(w4.prepare_gemm(x, *w, group=GROUP, out=o, config=cfg or gemm_cfg))
            else:
                fns.append(lambda x=x, w=w, o=o: w4.gemm_ex(x, *w, group=GROUP, out=o,
                                                            config=cfg or gemm_cfg))
        return fns

    def part_fns(cfgname, steps):
        fns = []
        for _ in range(steps):
            for s in shapes:
                if s["cfg"] == cfgname:
                    for M in Ms:
                        fns += call_fns(s, M)
        return fns

    calls_per_step = {c: sum(s["experts"] * len(Ms) for s in shapes if s["cfg"] == c)
                      for c in wl["configs"]}
    wbytes_step = {c: sum(s["experts"] * len(Ms) * weight_bytes(s["K"], s["N"])
                          for s in shapes if s["cfg"] == c) for c in wl["configs"]}
    tbytes_step = {c: sum(s["experts"] * total_bytes(M, s["K"], s["N"])
                          for s in shapes if s["cfg"] == c for M in Ms) for c in wl["configs"]}
    flops_step = {c: sum(s["experts"] * 2.0 * M * s["K"] * s["N"]
                         for s in shapes if s["cfg"] == c for M in Ms) for c in wl["configs"]}

    # warm-up steps (eager: also loads the kernels and fills the plan caches)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for c in wl["configs"]:
                for f in part_fns(c, 1):
                    f()
    torch.cuda.synchronize(dev)

    # the timed region: `steps` steps as replays of one graph per configuration
    spr = steps_per_replay(args.steps, max(calls_per_step.values()))
    replays = args.steps // spr
    graphs = {c: graph_of(part_fns(c, spr), stream) for c in wl["configs"]}
    with torch.cuda.stream(stream):
        for g in graphs.values():
            g.replay()                      # untimed replay (graph upload)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(pg)
    torch.cuda.synchronize(dev)
    evs = []
    if clocks:
        clocks.mark_start()
    with torch.cuda.stream(stream):          # replay() launches on the current stream
        for _ in range(replays):
            for c in wl["configs"]:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graphs[c].replay()
                b.record(stream)
                evs.append((c, a, b))
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.mark_end()
    barrier(pg)
    clock_rec = clocks.stop() if clocks else None
    part_ms = {c: 0.0 for c in wl["configs"]}
    replay_ms = []
    for i in range(0, len(evs), len(wl["configs"])):
        t = 0.0
        for c, a, b in evs[i:i + len(wl["configs"])]:
            ms_ = a.elapsed_time(b)
            part_ms[c] += ms_
            t += ms_
        replay_ms.append(t)
    ms = sum(replay_ms)
    ms = reduce_max(pg, ms, dev)
    for c in part_ms:
        part_ms[c] = reduce_max(pg, part_ms[c], dev)
    ms_step = ms / args.steps
    step_weight_bytes = sum(wbytes_step.values())
    gbs = world * step_weight_bytes * args.steps / (ms * 1e-3) / 1e9
    launches = sum(calls_per_step.values()) * args.steps
    per_config = {}
    for c in wl["configs"]:
        t_s = part_ms[c] * 1e-3
        per_config[c] = {
            "ms_in_timed_region": round(part_ms[c], 3),
            "weight_GBs": round(world * wbytes_step[c] * args.steps / t_s / 1e9, 1),
            "us_per_call": round(part_ms[c] * 1e3 / (calls_per_step[c] * args.steps), 3),
            "roofline_frac": round(tbytes_step[c] * args.steps / t_s / (peaks["hbm_gbs"] * 1e9), 4)
            if decode else round(flops_step[c] * args.steps / t_s /
                                 (peaks["bf16_tflops_sustained"] * 1e12), 4),
        }

    # ---- per shape and M: graphs of R rotating calls (every weight copy once)
    def one_graph_us(fns, n_calls, reps=args.reps):
        return statistics.median(timed_replays(graph_of(fns, stream), stream, reps, n_calls))

    sink = torch.zeros(max(n_sm, 1024), dtype=torch.int32, device=dev)
    per_m = {}
    for s in shapes:
        K, N, E = s["K"], s["N"], s["experts"]
        R = len(s["copies"])
        tb = lambda M: total_bytes(M, K, N)
        frac = lambda M, us: max(tb(M) / (peaks["hbm_gbs"] * 1e9),
                                 2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12)) / (us * 1e-6)
        for M in Ms:
            x, o = s["xs"][M][0], s["outs"][M][0]
            fns = [lambda i=i: w4.gemm_ex(x, *s["copies"][i], group=GROUP, out=o, config=gemm_cfg)
                   for i in range(R)]
            us = one_graph_us(fns, R)
            eager = [w4.prepare_gemm(x, *s["copies"][i], group=GROUP, out=o, config=gemm_cfg)
                     for i in range(R)]
            us_eager = statistics.median(timed_eager(eager, stream, args.reps))
            rec = {"us_per_call": round(us, 3), "us_per_call_eager": round(us_eager, 3),
                   "weight_GBs": round(weight_bytes(K, N) / us / 1e3, 1),
                   "packed_GBs": round(K * N // 2 / us / 1e3, 1),
                   "total_GBs": round(tb(M) / us / 1e3, 1),
                   "roofline_frac": round(frac(M, us), 4)}
            if s["dq"] is not None:
                Rq = len(s["dq"])
                with torch.cuda.stream(stream):       # cuBLAS handle/workspace outside capture
                    torch.matmul(x, s["dq"][0], out=o)
                torch.cuda.synchronize(dev)
                tq = one_graph_us([lambda i=i: torch.matmul(x, s["dq"][i], out=o)
                                   for i in range(Rq)], Rq)
                rec["cublas_fp16_us_per_call"] = round(tq, 3)
                rec["speedup_vs_cublas"] = round(tq / us, 3)
            if s["bf16_copies"] is not None:
                # the bfloat16 variant: bf16 x, scales, zeros and out
                xb = x.bfloat16()
                ob = torch.empty(o.shape, dtype=torch.bfloat16, device=dev)
                ub16 = one_graph_us([lambda i=i: w4.gemm_ex(
                    xb, *s["bf16_copies"][i], group=GROUP, out=ob, config=gemm_cfg)
                    for i in range(R)], R)
                rec["bf16_us_per_call"] = round(ub16, 3)
                rec["bf16_roofline_frac"] = round(frac(M, ub16), 4)
            if decode and M == 1 and s["group_copies"]:
                # other group sizes (same weight, M = 1)
                for gsz, cps in s["group_copies"].items():
                    wb_g = K * N // 2 + 4 * (K // gsz) * N + 2 * K + 2 * N
                    ug = one_graph_us([lambda i=i, cps=cps, gsz=gsz: w4.gemm_ex(
                        x, *cps[i], group=gsz, out=o, config=gemm_cfg) for i in range(R)], R)
                    rec["group%d_us_per_call" % gsz] = round(ug, 3)
                    rec["group%d_roofline_frac" % gsz] = round(
                        wb_g / (peaks["hbm_gbs"] * 1e9) / (ug * 1e-6), 4)
            if decode and not args.no_extras:
                if s["repacked"] is not None:
                    ur = one_graph_us([lambda i=i: w4.gemm_repacked(
                        x, s["repacked"][i], N, group=GROUP, out=o, config=gemm_cfg)
                        for i in range(R)], R)
                    rec["repacked_us_per_call"] = round(ur, 3)
                    rec["repacked_roofline_frac"] = round(frac(M, ur), 4)
                # the streaming-read ceiling: a chain of launches reading the
                # same weight bytes the same way, doing no arithmetic
                ucs = one_graph_us([lambda i=i: w4.native.stream_read(
                    s["copies"][i][0], sink, pdl=not args.no_pdl) for i in range(R)], R)
                rec["stream_read_us"] = round(ucs, 3)
                rec["stream_read_GBs"] = round(K * N // 2 / ucs / 1e3, 1)
                rec["stream_read_frac"] = round(K * N // 2 / (peaks["hbm_gbs"] * 1e9) /
                                                (ucs * 1e-6), 4)
                if E > 1:
                    nG = max(1, R // E)
                    grp = [lambda j=j: w4.gemm_grouped(
                        s["xs"][M], *[[s["copies"][(j * E + e) % R][t] for e in range(E)]
                                      for t in range(3)],
                        group=GROUP, out=s["outs"][M], config=gemm_cfg) for j in range(nG)]
                    tg = one_graph_us(grp, nG)
                    rec["grouped_us_per_%d_experts" % E] = round(tg, 3)
                    rec["grouped_roofline_frac"] = round(E * tb(M) / (peaks["hbm_gbs"] * 1e9) /
                                                         (tg * 1e-6), 4)
                    if s["repacked"] is not None:
                        grr = [lambda j=j: w4.gemm_grouped_repacked(
                            s["xs"][M], [s["repacked"][(j * E + e) % R] for e in range(E)], N,
                            group=GROUP, out=s["outs"][M], config=gemm_cfg) for j in range(nG)]
                        tr = one_graph_us(grr, nG)
                        rec["grouped_repacked_us_per_%d_experts" % E] = round(tr, 3)
                        rec["grouped_repacked_roofline_frac"] = round(
                            E * tb(M) / (peaks["hbm_gbs"] * 1e9) / (tr * 1e-6), 4)
                    rec["single_calls_us_per_%d_experts" % E] = round(E * us, 3)
            per_m["K=%d,N=%d,M=%d" % (K, N, M)] = rec

    # ---- end to end through the public API: every step copies all of its
    # activations from pinned host memory in one transfer, issues its calls
    # (prepared GEMM calls, configured as in the timed region), and reads all results back
    # into pinned host memory in one transfer; weights stay resident.
    h2d = x_arena.numel() * 2
    d2h = o_arena.numel() * 2
    host_x = x_arena.cpu().pin_memory()
    host_o = torch.empty(o_arena.numel(), dtype=torch.float16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    e2e_calls = [[f for s in shapes for M in Ms for f in call_fns(s, M, api=True)]
                 for _ in range(e2e_steps + 1)]
    with torch.cuda.stream(stream):
        def e2e_step(calls):
            x_arena.copy_(host_x, non_blocking=True)
            for f in calls:
                f()
            host_o.copy_(o_arena, non_blocking=True)
            stream.synchronize()
        e2e_step(e2e_calls[-1])
        barrier(pg)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(e2e_calls[i])
        e2e_s = time.perf_counter() - t0
    e2e_s = reduce_max(pg, e2e_s, dev)
    e2e_gbs = world * step_weight_bytes * e2e_steps / e2e_s / 1e9

    # ---- roofline of the dominant kernel: the configuration that takes most
    # of the timed region; its algorithmic bytes (flops) per launch over its
    # mean launch time, both from the timed region's events
    dom = max(wl["configs"], key=lambda c: part_ms[c])
    mean_launch_s = part_ms[dom] * 1e-3 / (calls_per_step[dom] * args.steps)
    if not decode:
        achieved = flops_step[dom] / calls_per_step[dom] / mean_launch_s / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "frac": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "traffic": ncu_traffic(dom), "kernel_of": dom,
                    "peak_source": (peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops_sustained: "
                                    "a seconds-long step)") if peaks["source"] == "measured"
                    else "fallback 1700 TFLOP/s sustained"}
    else:
        achieved = tbytes_step[dom] / calls_per_step[dom] / mean_launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": ncu_traffic(dom), "kernel_of": dom,
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
            "config": config_obj(args, world),
            "timed_region": {"replays": replays, "steps_per_replay": spr,
                             "replay_ms_median": round(statistics.median(replay_ms), 4),
                             "replay_ms_min": round(min(replay_ms), 4),
                             "replay_ms_max": round(max(replay_ms), 4)},
            "per_config": per_config,
            "us_per_call": per_m,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_gbs, 3), "unit": "GB/s (weight stream)",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "public API (prepared GEMM calls, the timed region's configuration) for every GEMM of "
                            "the step; all of the step's activations copied from pinned host "
                            "memory in one transfer before the calls and all results copied "
                            "back in one transfer after them; weights resident in HBM"},
            "gpu_launches": launches,
            "clocks": clock_rec,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--reps", type=int, default=20, help="repeats of the per-shape timing graphs")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--variant", choices=["auto", "tma", "registers", "stream"], default="auto",
                    help="decode kernel variant (auto = the library's dispatch)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the repacked, grouped and streaming-read fields")
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
            sh = shapes_of(wl)[args.only_shape]
            CONFIGS["_only"] = [{k: v for k, v in sh.items() if k != "cfg"}]
            wl["configs"] = ["_only"]
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
