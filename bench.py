#!/usr/bin/env python3
"""Throughput of the exact-attention forward on GB300, as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}] [--workload NAME]

A step is one full forward pass (one kernel launch) over the workload's whole
batch: by default B=1, H=16, N=16384, d=128, non-causal, bf16 inputs already
resident in device memory. Each timed step is bracketed by CUDA events on the
launching stream; L2 is flushed (a 256 MiB write) between timed steps, outside
the events. `e2e` times the same pass through the host-buffer C-ABI entry
(attn_fwd_host): pinned host Q, K, V in, O and LSE out, copies included.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of query rows of the same workload.

`--fp8` times the FP8 forward (attn_fwd_fp8: E4M3 Q, K, V with per-tensor
scales; two launches per step, the transpose of V and the attention kernel)
against the FP8 peak, taken as the measured bf16 peak times the nominal FP8 /
BF16 ratio of 2.

`--pass softmax` and `--pass layernorm` time the standalone streaming row
operations on their row workloads (`--workload` names one of
workloads.ROW_WORKLOADS) in GB/s of one read and one write of every element,
against the measured HBM copy bandwidth.

`--pass bwd` times the backward instead (attn_bwd: dQ, dK, dV from Q, K, V, O,
LSE and dO, three launches per step), counted as 2.5x the forward's FLOPs (five
GEMM-shaped products against the forward's two); its CPU baseline is the fp64
backward oracle on one (batch, head) at a reduced N.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the forward pass shards into independent (batch, head)
problems, so there is no data-path collective); rank 0 reports the units of
all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak at N=16K, d=128"
METRIC_BWD = "attention bwd TFLOP/s on 1 GB300 (2.5x forward FLOPs) and % of dense bf16 tensor peak"
BWD_FLOP_FACTOR = 2.5
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["attn_fwd_kernel.cuh", "sm103_ptx.cuh", "exp2_poly.h", "plan.h", "plan.cpp", "split_policy.cpp",
                  "attn_api.cu"]
# The sources each pass's recorded traffic depends on: an entry of the traffic file is used only
# while their hash is the one it was captured with.
PASS_SOURCES = {
    "fwd": KERNEL_SOURCES,
    "fp8": ["attn_fwd_fp8_kernel.cuh", "attn_fwd_kernel.cuh", "sm103_ptx.cuh", "exp2_poly.h", "plan.h", "plan.cpp",
            "split_policy.cpp", "attn_fp8_api.cu"],
    "bwd": ["attn_bwd_kernel.cuh", "sm103_ptx.cuh", "sm103_bulk.cuh", "plan.h", "attn_bwd_api.cu"],
    "rows": ["rowwise_kernels.cuh", "rowwise_api.cu"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=None, help="named workload (default: the long-sequence headline case)")
    ap.add_argument("--skip-e2e", action="store_true", help="omit the host-buffer end-to-end leg")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-oracle baseline leg")
    ap.add_argument("--keep-l2", action="store_true",
                    help="no L2 flush between steps: back-to-back launches whose DRAM counters (ncu, cache control "
                         "off) give a step's steady-state traffic; not a timing configuration")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target wall time of the CPU-baseline sample")
    ap.add_argument("--fp8", action="store_true", help="time the FP8 (E4M3) forward instead of the bf16 one")
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd", "softmax", "layernorm"], default="fwd",
                    help="time the forward (default, the headline metric), the backward, or a row operation")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- distributed helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def whole_job(units_per_rank: float, rank_seconds: list[float]) -> tuple[float, float]:
    """(total units / slowest rank's seconds, slowest seconds): the aggregate over ranks."""
    slowest = max(rank_seconds)
    return units_per_rank * len(rank_seconds) / slowest, slowest


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- measurement helpers
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0.0)) or None, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, None, "fallback"


def kernel_source_hash(kind: str = "fwd") -> str:
    h = hashlib.sha256()
    for f in PASS_SOURCES[kind]:
        with open(os.path.join(ROOT, "exact_long_sequence_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(key: str, kind: str = "fwd"):
    """DRAM bytes per launch (per step for two-launch row passes) from the committed ncu
    capture, or None if the pass's kernel sources changed since it was taken (or there is none)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(key)
    if not entry or entry.get("kernel_source_sha256") != kernel_source_hash(kind):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = []
        reasons = set()
        smax = None
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                smax = float(r[1])
            except ValueError:
                continue
            for n, v in zip(names, r[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle leg
def cpu_oracle_sample(w, target_seconds: float, seed: int = 0):
    """Time the fp64 oracle on a bounded sample of query rows of workload `w`.

    Returns (TFLOP/s, seconds, rows, threads, description). FLOPs of a sampled
    row are counted as the GPU's are: 4*N*d per row non-causal (2*N*d causal,
    the same half count), so the rate is comparable with the GPU number.
    """
    import numpy as np
    import torch

    import oracle
    from exact_long_sequence_gb300 import workloads

    oracle.build()
    threads = os.cpu_count() or 1
    # one (b, h) of the workload, seeded like the workload itself
    q, k, v = workloads.make_inputs(1, 1, w.N, w.d, w.seed, w.qk_dist, w.v_dist)
    flops_per_row = (2.0 if w.causal else 4.0) * w.N * w.d

    def timed(rows):
        r = workloads.sample_rows(1, w.N, rows, seed + w.seed).numpy()
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.causal, w.scale, rows=r, nthreads=threads)
        return time.perf_counter() - t0, r.shape[1]

    probe_rows = max(threads, 32)
    dt, n = timed(probe_rows)
    rows = int(min(w.N, max(probe_rows, probe_rows * target_seconds / max(dt, 1e-6))))
    dt, n = timed(rows)
    desc = (f"{n} random query rows of one (batch, head) of {w.name} (N={w.N}, d={w.d}, causal={w.causal}), "
            f"fp64, {threads} threads; rate = {flops_per_row:.3g} FLOP per row / wall time")
    return flops_per_row * n / dt / 1e12, dt, n, threads, desc


# ----------------------------------------------------------------------------- arms
def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    per_step = max(1.0, min(args.cpu_seconds, 90.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, per_step / 4)
    vals, secs = [], []
    desc, threads, rows = "", 0, 0
    for _ in range(args.steps):
        v, dt, rows, threads, desc = cpu_oracle_sample(w, per_step)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, "none (host CPU)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_note(args) -> str:
    if args.keep_l2:
        return "kept between steps (back-to-back launches for DRAM counter captures; not a timing configuration)"
    return f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, untimed)"


def workload_config(w, l2_note):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": w.scale, "inputs": f"seeded synthetic ({w.qk_dist} Q,K; {w.v_dist} V), bf16",
            "l2": l2_note, "parallelism": "replicas"}


def cpu_oracle_bwd_sample(w, target_seconds: float):
    """Time the fp64 backward oracle on one (batch, head) of workload `w` at a
    reduced N chosen to take about `target_seconds`. Returns (TFLOP/s, seconds,
    threads, description), FLOPs counted as the GPU's (2.5x the forward's)."""
    import oracle
    from exact_long_sequence_gb300 import workloads

    oracle.build()
    threads = os.cpu_count() or 1

    def timed(n):
        q, k, v = workloads.make_inputs(1, 1, n, w.d, w.seed, w.qk_dist, w.v_dist)
        do = workloads.make_inputs(1, 1, n, w.d, w.seed + 1000)[0]
        t0 = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, w.causal, w.scale, nthreads=threads)
        return time.perf_counter() - t0

    n = min(w.N, 512)
    dt = timed(n)
    while n < w.N and dt * 4 < target_seconds:  # cost grows as N^2
        n, dt = min(w.N, 2 * n), None
        dt = timed(n)
    flops = BWD_FLOP_FACTOR * (2.0 if w.causal else 4.0) * n * n * w.d
    desc = (f"full backward of one (batch, head) at N={n} (of {w.N}), d={w.d}, causal={w.causal}, fp64, "
            f"{threads} threads; rate = {flops:.3g} FLOP / wall time")
    return flops / dt / 1e12, dt, threads, desc


def cpu_oracle_fp8_sample(w, target_seconds: float, seed: int = 0):
    """Time the fp64 oracle of the FP8 forward (decode + forward) on sampled query rows
    of one (batch, head) of workload `w`. Returns (TFLOP/s, seconds, rows, threads, description)."""
    import oracle
    from exact_long_sequence_gb300 import workloads

    oracle.build()
    threads = os.cpu_count() or 1
    q8, k8, v8, sc = workloads.make_inputs_fp8(1, 1, w.N, w.d, w.seed, w.qk_dist, w.v_dist)
    flops_per_row = (2.0 if w.causal else 4.0) * w.N * w.d

    def timed(rows):
        r = workloads.sample_rows(1, w.N, rows, seed + w.seed).numpy()
        t0 = time.perf_counter()
        oracle.attention_fp8(q8, k8, v8, w.causal, w.scale, scales=sc, rows=r, nthreads=threads)
        return time.perf_counter() - t0, r.shape[1]

    probe_rows = max(threads, 32)
    dt, n = timed(probe_rows)
    rows = int(min(w.N, max(probe_rows, probe_rows * target_seconds / max(dt, 1e-6))))
    dt, n = timed(rows)
    desc = (f"{n} random query rows of one (batch, head) of {w.name} in E4M3 (N={w.N}, d={w.d}, "
            f"causal={w.causal}), decoded exactly, fp64, {threads} threads")
    return flops_per_row * n / dt / 1e12, dt, n, threads, desc


def run_gb300_fp8(args, w):
    import torch

    import exact_long_sequence_gb300 as ela
    from exact_long_sequence_gb300 import _build, workloads

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a); no CPU fallback exists")
    if w.d != 128:
        raise SystemExit("the FP8 forward supports d = 128 only")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(ela.LIB_PATH):
        _build.build()
    if world > 1:
        dist.barrier()
    ela.load_library()
    stream = torch.cuda.current_stream(dev)
    shape = (w.B, w.H, w.N, w.d)
    # The workload's seeded draws quantised per tensor to E4M3 (scale = max|x| / 448) on the host,
    # as the parity tests take them, then made resident in device memory.
    q8, k8, v8, scales = workloads.make_inputs_fp8(w.B, w.H, w.N, w.d, w.seed, w.qk_dist, w.v_dist)
    q8, k8, v8 = (t.to(dev) for t in (q8, k8, v8))
    o = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(ela.load_library().attn_fwd_fp8_workspace_bytes(*shape), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        ela.attn_fwd_fp8(q8, k8, v8, scales, causal=w.causal, scale=w.scale, out=o, lse=lse, workspace=ws,
                         stream=stream)
    torch.cuda.synchronize(dev)
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            if not args.keep_l2:
                flush.zero_()
            starts[i].record(stream)
            ela.attn_fwd_fp8(q8, k8, v8, scales, causal=w.causal, scale=w.scale, out=o, lse=lse, workspace=ws,
                             stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    slowest = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    value = w.flops * args.steps * world / slowest / 1e12
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak_bf16, peak_bf16_sustained, peak_kind = read_peaks()
    peak = 2.0 * peak_bf16
    # the V transpose and the attention kernel, plus the combine kernel of a K/V split
    # the V transpose and the attention kernel, plus the counter-zeroing kernel of the dynamic
    # schedule and the combine kernel of a K/V split
    choice = ela.split_choice(w.B, w.H, w.N, w.d, w.causal)
    fp8_launches = 2 + int(choice["dynamic"]) + int(choice["segs"] > 1)
    kernel_ms = statistics.mean(step_ms)
    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "peak_kind": (f"{peak_kind} dense bf16 burst (MEASURED_PEAKS.json) x 2, the nominal FP8/BF16 "
                              "tensor ratio (4.5 / 2.25 PFLOP/s)"),
                "traffic": recorded_traffic("fp8:" + w.name, "fp8"), "algorithmic_flops_per_launch": w.flops,
                "kernel_ms": kernel_ms,
                "note": ("step = the V transpose, the attention kernel and, for a K/V split, the combine kernel; "
                         "the step time is used for all"),
                "frac_of_bf16_peak": achieved / peak_bf16}
    if peak_bf16_sustained:
        roofline["frac_of_sustained"] = achieved / (2.0 * peak_bf16_sustained)
    line = {
        "metric": METRIC + " (FP8 E4M3 inputs)", "precision": "e4m3", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": slowest * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": workload_config(w, l2_note(args)),
        "roofline": roofline, "gpu_launches": fp8_launches * args.steps, "clocks": clocks.summary(),
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "e2e": None,
    }
    line["config"]["inputs"] = f"seeded synthetic ({w.qk_dist} Q,K; {w.v_dist} V), E4M3 per-tensor amax scaling"
    if not args.skip_cpu and world == 1:
        v_cpu, dt, rows, threads, desc = cpu_oracle_fp8_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def read_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def cpu_oracle_rows_sample(kind, N, target_seconds: float):
    """Time the fp64 oracle of a row operation on whole rows of length N; returns
    (GB/s of one bf16 read + write per element, seconds, rows, description)."""
    import oracle
    from exact_long_sequence_gb300 import workloads

    oracle.build()

    def timed(r):
        inp = workloads.row_inputs(kind, r, N, seed=1)
        t0 = time.perf_counter()
        if kind == "softmax":
            oracle.softmax_rows(inp)
        else:
            oracle.layernorm_rows(*inp, 1e-5)
        return time.perf_counter() - t0

    r = 1
    dt = timed(r)
    while dt * 2 < target_seconds and r < 4096:
        r *= 2
        dt = timed(r)
    desc = f"{r} rows of length {N}, fp64, 1 thread (plain loops)"
    return 4.0 * r * N / dt / 1e9, dt, r, desc


def run_gb300_rows(args, kind):
    import torch

    import exact_long_sequence_gb300 as ela
    from exact_long_sequence_gb300 import _build, workloads

    name = args.workload or ("softmax_r16384_n16384" if kind == "softmax" else "layernorm_r65536_n8192")
    if name not in workloads.ROW_WORKLOADS or workloads.ROW_WORKLOADS[name][0] != kind:
        raise SystemExit(f"unknown {kind} workload {name}; choose from "
                         f"{[k for k, v in workloads.ROW_WORKLOADS.items() if v[0] == kind]}")
    _, R, N = workloads.ROW_WORKLOADS[name]
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a); no CPU fallback exists")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(ela.LIB_PATH):
        _build.build()
    if world > 1:
        dist.barrier()
    ela.load_library()
    stream = torch.cuda.current_stream(dev)
    # seeded host draws (the recipe the parity test checks), copied to the device
    inp = workloads.row_inputs(kind, R, N, seed=1)
    inp = inp.to(dev) if kind == "softmax" else tuple(t.to(dev) for t in inp)
    out = torch.empty(R, N, dtype=torch.bfloat16, device=dev)
    ws_bytes = ela.load_library().attn_softmax_rows_workspace_bytes(R, N) if kind == "softmax" else 0
    ws = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=dev) if ws_bytes else None
    passes = 1 if kind == "layernorm" or ws_bytes == 0 else 2  # reads of x per step

    def step():
        if kind == "softmax":
            ela.softmax_rows(inp, out=out, workspace=ws, stream=stream)
        else:
            ela.layernorm_rows(*inp, eps=1e-5, out=out, stream=stream)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            if not args.keep_l2:
                flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    slowest = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    alg_bytes = 4.0 * R * N + (4.0 * N if kind == "layernorm" else 0.0)  # one bf16 read and write per element
    value = alg_bytes * args.steps * world / slowest / 1e9
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = read_hbm_peak()
    kernel_ms = statistics.mean(step_ms)
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    line = {
        "metric": f"standalone streaming {kind} GB/s (one bf16 read and write per element) on 1 GB300",
        "pass": kind, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slowest * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "R": R, "N": N, "inputs": "seeded synthetic normal rows, bf16",
                   "l2": l2_note(args),
                   "parallelism": "replicas", "reads_of_x_per_step": passes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json)",
                     "traffic": recorded_traffic(name, "rows"),
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": kernel_ms},
        "gpu_launches": args.steps * (1 if passes == 1 else 2), "clocks": clocks.summary(),
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "e2e": None,
    }
    if not args.skip_cpu and world == 1:
        v_cpu, dt, r, desc = cpu_oracle_rows_sample(kind, N, min(args.cpu_seconds, 5.0))
        line["cpu_baseline"] = {"value": v_cpu, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_gb300_bwd(args, w):
    import torch

    import exact_long_sequence_gb300 as ela
    from exact_long_sequence_gb300 import _build, workloads

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a); no CPU fallback exists")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(ela.LIB_PATH):
        _build.build()
    if world > 1:
        dist.barrier()
    ela.load_library()
    stream = torch.cuda.current_stream(dev)
    shape = (w.B, w.H, w.N, w.d)
    # seeded host draws of the workload's recipe (dO: the recipe's normal draw with seed + 1000)
    q, k, v = (t.to(dev) for t in workloads.workload_inputs(w))
    do = workloads.make_inputs(w.B, w.H, w.N, w.d, w.seed + 1000)[0].to(dev)
    o, lse = ela.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, stream=stream)
    ws = torch.empty(ela.load_library().attn_bwd_workspace_bytes(*shape), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(3, args.warmup)):
        ela.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, workspace=ws, stream=stream)
    torch.cuda.synchronize(dev)
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            if not args.keep_l2:
                flush.zero_()
            starts[i].record(stream)
            ela.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, workspace=ws, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    slowest = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    flops = BWD_FLOP_FACTOR * w.flops
    value = flops * args.steps * world / slowest / 1e12
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_sustained, peak_kind = read_peaks()
    kernel_ms = statistics.mean(step_ms)
    achieved = flops / (kernel_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "peak_kind": f"{peak_kind} dense bf16 burst (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback dense bf16 burst",
                "traffic": recorded_traffic("bwd:" + w.name, "bwd"), "algorithmic_flops_per_launch": flops,
                "kernel_ms": kernel_ms,
                "note": ("step = the three launches of attn_bwd (row statistics, gradients, dQ to bf16); "
                         "traffic is the gradient kernel's")}
    if peak_sustained:
        roofline["frac_of_sustained"] = achieved / peak_sustained
    line = {
        "metric": METRIC_BWD, "pass": "bwd", "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slowest * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, l2_note(args)),
        "roofline": roofline, "gpu_launches": 3 * args.steps, "clocks": clocks.summary(),
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "e2e": None,
    }
    if not args.skip_cpu and world == 1:
        v_cpu, dt, threads, desc = cpu_oracle_bwd_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_gb300(args, w):
    import torch

    import exact_long_sequence_gb300 as ela
    from exact_long_sequence_gb300 import _build, workloads

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a); no CPU fallback exists")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(ela.LIB_PATH):
        _build.build()
    if world > 1:
        dist.barrier()
    ela.load_library()

    stream = torch.cuda.current_stream(dev)
    shape = (w.B, w.H, w.N, w.d)
    # The workload's seeded inputs, drawn on the host by the same recipe the parity tests check
    # against the oracle, then made resident in device memory.
    q, k, v = (t.to(dev) for t in workloads.workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # Workloads with fewer work units than SMs, or a partial last wave, take the K/V split (the
    # attention kernel and the combine kernel); causal workloads take the dynamic schedule (a
    # counter zeroed by a one-thread kernel on the stream before each launch).  The workspace is
    # allocated once, outside the timed region.
    split_bytes = ela.split_workspace_bytes(w.B, w.H, w.N, w.d, w.causal)
    split_ws = torch.empty(split_bytes, dtype=torch.uint8, device=dev) if split_bytes else None
    choice = ela.split_choice(w.B, w.H, w.N, w.d, w.causal)
    split_step = choice["segs"] > 1
    # the attention kernel, plus the counter-zeroing kernel of the dynamic schedule and the
    # combine kernel of a K/V split
    launches_per_step = 1 + int(choice["dynamic"]) + int(split_step)

    for _ in range(max(3, args.warmup)):
        ela.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse, stream=stream, workspace=split_ws)
    torch.cuda.synchronize(dev)
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            if not args.keep_l2:
                flush.zero_()
            starts[i].record(stream)
            ela.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse, stream=stream, workspace=split_ws)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    if ela.last_device_error(stream) != ela.ATTN_OK:
        raise SystemExit("kernel reported a device error during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    my_seconds = sum(step_ms) / 1e3
    slowest = max_over_ranks(my_seconds, world, dev)
    value = w.flops * args.steps * world / slowest / 1e12
    ms_per_step = slowest * 1e3 / args.steps
    kernel_ms = statistics.mean(step_ms)

    # ------------------------------------------------------------- end to end through the host-buffer entry
    e2e = None
    if not args.skip_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty(shape[:3], dtype=torch.float32).pin_memory()
        ws = torch.empty(ela.host_workspace_bytes(*shape), dtype=torch.uint8, device=dev)
        for _ in range(2):
            ela.attn_fwd_host(qh, kh, vh, causal=w.causal, scale=w.scale, out_h=oh, lse_h=lh, workspace=ws,
                              stream=stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        e_ms = []
        for _ in range(max(3, args.steps // 2)):
            if not args.keep_l2:
                flush.zero_()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            ela.attn_fwd_host(qh, kh, vh, causal=w.causal, scale=w.scale, out_h=oh, lse_h=lh, workspace=ws,
                              stream=stream)
            stream.synchronize()
            e_ms.append((time.perf_counter() - t0) * 1e3)
        e_slow = max_over_ranks(sum(e_ms) / 1e3, world, dev)
        nbytes = q.numel() * 2
        e2e = {"value": w.flops * len(e_ms) * world / e_slow / 1e12, "unit": UNIT,
               "ms_per_step": e_slow * 1e3 / len(e_ms),
               "h2d_bytes_per_step": 3 * nbytes, "d2h_bytes_per_step": nbytes + lse.numel() * 4,
               "api": "attn_fwd_host (pinned host buffers; chunked copies overlapped with the kernels; wall clock until the caller's stream completes)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_sustained, peak_kind = read_peaks()
    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "peak_kind": f"{peak_kind} dense bf16 burst (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback dense bf16 burst",
                "traffic": recorded_traffic(w.name),
                "algorithmic_flops_per_launch": w.flops, "kernel_ms": kernel_ms,
                "io_bound_bytes": w.io_bytes}
    if split_step:
        roofline["note"] = ("K/V split: the step is the attention kernel plus the combine kernel (about 1 % of "
                            "it); the step time is used for both")
    if peak_sustained:
        roofline["frac_of_sustained"] = achieved / peak_sustained
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, l2_note(args)),
        "roofline": roofline,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.skip_cpu and world == 1:
        v_cpu, dt, rows, threads, desc = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
                                "seconds": dt}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    from exact_long_sequence_gb300 import workloads

    if args.which in ("softmax", "layernorm"):
        return run_gb300_rows(args, args.which)
    name = args.workload or workloads.HEADLINE
    if name not in workloads.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(workloads.WORKLOADS)}")
    w = workloads.WORKLOADS[name]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.which == "bwd":
        return run_gb300_bwd(args, w)
    if args.fp8:
        return run_gb300_fp8(args, w)
    return run_gb300(args, w)


if __name__ == "__main__":
    sys.exit(main())
