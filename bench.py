#!/usr/bin/env python3
"""Benchmark of the w8a16 decode GEMV (one JSON line on rank 0).

Workload (default): the GLM-5.2 fused_qkv_a_proj plane, E4M3 W [2624, 6144]
with fp32 row scales, and its three decode batches M = 1, 4, 16 (bf16
activations).  One step = one w8_gemv call per batch, i.e. three kernel
launches, each on its own copy of the plane.

Timing: the plane is bound into C copies with C * 16 MB > 2 x L2, calls cycle
through the copies, so every call streams its weights from HBM; the steps are
captured in CUDA graphs and replayed; CUDA events on the launching stream
bracket exactly K steps after W warm-up steps, with a barrier and a device
synchronize on both sides; the max over ranks is taken.  value = algorithmic
bytes (W + scales + x + y, logical K) of all steps of all ranks / that time.

Also reported: per-batch microseconds per call, the roofline of the GEMV
kernel against the measured HBM copy bandwidth, the CPU oracle timed on the
host cores (cpu_baseline), an end-to-end figure through the C ABI with host
buffers (e2e), SM clocks sampled during the timed region and the number of
kernels launched.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep [--out FILE]   # every workload and M, one line each
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_weight_only_w8a16_gb300 import synth, workloads  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of ~8 TB/s) for FP8 GEMV, M=1–64"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = workloads.FUSED_QKV_A


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def strip_c_comments(src: str) -> str:
    """C/C++/CUDA source without its // and /* */ comments (string and
    character literals kept as they are): what the compiler sees."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "".join(out)


def gemv_source_sha() -> str:
    """A hash of the GEMV kernels' source code, comments excluded: a recorded
    DRAM traffic figure stays valid while the compiled kernels cannot have
    changed."""
    h = hashlib.sha256()
    for f in ("w8_gemv.cu", "w8_tc.cu", "w8_device.cuh", "w8_layout.h", "w8_internal.h"):
        with open(os.path.join(ROOT, "fp8_weight_only_w8a16_gb300", "csrc", f)) as fh:
            code = strip_c_comments(fh.read())
        # code lines only: trailing blanks and lines left empty do not count
        lines = [ln.rstrip() for ln in code.splitlines()]
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, m: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemv_dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = gemv_source_sha()
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if (kv.get("kernel_sha") == sha and kv.get("workload") == workload
                    and kv.get("m") == str(m)):
                return int(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags)
                          if fl.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def source_plane(w8, proj, w_d, s_d):
    """The w8.Plane of a workload's source tensors and the gemv call it takes."""
    if proj.dtype == "mxfp4":
        return w8.Plane.mxfp4(w_d, s_d, k=proj.k), w8.mxfp4_gemv
    if proj.dtype == "e4m3fn_b128":
        return w8.Plane.e4m3_b128(w_d, s_d, k=proj.k), w8.w8_gemv
    silu = proj.act == "silu_mul"
    fp8 = proj.dtype == "e4m3fn"
    src = w8.Plane.from_tensor(w_d, s_d, k=proj.k, dtype=w8.DT_E4M3FN if fp8 else w8.DT_BF16,
                               layout=w8.SRC_GATE_UP if silu else w8.SRC_ROW_MAJOR)
    return src, (w8.w8_gemv_silu_mul if silu else w8.w8_gemv if fp8 else w8.bf16_gemv)


class GemvBench:
    """Bound copies of one workload plane, activations, outputs, workspace."""

    def __init__(self, proj, ms, w8, torch, device, min_bytes=None):
        self.proj, self.ms, self.w8, self.torch, self.device = proj, tuple(ms), w8, torch, device
        plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
        self.plane = plane
        props = torch.cuda.get_device_properties(device)
        l2 = getattr(props, "L2_cache_size", 0) or getattr(props, "l2_cache_size", 0) or (128 << 20)
        self.l2 = l2
        wbytes = plane.w.nbytes
        need = min_bytes if min_bytes is not None else 2 * l2
        copies = max(1, math.ceil(need / wbytes) + 1)
        # a whole number of steps per cycle through the copies
        per_step = len(self.ms)
        copies = per_step * math.ceil(copies / per_step)
        self.copies = copies
        w_d = torch.from_numpy(plane.w).to(device)
        s_d = torch.from_numpy(plane.scale).to(device) if plane.scale is not None else None
        src, self.fn = source_plane(w8, proj, w_d, s_d)
        self.build = w8.bind([src] * copies)
        torch.cuda.synchronize()
        del w_d, s_d, src
        mmax = max(self.ms)
        assert x_all.shape[0] >= mmax, "the workload draws fewer token rows than the largest M"
        self.x_host = np.ascontiguousarray(x_all[:mmax])
        self.x = torch.from_numpy(self.x_host.view(np.int16)).to(device)
        # every call's output rows in one buffer (row blocks of m rows, in the
        # order of ms), so that a step's results leave the device in one copy
        self.y_all = torch.zeros((sum(self.ms), proj.out_n), dtype=torch.int16, device=device)
        self.y, row = {}, 0
        for m in self.ms:
            self.y[m] = self.y_all[row: row + m]
            row += m
        self.ws = self.build.new_workspace()

    def step_bytes(self):
        return sum(self.proj.algorithmic_bytes(m) for m in self.ms)

    def launch(self, copy, m, stream=None):
        self.fn(self.build, copy, self.x[:m], self.y[m], self.ws, stream=stream)

    def capture(self, calls):
        """A CUDA graph of the given (copy, m) launches, in order."""
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm the path outside capture
            for c, m in calls:
                self.launch(c, m)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for c, m in calls:
                self.launch(c, m)
        torch.cuda.synchronize()
        return g

    def step_calls(self, j):
        base = (j * len(self.ms)) % self.copies
        return [((base + i) % self.copies, m) for i, m in enumerate(self.ms)]

    def step_graphs(self):
        cyc = self.copies // len(self.ms)
        full = self.capture([c for j in range(cyc) for c in self.step_calls(j)])
        partial = {r: self.capture([c for j in range(r) for c in self.step_calls(j)])
                   for r in range(1, cyc)}
        return cyc, full, partial

    def run_steps(self, k, graphs):
        cyc, full, partial = graphs
        for _ in range(k // cyc):
            full.replay()
        if k % cyc:
            partial[k % cyc].replay()

    def per_call_us(self, m, reps=200):
        """Median-of-5 microseconds per call for one batch size (graph of one
        launch per copy, replayed), timed with events on the launching stream."""
        torch = self.torch
        g = self.capture([(c, m) for c in range(self.copies)])
        for _ in range(3):
            g.replay()
        samples = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            samples.append(e0.elapsed_time(e1) * 1e3 / (reps * self.copies))
        return statistics.median(samples)


def cpu_oracle_rate(proj, ms, budget_s=10.0, rows=None, threads=None):
    """The oracle (as it stands) on the host cores: algorithmic bytes per
    second over full steps of the workload, repeated for about budget_s."""
    import oracle

    plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
    threads = threads or host_cores()
    dt = oracle.DT_E4M3FN if proj.dtype == "e4m3fn" else oracle.DT_BF16
    n_rows = proj.n if rows is None else rows
    w = np.ascontiguousarray(plane.w[:n_rows])
    sc = None if plane.scale is None else np.ascontiguousarray(plane.scale[:n_rows])
    frac = n_rows / proj.n
    xs = {m: np.ascontiguousarray(x_all[:m]) for m in ms}
    reps, elapsed = 0, 0.0
    t0 = time.perf_counter()
    while True:
        for m in ms:
            oracle.gemv(w, dt, sc, xs[m], k=proj.k, threads=threads)
        reps += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s:
            break
    step_bytes = sum(proj.algorithmic_bytes(m) for m in ms) * frac
    return {"value": step_bytes * reps / elapsed / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} x {proj.name} step (M={','.join(map(str, ms))}) on {n_rows} of "
                      f"{proj.n} rows, {threads} threads, {elapsed:.1f} s",
            "seconds_per_step": elapsed / reps / frac}


def e2e_rate(b: GemvBench, steps, torch):
    """Through the public API with host buffers: per step, copy the step's
    tokens from pinned host memory, run the three calls, read every output
    back into pinned host memory (the calls write row blocks of one buffer,
    read back in one copy) and wait for it on the host.  As a serving
    loop would, each step's device work (the copies and the three library
    calls, made through the Python binding of the C ABI) is captured once in
    a CUDA graph and replayed; the host waits for every step."""
    mmax = max(b.ms)
    x_pin = torch.from_numpy(b.x_host.view(np.int16)).pin_memory()
    y_pin = torch.empty(tuple(b.y_all.shape), dtype=torch.int16).pin_memory()

    def body(j):
        b.x.copy_(x_pin, non_blocking=True)
        for c, m in b.step_calls(j):
            b.launch(c, m)
        y_pin.copy_(b.y_all, non_blocking=True)  # every call's output, one copy

    cyc = b.copies // len(b.ms)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        body(0)  # warm the path outside capture
    torch.cuda.synchronize()
    graphs = []
    for j in range(cyc):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body(j)
        graphs.append(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def one(j):
        graphs[j % cyc].replay()
        stream.synchronize()

    for j in range(5):
        one(j)
    t0 = time.perf_counter()
    for j in range(steps):
        one(j)
    dt = time.perf_counter() - t0
    h2d = mmax * b.proj.k * 2
    d2h = sum(m * b.proj.out_n * 2 for m in b.ms)
    return {"value": b.step_bytes() * steps / dt / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "us_per_step": dt / steps * 1e6, "steps": steps}


def slowest_time_ms(dist, t_ms: float, device="cpu") -> float:
    """The whole job's timed region: the slowest rank's (max over ranks; with
    dist None, one GPU, it passes through)."""
    if dist is None:
        return t_ms
    import torch

    t = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(dist, rate: float, device="cpu") -> float:
    """Whole-job rate of N independent replicas: the slowest rank's rate times
    the number of ranks (with dist None it passes through)."""
    if dist is None:
        return rate
    import torch

    t = torch.tensor([rate], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return float(t.item()) * dist.get_world_size()


def job_value(world: int, step_bytes: int, steps: int, t_ms: float) -> float:
    """GB/s of the whole job: every rank's algorithmic bytes over the slowest
    rank's time (weak scaling: each replica streams the same workload)."""
    return world * step_bytes * steps / (t_ms * 1e-3) / 1e9


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def barrier():
        if dist is not None:
            dist.barrier()

    from fp8_weight_only_w8a16_gb300 import w8

    proj, ms = DEFAULT_WORKLOAD, DEFAULT_WORKLOAD.ms
    b = GemvBench(proj, ms, w8, torch, device)
    graphs = b.step_graphs()

    # warm-up
    b.run_steps(max(args.warmup, 3), graphs)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    b.run_steps(args.steps, graphs)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    time.sleep(0.25)
    clocks = sampler.stop()
    t_ms = slowest_time_ms(dist, e0.elapsed_time(e1), device)
    step_bytes = b.step_bytes()
    value = job_value(world, step_bytes, args.steps, t_ms)

    # per-batch microseconds and the kernel roofline
    per_m = {}
    reps = max(5, min(200, args.steps // 50))
    for m in ms:
        us = b.per_call_us(m, reps=reps)
        per_m[m] = {"us_per_call": round(us, 3),
                    "gbs": round(proj.algorithmic_bytes(m) / (us * 1e-6) / 1e9, 1),
                    "pct_of_8tbs": round(100 * proj.algorithmic_bytes(m) / (us * 1e-6) / 1e9
                                         / NOMINAL_HBM_GBS, 1)}
    peak, peak_kind = measured_peaks()
    launches = len(ms) * args.steps
    achieved = step_bytes * args.steps / (t_ms * 1e-3) / 1e9  # per GPU, kernel-time average
    # DRAM bytes per launch, averaged over the step's launches like `achieved`
    # (None unless the committed ncu summary was taken on this kernel source)
    per_m_traffic = [recorded_traffic(proj.name, m) for m in ms]
    traffic = (round(sum(per_m_traffic) / len(ms))
               if all(t is not None for t in per_m_traffic) else None)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"hbm_gbs of {peak_kind}",
                "kernel": f"gemv_kernel<fp8> (M={','.join(map(str, ms))})",
                "alg_bytes_per_launch": {str(m): proj.algorithmic_bytes(m) for m in ms}}

    e2e = e2e_rate(b, min(args.steps, args.e2e_steps), torch)
    e2e["value"] = job_rate(dist, e2e["value"], device)

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu:
            cpu = cpu_oracle_rate(proj, ms, budget_s=args.cpu_seconds)
            one = cpu_oracle_rate(proj, ms, budget_s=min(3.0, args.cpu_seconds), rows=256,
                                  threads=1)
            cpu["value_1_thread"] = one["value"]
            cpu["sample_1_thread"] = one["sample"]
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_ms / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3fn weights x bf16 -> f32",
            "data": "synthetic (seeded N(0,0.02) weights quantized ptpc_fp8, N(0,1) bf16 tokens)",
            "config": {"workload": f"{proj.name} E4M3 [{proj.n}, {proj.k}] + fp32 row scales, "
                                   f"M in {{{','.join(map(str, ms))}}} (one call each per step)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2_policy": f"inputs larger than L2: {b.copies} plane copies "
                                    f"({b.copies * b.plane.w.nbytes / 2**20:.0f} MiB) rotated, "
                                    f"L2 {b.l2 / 2**20:.0f} MiB",
                       "timing": "CUDA graphs of rotated calls, CUDA events on the launching "
                                 "stream, max over ranks",
                       "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 1),
                       "per_m": {str(m): v for m, v in per_m.items()}},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": {
                k: (round(v, 1) if isinstance(v, float) else v) for k, v in e2e.items()},
            "clocks": clocks, "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle on the same workload and metric
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    proj, ms = DEFAULT_WORKLOAD, DEFAULT_WORKLOAD.ms
    import oracle

    plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
    threads = host_cores()
    dt = oracle.DT_E4M3FN if proj.dtype == "e4m3fn" else oracle.DT_BF16
    xs = {m: np.ascontiguousarray(x_all[:m]) for m in ms}
    # size each step's row sample so that warm-up + steps take ~args.ref_seconds
    probe_rows = min(proj.n, 128)
    t0 = time.perf_counter()
    for m in ms:
        oracle.gemv(np.ascontiguousarray(plane.w[:probe_rows]), dt,
                    None if plane.scale is None else plane.scale[:probe_rows], xs[m], k=proj.k,
                    threads=threads)
    per_row = (time.perf_counter() - t0) / probe_rows
    total_steps = args.steps + args.warmup
    rows = int(max(1, min(proj.n, args.ref_seconds / max(total_steps, 1) / per_row)))
    w = np.ascontiguousarray(plane.w[:rows])
    sc = None if plane.scale is None else np.ascontiguousarray(plane.scale[:rows])

    def step():
        for m in ms:
            oracle.gemv(w, dt, sc, xs[m], k=proj.k, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    frac = rows / proj.n
    step_bytes = sum(proj.algorithmic_bytes(m) for m in ms) * frac
    value = step_bytes * args.steps / el / 1e9
    sample = (f"{rows} of {proj.n} rows per step (bytes scaled to the sample), M="
              f"{','.join(map(str, ms))}, {threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3fn weights x bf16 -> f32",
        "data": "synthetic (seeded N(0,0.02) weights quantized ptpc_fp8, N(0,1) bf16 tokens)",
        "config": {"workload": f"{proj.name} E4M3 [{proj.n}, {proj.k}] + fp32 row scales, "
                               f"M in {{{','.join(map(str, ms))}}} (one call each per step)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------------------------
# sweep: every workload and token count
# ---------------------------------------------------------------------------

def run_sweep(args):
    import torch
    from fp8_weight_only_w8a16_gb300 import w8

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    out = open(args.out, "w") if args.out else None
    names = args.only.split(",") if args.only else [p.name for p in workloads.ALL]
    for name in names:
        proj = workloads.BY_NAME[name]
        b = GemvBench(proj, proj.ms, w8, torch, device)
        for m in proj.ms:
            us = b.per_call_us(m, reps=max(20, int(2e5 / max(1, b.copies * 5))))
            plan = b.build.plan(0, m)
            gbs = proj.algorithmic_bytes(m) / (us * 1e-6) / 1e9
            rec = {"workload": name, "dtype": proj.dtype, "n": proj.n, "k": proj.k, "m": m,
                   "us_per_call": round(us, 3), "gbs": round(gbs, 1),
                   "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 1),
                   "frac_of_peak": round(gbs / peak, 4), "peak": f"{peak} ({peak_kind})",
                   "tflops": round(proj.flops(m) / (us * 1e-6) / 1e12, 1),
                   "alg_bytes": proj.algorithmic_bytes(m), "grid": plan.grid,
                   "splits": plan.splits, "copies": b.copies}
            line = json.dumps(rec)
            print(line, flush=True)
            if out:
                out.write(line + "\n")
        del b
        torch.cuda.empty_cache()
    if out:
        out.close()


def run_one(args):
    """Bind one workload and run its GEMV a few times, flushing L2 between
    calls (the small case the ncu captures profile)."""
    import torch
    from fp8_weight_only_w8a16_gb300 import w8

    proj = workloads.BY_NAME[args.one]
    m = args.m
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
    w_d = torch.from_numpy(plane.w).to(device)
    s_d = torch.from_numpy(plane.scale).to(device) if plane.scale is not None else None
    src, fn = source_plane(w8, proj, w_d, s_d)
    b = w8.bind([src])
    ws = b.new_workspace()
    x = torch.from_numpy(np.ascontiguousarray(x_all[:m]).view(np.int16)).to(device)
    y = torch.zeros((m, proj.out_n), dtype=torch.int16, device=device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # 2 x L2
    for _ in range(args.calls):
        flush.zero_()
        fn(b, 0, x, y, ws)
    torch.cuda.synchronize()
    p = b.plan(0, m)
    print(json.dumps({"workload": proj.name, "m": m, "calls": args.calls, "grid": p.grid,
                      "warps_k": p.warps_k, "row_tiles_per_warp": p.row_tiles_per_warp,
                      "splits": p.splits, "alg_bytes": proj.algorithmic_bytes(m)}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--only", default="")
    ap.add_argument("--out", default="")
    ap.add_argument("--one", default="", help="run one workload's GEMV --calls times")
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--calls", type=int, default=6)
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.one:
        run_one(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
