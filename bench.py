#!/usr/bin/env python3
"""Benchmark of the w8a16 decode GEMV (one JSON line on rank 0).

Workload (default): one GLM-5.2 decode layer's weight-streaming projections
plus the output head, one GEMV call per (plane, token count):

  o_proj        E4M3 [6144, 16384] + fp32 row scales   M in {1, 2, 8, 32}
  o_proj        bf16 [6144, 16384] (the same shape)    M in {1, 2, 8, 32}
  q_b_proj      E4M3 [16384, 2048]                     M in {1, 2, 4, 8, 16, 32, 64}
  kv_b_proj     E4M3 [28672, 512]                      M in {1, 2, 4, 8, 16, 32, 64}
  indexer wq_b  E4M3 [4096, 2048]                      M in {1, 2, 4, 8, 16, 32, 64}
  indexer wk + weights_proj, bf16 [128 + 32, 6144], bound as one plane
                                                       M in {1, 2, 4, 8, 16, 32, 64}
  lm_head       bf16 [154880, 6144]                    M = 1

37 calls a step.  Every call reads a plane copy that no call has touched for
at least one whole step (~3.5 GB of weights, many times L2), so every call
streams its weights from HBM.

Timing: the step's calls are grouped by the kernel they launch (register ring
or tensor memory, FP8 or bf16); each group is one CUDA graph.  The timed
region replays the groups of exactly K steps after W warm-up steps, with a
barrier and a device synchronize on both sides, and records a CUDA event on
the launching stream after every group: the groups' times are measured live
inside the timed region and add up to it.  The max over ranks is taken.
value = algorithmic bytes (W + scales + x + y, logical K) of all steps of all
ranks / that time.

Also reported: microseconds per call for every (plane, M) (graphs of calls
rotating over >= 2 x L2 of plane copies), the roofline of the dominant kernel
(and of the FP8 register-ring kernel) against the measured HBM copy
bandwidth, the CPU oracle timed on the host cores (cpu_baseline), end-to-end
figures through the public API with host buffers (e2e: the calls issued every
step; e2e_graph: the step's copies and calls replayed as one CUDA graph), SM
clocks sampled during the timed region and the number of kernels launched.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep [--only NAMES] [--out FILE]   # every workload and M
  python bench.py --one NAME --m M                        # one workload (ncu)
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
STEP = workloads.BENCH_STEP
L2_FALLBACK = 126 << 20


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

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

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
# the step: what both arms compute, and the config line they share
# ---------------------------------------------------------------------------

def step_calls(step=STEP):
    """(projection, seed, m) of every call of one step, in plane order."""
    return [(p, seed, m) for seed, p in enumerate(step) for m in p.ms]


def step_bytes(step=STEP) -> int:
    return sum(p.algorithmic_bytes(m) for p, _, m in step_calls(step))


def plane_text(p) -> str:
    dt = {"e4m3fn": "E4M3 + fp32 row scales", "bf16": "bf16"}.get(p.dtype, p.dtype)
    return f"{p.name} {dt} [{p.n}, {p.k}] at M in {{{','.join(map(str, p.ms))}}}"


def bench_config(step=STEP) -> dict:
    """The config both arms print (identical by construction)."""
    return {
        "workload": "GLM-5.2 decode layer projections + lm_head, one GEMV call per (plane, M): "
                    + "; ".join(plane_text(p) for p in step)
                    + " (indexer wk [128, 6144] and weights_proj [32, 6144] bound as one plane)",
        "calls_per_step": len(step_calls(step)),
        "alg_bytes_per_step": step_bytes(step),
        "l2_policy": "inputs larger than L2: every call reads a plane copy no call has touched "
                     "for a whole step (~3.5 GB streamed); per-call timings rotate over >= 2 x L2 "
                     "of copies",
        "timing": "per kernel group a CUDA graph of its calls; CUDA events on the launching "
                  "stream after every group of every timed step; max over ranks",
    }


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


def l2_bytes(torch, device) -> int:
    props = torch.cuda.get_device_properties(device)
    return getattr(props, "L2_cache_size", 0) or getattr(props, "l2_cache_size", 0) or L2_FALLBACK


class PlaneSet:
    """Bound copies of one workload plane (enough that the copies span at
    least twice L2, and one per token count of the workload), its decode
    tokens and its outputs (one row block per token count)."""

    def __init__(self, proj, seed, w8, torch, device, l2, ms=None):
        self.proj, self.seed, self.w8, self.torch = proj, seed, w8, torch
        self.ms = tuple(proj.ms if ms is None else ms)
        plane = synth.plane_rows(proj.n, proj.k, proj.dtype, seed=seed, ldw=proj.ldw)
        self.plane = plane
        self.copies = max(len(self.ms), math.ceil(2 * l2 / proj.weight_bytes))
        w_d = torch.from_numpy(plane.w).to(device)
        s_d = torch.from_numpy(plane.scale).to(device) if plane.scale is not None else None
        src, self.fn = source_plane(w8, proj, w_d, s_d)
        self.build = w8.bind([src] * self.copies)
        torch.cuda.synchronize()
        del w_d, s_d, src
        self.x_host = synth.tokens(proj.k, max(self.ms), seed=seed)
        self.x = torch.from_numpy(self.x_host.view(np.int16)).to(device)
        self.y_all = torch.zeros((sum(self.ms), proj.out_n), dtype=torch.int16, device=device)
        self.y, row = {}, 0
        for m in self.ms:
            self.y[m] = self.y_all[row: row + m]
            row += m
        self.ws = self.build.new_workspace()

    def launch(self, copy, m, stream=None):
        self.fn(self.build, copy, self.x[:m], self.y[m], self.ws, stream=stream)

    def kernel(self, m) -> str:
        """The kernel a call with m tokens launches (as ncu names it, in short)."""
        p = self.build.plan(0, m)
        dt = {"e4m3fn": "fp8", "bf16": "bf16"}.get(self.proj.dtype, self.proj.dtype)
        return f"{'tc_gemv_kernel' if p.kernel == 1 else 'gemv_kernel'}<{dt}>"

    def per_call_us(self, m):
        """Median-of-5 microseconds per call with m tokens: a graph of one call
        per copy (>= 2 x L2 of weights), replayed, CUDA events on the
        launching stream."""
        torch = self.torch
        g = capture(torch, [(self, c, m) for c in range(self.copies)])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        reps = max(3, math.ceil(3.0 / max(e0.elapsed_time(e1), 1e-3)))
        samples = []
        for _ in range(5):
            torch.cuda.synchronize()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            samples.append(e0.elapsed_time(e1) * 1e3 / (reps * self.copies))
        return statistics.median(samples)


def capture(torch, calls):
    """A CUDA graph of the given (plane set, copy, m) launches, in order."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm the path outside capture
        for ps, c, m in calls:
            ps.launch(c, m)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for ps, c, m in calls:
            ps.launch(c, m)
    torch.cuda.synchronize()
    return g


class StepBench:
    """The bench step on one GPU: every plane bound, the calls grouped by the
    kernel they launch, one CUDA graph per group."""

    def __init__(self, step, w8, torch, device):
        self.torch = torch
        self.l2 = l2_bytes(torch, device)
        self.sets = [PlaneSet(p, seed, w8, torch, device, self.l2) for seed, p in enumerate(step)]
        calls = []  # (plane set, copy, m): copy i for the i-th token count
        for ps in self.sets:
            for i, m in enumerate(ps.ms):
                calls.append((ps, i, m))
        order = []
        for c in calls:
            k = c[0].kernel(c[2])
            if k not in order:
                order.append(k)
        self.groups = [(k, [c for c in calls if c[0].kernel(c[2]) == k]) for k in order]
        self.calls = calls
        self.graphs = [capture(torch, cs) for _, cs in self.groups]

    def group_bytes(self, gi) -> int:
        return sum(ps.proj.algorithmic_bytes(m) for ps, _, m in self.groups[gi][1])

    def step_bytes(self) -> int:
        return sum(self.group_bytes(gi) for gi in range(len(self.groups)))

    def run(self, steps):
        for _ in range(steps):
            for g in self.graphs:
                g.replay()

    def timed(self, steps, stream):
        """The timed region: (total ms, ms per group) from events recorded on
        the launching stream after every group of every step."""
        torch = self.torch
        ng = len(self.graphs)
        start = torch.cuda.Event(enable_timing=True)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ng)] for _ in range(steps)]
        start.record(stream)
        for s in range(steps):
            for gi, g in enumerate(self.graphs):
                g.replay()
                evs[s][gi].record(stream)
        torch.cuda.synchronize()
        group_ms = [0.0] * ng
        prev = start
        for s in range(steps):
            for gi in range(ng):
                group_ms[gi] += prev.elapsed_time(evs[s][gi])
                prev = evs[s][gi]
        total = start.elapsed_time(evs[-1][-1]) if steps else 0.0
        return total, group_ms


def roofline_of(sb: StepBench, gi, steps, group_ms, peak, peak_kind):
    name, calls = sb.groups[gi]
    launches = len(calls) * steps
    byts = sb.group_bytes(gi) * steps
    t_s = group_ms[gi] * 1e-3
    achieved = byts / t_s / 1e9 if t_s > 0 else 0.0
    traffic = [recorded_traffic(ps.proj.name, m) for ps, _, m in calls]
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": (round(sum(traffic) / len(traffic))
                        if traffic and all(t is not None for t in traffic) else None),
            "peak_source": f"hbm_gbs of {peak_kind}", "kernel": name,
            "launches": launches, "avg_launch_us": round(t_s / launches * 1e6, 3),
            "alg_bytes_per_launch": round(byts / launches),
            "time_share": round(group_ms[gi] / sum(group_ms), 4),
            "calls": [f"{ps.proj.name}@{m}" for ps, _, m in calls]}


# ---------------------------------------------------------------------------
# the oracle over the step (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleStep:
    """The oracle (as it stands) over one step of the bench workload on a
    sample of each plane's rows: the first `rows` rows of every plane (the
    same draws as the GPU arm's planes), all of its token counts.  Bytes are
    scaled to the sample."""

    def __init__(self, step, frac, threads):
        import oracle

        self.oracle, self.threads, self.frac = oracle, threads, frac
        self.items = []
        self.bytes = 0.0
        self.rows_total = 0
        for seed, p in enumerate(step):
            rows = max(16, min(p.n, int(round(p.n * frac))))
            plane = synth.plane_rows(p.n, p.k, p.dtype, seed=seed, rows=rows, ldw=p.ldw)
            x = synth.tokens(p.k, max(p.ms), seed=seed)
            dt = oracle.DT_E4M3FN if p.dtype == "e4m3fn" else oracle.DT_BF16
            xs = {m: np.ascontiguousarray(x[:m]) for m in p.ms}
            self.items.append((p, plane, dt, xs))
            self.bytes += sum(p.algorithmic_bytes(m) for m in p.ms) * rows / p.n
            self.rows_total += rows

    def run(self):
        """One sampled step; returns the seconds each plane took."""
        secs = []
        for p, plane, dt, xs in self.items:
            t0 = time.perf_counter()
            for m in p.ms:
                self.oracle.gemv(plane.w, dt, plane.scale, xs[m], k=p.k, threads=self.threads)
            secs.append(time.perf_counter() - t0)
        return secs

    def sample_text(self):
        return (f"the first {self.frac:.3%} of every plane's rows ({self.rows_total} rows in all, "
                f"at least 16 a plane) with all of its token counts, {self.threads} threads; "
                f"bytes scaled to the sample")


def oracle_frac(step, threads, seconds_per_step):
    """The row fraction that makes one sampled oracle step take about
    seconds_per_step (from a timed probe of 16 rows a plane)."""
    probe = OracleStep(step, 0.0, threads)
    secs = probe.run()
    # seconds of a whole-plane step: each plane's probe time per row x its rows
    full = sum(t / max(16, min(p.n, 16)) * p.n for t, p in zip(secs, step))
    return min(1.0, seconds_per_step / max(full, 1e-9))


def cpu_oracle_rate(step, budget_s=10.0, threads=None, frac=None):
    """The oracle on the host cores: algorithmic bytes per second over
    sampled steps of the workload, repeated for about budget_s."""
    threads = threads or host_cores()
    if frac is None:
        frac = oracle_frac(step, threads, budget_s / 3)
    o = OracleStep(step, frac, threads)
    reps, t0 = 0, time.perf_counter()
    while True:
        o.run()
        reps += 1
        elapsed = time.perf_counter() - t0
        if elapsed >= budget_s:
            break
    return {"value": o.bytes * reps / elapsed / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle", "sample": f"{reps} x one step on " + o.sample_text()
                                        + f", {elapsed:.1f} s"}


# ---------------------------------------------------------------------------
# end to end through the public API, host buffers
# ---------------------------------------------------------------------------

def e2e_rates(sb: StepBench, steps, torch):
    """Per step: copy every plane's tokens from pinned host memory, make the
    step's 37 library calls, read every output back into pinned host memory
    and wait for it on the host.  `direct`: the calls are made through the
    Python binding of the C ABI every step.  `graph`: each step's device work
    (copies and calls) captured once in a CUDA graph and replayed."""
    x_pin = [torch.from_numpy(ps.x_host.view(np.int16)).pin_memory() for ps in sb.sets]
    y_pin = [torch.empty(tuple(ps.y_all.shape), dtype=torch.int16).pin_memory()
             for ps in sb.sets]
    stream = torch.cuda.current_stream()

    def body():
        for ps, xp in zip(sb.sets, x_pin):
            ps.x.copy_(xp, non_blocking=True)
        for ps, c, m in sb.calls:
            ps.launch(c, m)
        for ps, yp in zip(sb.sets, y_pin):
            yp.copy_(ps.y_all, non_blocking=True)

    h2d = sum(ps.x_host.nbytes for ps in sb.sets)
    d2h = sum(ps.y_all.numel() * 2 for ps in sb.sets)
    out = {}
    for _ in range(3):
        body()
        stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        body()
        stream.synchronize()
    dt = time.perf_counter() - t0
    out["direct"] = {"value": sb.step_bytes() * steps / dt / 1e9, "unit": "GB/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "us_per_step": dt / steps * 1e6, "steps": steps}
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        body()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
        stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        g.replay()
        stream.synchronize()
    dt = time.perf_counter() - t0
    out["graph"] = {"value": sb.step_bytes() * steps / dt / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_step": dt / steps * 1e6, "steps": steps}
    return out


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


def _r(d):
    return {k: (round(v, 1) if isinstance(v, float) else v) for k, v in d.items()}


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

    sb = StepBench(STEP, w8, torch, device)
    stream = torch.cuda.current_stream()
    sb.run(max(args.warmup, 3))
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    t_ms, group_ms = sb.timed(args.steps, stream)
    barrier()
    time.sleep(0.25)
    clocks = sampler.stop()
    t_ms = slowest_time_ms(dist, t_ms, device)
    sbytes = sb.step_bytes()
    value = job_value(world, sbytes, args.steps, t_ms)

    peak, peak_kind = measured_peaks()
    dom = max(range(len(group_ms)), key=lambda i: group_ms[i])
    roofline = roofline_of(sb, dom, args.steps, group_ms, peak, peak_kind)
    by_kernel = [roofline_of(sb, gi, args.steps, group_ms, peak, peak_kind)
                 for gi in range(len(group_ms))]
    fp8_ring = [r for r in by_kernel if r["kernel"] == "gemv_kernel<fp8>"]

    # microseconds per call of every (plane, M), rotating over >= 2 x L2 of copies
    per_call = {}
    for ps in sb.sets:
        for m in ps.ms:
            us = ps.per_call_us(m)
            b = ps.proj.algorithmic_bytes(m)
            per_call[f"{ps.proj.name}@{m}"] = {
                "plane": ps.proj.name, "dtype": ps.proj.dtype, "n": ps.proj.n, "k": ps.proj.k,
                "m": m, "us_per_call": round(us, 3), "gbs": round(b / (us * 1e-6) / 1e9, 1),
                "pct_of_8tbs": round(100 * b / (us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 1),
                "frac_of_measured": round(b / (us * 1e-6) / 1e9 / peak, 4),
                "kernel": ps.kernel(m), "alg_bytes": b}
    fp8_le8 = [v for v in per_call.values() if v["dtype"] == "e4m3fn" and v["m"] <= 8]
    fp8_le8_gbs = (sum(v["alg_bytes"] for v in fp8_le8)
                   / sum(v["us_per_call"] * 1e-6 for v in fp8_le8) / 1e9)

    e2e = e2e_rates(sb, min(args.steps, args.e2e_steps), torch)
    for v in e2e.values():
        v["value"] = job_rate(dist, v["value"], device)

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu:
            cpu = cpu_oracle_rate(STEP, budget_s=args.cpu_seconds)
            one = cpu_oracle_rate(STEP, budget_s=min(3.0, args.cpu_seconds), threads=1)
            cpu["value_1_thread"] = one["value"]
            cpu["sample_1_thread"] = one["sample"]
        launches = len(sb.calls) * args.steps
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_ms / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3fn (and bf16) weights x bf16 -> f32",
            "data": "synthetic (seeded N(0,0.02) weights, FP8 quantized ptpc_fp8; N(0,1) bf16 "
                    "tokens)",
            "config": bench_config(STEP),
            "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 1),
            "fp8_m_le_8": {"gbs": round(fp8_le8_gbs, 1),
                           "pct_of_8tbs": round(100 * fp8_le8_gbs / NOMINAL_HBM_GBS, 1),
                           "frac_of_measured": round(fp8_le8_gbs / peak, 4),
                           "calls": len(fp8_le8),
                           "how": "sum of algorithmic bytes / sum of per-call times of the "
                                  "FP8 calls with M <= 8"},
            "roofline": roofline,
            "roofline_fp8_ring": fp8_ring[0] if fp8_ring else None,
            "roofline_by_kernel": [{k: r[k] for k in ("kernel", "achieved", "frac", "traffic",
                                                      "launches", "avg_launch_us", "time_share")}
                                   for r in by_kernel],
            "per_call": per_call,
            "cpu_baseline": cpu,
            "e2e": _r(e2e["direct"]), "e2e_graph": _r(e2e["graph"]),
            "clocks": clocks, "gpu_launches": launches,
            "timing_detail": {"plane_copies": {ps.proj.name: ps.copies for ps in sb.sets},
                              "l2_mib": round(sb.l2 / 2**20, 1),
                              "device_gib_bound": round(sum(ps.build.dst.numel()
                                                            for ps in sb.sets) / 2**30, 2)},
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
    threads = host_cores()
    total_steps = args.steps + args.warmup
    frac = oracle_frac(STEP, threads, args.ref_seconds / max(total_steps, 1))
    o = OracleStep(STEP, frac, threads)
    for _ in range(args.warmup):
        o.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.run()
    el = time.perf_counter() - t0
    value = o.bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3fn (and bf16) weights x bf16 -> f32",
        "data": "synthetic (seeded N(0,0.02) weights, FP8 quantized ptpc_fp8; N(0,1) bf16 "
                "tokens)",
        "config": bench_config(STEP),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": "each step: " + o.sample_text()},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------------------------
# sweep: every workload and token count; one workload for ncu
# ---------------------------------------------------------------------------

def run_sweep(args):
    import torch
    from fp8_weight_only_w8a16_gb300 import w8

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    peak, peak_kind = measured_peaks()
    l2 = l2_bytes(torch, device)
    out = open(args.out, "w") if args.out else None
    names = args.only.split(",") if args.only else [p.name for p in workloads.ALL]
    for name in names:
        proj = workloads.BY_NAME[name]
        ps = PlaneSet(proj, 0, w8, torch, device, l2)
        for m in proj.ms:
            us = ps.per_call_us(m)
            plan = ps.build.plan(0, m)
            gbs = proj.algorithmic_bytes(m) / (us * 1e-6) / 1e9
            rec = {"workload": name, "dtype": proj.dtype, "n": proj.n, "k": proj.k, "m": m,
                   "us_per_call": round(us, 3), "gbs": round(gbs, 1),
                   "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 1),
                   "frac_of_peak": round(gbs / peak, 4), "peak": f"{peak} ({peak_kind})",
                   "tflops": round(proj.flops(m) / (us * 1e-6) / 1e12, 1),
                   "alg_bytes": proj.algorithmic_bytes(m), "grid": plan.grid,
                   "splits": plan.splits, "kernel": ps.kernel(m), "copies": ps.copies}
            line = json.dumps(rec)
            print(line, flush=True)
            if out:
                out.write(line + "\n")
        del ps
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
    plane = synth.plane_rows(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
    x_all = synth.tokens(proj.k, m, seed=0)
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=500)
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
