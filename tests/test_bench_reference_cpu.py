"""The bench's reference arm (the CPU oracle on the bench workload) keeps the
one-line JSON contract: run on the host cores, it prints the same metric,
unit and direction as the GPU arm, with impl = reference, a cpu_baseline that
describes this run and an e2e whose value is the line's own with no host to
device traffic.  CPU only; the arm never needs a GPU."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["ms_per_step"] > 0 and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"] == bench.bench_config()  # the GPU arm prints the same config
    assert d["config"]["calls_per_step"] == 37
    for name in ("o_proj", "o_proj_bf16", "q_b_proj", "kv_b_proj", "indexer_wq_b",
                 "indexer_wk_weights_proj", "lm_head"):
        assert name in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_cpu_baseline_rate_on_one_thread_and_all():
    for threads in (1, None):
        r = bench.cpu_oracle_rate(bench.STEP, budget_s=0.2, threads=threads, frac=0.0)
        assert r["value"] > 0 and r["unit"] == "GB/s" and r["kind"] == "oracle"
        assert r["cores"] == (threads or bench.host_cores())
        assert "112 rows in all" in r["sample"]  # 16 rows of each of the 7 planes


def test_step_is_the_layer_sweep_and_o_proj():
    calls = bench.step_calls()
    assert len(calls) == 37
    names = {p.name for p, _, _ in calls}
    assert names == {"o_proj", "o_proj_bf16", "q_b_proj", "kv_b_proj", "indexer_wq_b",
                     "indexer_wk_weights_proj", "lm_head"}
    ms = {(p.name, m) for p, _, m in calls}
    assert ("lm_head", 1) in ms and ("o_proj", 32) in ms and ("q_b_proj", 64) in ms
    # algorithmic bytes: W (+ fp32 row scales) + x + y with the logical K
    o = next(p for p, _, _ in calls if p.name == "o_proj")
    assert o.algorithmic_bytes(8) == 6144 * 16384 + 4 * 6144 + 2 * 8 * 16384 + 2 * 8 * 6144
    assert bench.step_bytes() == sum(p.algorithmic_bytes(m) for p, _, m in calls)


def test_oracle_sample_rows_are_the_planes_first_rows():
    import numpy as np
    from fp8_weight_only_w8a16_gb300 import synth

    p = bench.STEP[2]  # q_b_proj, FP8
    full = synth.plane_rows(p.n, 64, p.dtype, seed=2)  # a narrower plane: same row rule
    head = synth.plane_rows(p.n, 64, p.dtype, seed=2, rows=40)
    assert np.array_equal(full.w[:40], head.w) and np.array_equal(full.scale[:40], head.scale)


def test_source_hash_sees_code_not_comments():
    src = ('#define A 1\nint f(int x) { return x + A; } // add\n/* block\ncomment */\n'
           'const char *s = "// not a comment /* either */";\n')
    code = bench.strip_c_comments(src)
    assert "// add" not in code and "block" not in code
    assert '"// not a comment /* either */"' in code and "#define A 1\n" in code
    assert bench.strip_c_comments("char c = '/'; // x\n") == "char c = '/'; \n"
