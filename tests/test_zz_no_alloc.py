"""w8_gemv_noalloc: the FP8 GEMV for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc where they run the GEMV (a host callback,
an allocator hook, a framework that forbids device allocations while it
records or replays a step), so they cannot hand w8_gemv the workspace it asks
for when a plan splits K across CTAs.  w8_gemv_noalloc takes that scratch from
a fixed array inside the library instead.  These tests call it through the C
ABI and check, on two calls in a row, that it gives exactly what w8_gemv gives
with a caller workspace, and that both are within the parity tolerance of the
oracle's fp64 recompute, also when calls follow each other on one stream with
no synchronisation; and that calls needing more than the fixed array, or made
on a bf16 or block-scaled FP8 build, are refused before any launch.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process (the
first call on the device sets the array up).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_weight_only_w8a16_gb300 import synth

from .gpu_util import bind_plane, dev, from_dev, to_dev

pytestmark = pytest.mark.gpu

LIMIT = 64 << 10  # W8_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def w8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_weight_only_w8a16_gb300 import w8 as lib

    return lib


# (n, k, m): register-ring plans that split K across CTAs (and so use the
# scratch), a tensor-memory plan (its split partials meet on chip: no scratch)
# and a large plane whose plan does not split
CASES = [(128, 2048, 16), (32, 6144, 12), (40, 6144, 5), (6144, 1024, 32), (2624, 6144, 4),
         (256, 512, 100)]


@pytest.mark.parametrize("n,k,m", CASES)
def test_noalloc_equals_gemv_with_workspace(w8, n, k, m):
    rng = np.random.default_rng(n + k + m)
    plane = synth.weight_plane(rng, n, k)
    x = synth.activations(rng, k, m)
    b, _src = bind_plane(w8, plane)
    needs_scratch = b.plan(0, m).splits > 1
    if (n, k) in ((128, 2048), (32, 6144), (40, 6144)):
        assert needs_scratch and b.workspace_bytes(0, m) > 0
    assert b.workspace_bytes(0, m) <= LIMIT

    xd = to_dev(x)
    y_ref = torch.zeros((m, n), dtype=torch.int16, device=dev())
    w8.w8_gemv(b, 0, xd, y_ref, b.new_workspace(0, m))
    torch.cuda.synchronize()
    ref = from_dev(y_ref)
    y64, mag = oracle.gemv_f64(plane.w, oracle.DT_E4M3FN, plane.scale, x, k=k)

    for _ in range(2):  # two calls in a row share the library's scratch
        y = torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev())
        w8.w8_gemv_noalloc(b, 0, xd, y)
        torch.cuda.synchronize()
        got = from_dev(y)
        assert np.array_equal(got, ref)
        ok, worst = oracle.within_tolerance(got, y64, mag)
        assert ok, worst


def test_noalloc_back_to_back_calls_on_one_stream(w8):
    # split-K calls queued on one stream with no synchronisation between them,
    # each with its own tokens and output: programmatic dependent launch lets
    # a call's weight stream begin while the previous call drains, but its
    # scratch use waits for that call, so each result equals w8_gemv's
    n, k, m = 128, 2048, 16
    rng = np.random.default_rng(23)
    plane = synth.weight_plane(rng, n, k)
    b, _src = bind_plane(w8, plane)
    assert b.plan(0, m).splits > 1
    ws = b.new_workspace(0, m)
    xs = [synth.activations(rng, k, m) for _ in range(3)]
    refs = []
    for x in xs:
        y_ref = torch.zeros((m, n), dtype=torch.int16, device=dev())
        w8.w8_gemv(b, 0, to_dev(x), y_ref, ws)
        torch.cuda.synchronize()
        refs.append(from_dev(y_ref))
    xds = [to_dev(x) for x in xs]
    ys = [torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev()) for _ in xs]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for xd, y in zip(xds, ys):
        w8.w8_gemv_noalloc(b, 0, xd, y, stream=s)
    s.synchronize()
    for x, y, ref in zip(xs, ys, refs):
        got = from_dev(y)
        assert np.array_equal(got, ref)
        y64, mag = oracle.gemv_f64(plane.w, oracle.DT_E4M3FN, plane.scale, x, k=k)
        ok, worst = oracle.within_tolerance(got, y64, mag)
        assert ok, worst


def test_noalloc_on_a_gate_up_plane_keeps_source_order(w8):
    # a merged gate_up plane (gate rows first) whose plan splits K: the
    # packed rows are interleaved, the output is in source row order
    n, k, m = 32, 6144, 5
    rng = np.random.default_rng(11)
    plane = synth.weight_plane(rng, n, k)
    x = synth.activations(rng, k, m)
    w_d, s_d = to_dev(plane.w), to_dev(plane.scale)
    b = w8.bind([w8.Plane.from_tensor(w_d, s_d, k=k, layout=w8.SRC_GATE_UP)])
    assert b.plan(0, m).splits > 1
    xd = to_dev(x)
    y_ref = torch.zeros((m, n), dtype=torch.int16, device=dev())
    w8.w8_gemv(b, 0, xd, y_ref, b.new_workspace(0, m))
    y = torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev())
    w8.w8_gemv_noalloc(b, 0, xd, y)
    torch.cuda.synchronize()
    got = from_dev(y)
    assert np.array_equal(got, from_dev(y_ref))
    y64, mag = oracle.gemv_f64(plane.w, oracle.DT_E4M3FN, plane.scale, x, k=k)
    ok, worst = oracle.within_tolerance(got, y64, mag)
    assert ok, worst


def test_noalloc_refuses_what_it_cannot_serve(w8):
    # a plan whose split partials exceed the fixed scratch (the first such
    # shape for this GPU's SM count)
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    cands = [(n, k, 8) for n in (16, 32, 64, 128, 256, 512, 1024) for k in (6144, 16384)]
    over = [c for c in cands if w8.plan_shape(*c, sms).workspace_bytes > LIMIT]
    assert over, "no candidate shape needs more than the fixed scratch"
    n, k, m = over[0]
    rng = np.random.default_rng(7)
    plane = synth.weight_plane(rng, n, k)
    b, _src = bind_plane(w8, plane)
    assert b.plan(0, m).workspace_bytes > LIMIT
    x = to_dev(synth.activations(rng, k, m))
    y = torch.zeros((m, n), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_noalloc(b, 0, x, y)
    assert e.value.name == "W8_ERR_SCRATCH"
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    # a bf16 build is refused
    bp = synth.weight_plane(rng, 64, 256, "bf16")
    b16, _src16 = bind_plane(w8, bp)
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_noalloc(b16, 0, to_dev(synth.activations(rng, 256, 2)),
                           torch.zeros((2, 64), dtype=torch.int16, device=dev()))
    assert e.value.name == "W8_ERR_DTYPE"
    # so is a block-scaled FP8 build (one factor per 128 x 128 block), which
    # w8_gemv serves
    bplane, _x = synth.workload(256, 512, "e4m3fn_b128", seed=4)
    bb = w8.bind([w8.Plane.e4m3_b128(to_dev(bplane.w), to_dev(bplane.scale), k=512)])
    y8 = torch.zeros((2, 256), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_noalloc(bb, 0, to_dev(synth.activations(rng, 512, 2)), y8)
    assert e.value.name == "W8_ERR_DTYPE"
    torch.cuda.synchronize()
    assert torch.all(y8 == 0)
