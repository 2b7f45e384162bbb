"""The GEMV tolerance is not vacuous (CPU only).

Parity tests accept a kernel result when |y - y64| <= 2^-7 |y64| +
2^-12 sum_k |scale W x| on every output.  These tests show that bound rejects
the plausible mistakes of a kernel -- a K block dropped, repeated or taken
from the wrong place, a block's sign flipped, the wrong row's scale or none,
tokens mixed up -- on the bench's plane shapes, while it accepts the exact
definition: each mistake is made on the inputs, run through the oracle, and
held against the correct fp64 recompute."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from fp8_weight_only_w8a16_gb300 import synth

DT8 = oracle.DT_E4M3FN


def _case(n, k, m, seed):
    plane, x_all = synth.workload(n, k, "e4m3fn", seed=seed)
    return plane.w, plane.scale, np.ascontiguousarray(x_all[:m])


def _mistakes(w, scale, x):
    k = x.shape[1]
    out = {}
    xd = x.copy()
    xd[:, 32:64] = 0
    out["K block dropped"] = (w, scale, xd)
    xr = x.copy()
    xr[:, 64:96] = x[:, 32:64]
    out["K block repeated"] = (w, scale, xr)
    xs = x.copy()
    xs[:, 32:64], xs[:, 64:96] = x[:, 64:96], x[:, 32:64]
    out["two K blocks swapped"] = (w, scale, xs)
    wf = w.copy()
    wf[:, k - 32:] ^= 0x80
    out["last K block's sign flipped"] = (wf, scale, x)
    out["scale of the next row"] = (w, np.roll(scale, -1), x)
    out["scale dropped"] = (w, np.ones_like(scale), x)
    if x.shape[0] > 1:
        out["tokens mixed up"] = (w, scale, np.roll(x, 1, axis=0))
    return out


@pytest.mark.parametrize("n,k,m", [(256, 6144, 4), (256, 16384, 1), (256, 512, 8),
                                   (128, 2048, 16)])
def test_tolerance_accepts_the_definition_and_rejects_mistakes(n, k, m):
    w, scale, x = _case(n, k, m, seed=n + k + m)
    y64, mag = oracle.gemv_f64(w, DT8, scale, x, threads=8)
    ok, worst = oracle.within_tolerance(oracle.gemv(w, DT8, scale, x, threads=8), y64, mag)
    assert ok, worst
    for name, (wm, sm, xm) in _mistakes(w, scale, x).items():
        ym = oracle.gemv(wm, DT8, sm, xm, threads=8)
        ok, worst = oracle.within_tolerance(ym, y64, mag)
        assert not ok, f"{name} passes the tolerance (worst {worst:.3g})"


def test_silu_mul_tolerance_rejects_mistakes():
    """The propagated SiLU-and-multiply bound accepts the two-step result and
    rejects gate and up swapped, the SiLU left out, the multiply left out, a
    gate row paired with the next up row, and the sign of the SiLU's
    exponent flipped."""
    half, k, m = 128, 6144, 8
    w, scale, x = _case(2 * half, k, m, seed=3)
    y = oracle.gemv(w, DT8, scale, x, threads=8)
    y64, mag = oracle.gemv_f64(w, DT8, scale, x, threads=8)
    g, u = y[:, :half], y[:, half:]
    args = (y64[:, :half], mag[:, :half], y64[:, half:], mag[:, half:])
    ok, worst = oracle.silu_mul_within_tolerance(oracle.silu_mul(g, u), *args)
    assert ok, worst
    gf, uf = oracle.bf16_bits_to_f64(g), oracle.bf16_bits_to_f64(u)
    wrong = {
        "gate and up swapped": oracle.silu_mul(u, g),
        "SiLU left out": oracle.f64_to_bf16_rne(gf * uf),
        "multiply left out": oracle.f64_to_bf16_rne(oracle.silu_mul_f64(gf, 1.0)),
        "up row of the next gate row": oracle.silu_mul(g, np.roll(u, -1, axis=1)),
        "exponent sign flipped": oracle.f64_to_bf16_rne(gf / (1.0 + np.exp(gf)) * uf),
    }
    for name, h in wrong.items():
        ok, worst = oracle.silu_mul_within_tolerance(h, *args)
        assert not ok, f"{name} passes the tolerance (worst {worst:.3g})"


def test_block_scaled_tolerance_rejects_wrong_factors():
    """On a block-scaled plane the bound rejects the factor of the next column
    block, of the next row block, and factors applied to each 32-column K
    block's neighbour."""
    n, k, m = 300, 1000, 4
    plane, x_all = synth.workload(n, k, "e4m3fn_b128", seed=5)
    w, f, x = plane.w, plane.scale, np.ascontiguousarray(x_all[:m])
    y64, mag = oracle.gemv_b128_f64(w, f, x, threads=8)
    ok, worst = oracle.within_tolerance(oracle.gemv_b128(w, f, x, threads=8), y64, mag)
    assert ok, worst
    xs = x.copy()
    xs[:, 96:128], xs[:, 128:160] = x[:, 128:160], x[:, 96:128]  # across a block edge
    wrong = {
        "next column block's factor": (w, np.ascontiguousarray(np.roll(f, -1, axis=1)), x),
        "next row block's factor": (w, np.ascontiguousarray(np.roll(f, -1, axis=0)), x),
        "K blocks swapped across a factor edge": (w, f, xs),
    }
    for name, (wm, fm, xm) in wrong.items():
        ok, worst = oracle.within_tolerance(oracle.gemv_b128(wm, fm, xm, threads=8), y64, mag)
        assert not ok, f"{name} passes the tolerance (worst {worst:.3g})"
