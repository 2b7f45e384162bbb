"""Pins for the oracle's SiLU-and-multiply and its fp64 -> bf16 rounding (CPU only).

After a merged gate_up projection the MLP applies h = silu(g) * u with
silu(v) = v / (1 + exp(-v)) (ATOM Model Support Guide, Model architecture
details, Llama MLP; gate_proj is shard 0 and up_proj shard 1 of gate_up_proj,
Adding a new model, Step 5).  The oracle evaluates it in fp64 and rounds once
to bf16.  These tests hold it to things it cannot agree with by
construction:

* the one-step fp64 -> bf16 rounding equals the pinned fp32 rounding and
  torch's on every fp32-representable value, and on exact bf16 midpoints
  (and a hair either side, below fp32 resolution) it goes to the even
  neighbour (resp. the nearer one), which a detour through fp32 would not;
* silu(v) * u against torch's float64 silu, a closed form at v = ln 3
  (sigmoid = 3/4), the odd-part identity silu(v) - silu(-v) = v, the limits
  silu(v) = v for large v and the special values;
* the Lipschitz constant the parity tolerance uses, sup |silu'| = 1.0998...;
* the composed gated projection against an fp64 brute force, each output
  the nearest bf16 of the exact result on exact-sum inputs.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

DT8, DT16 = 1, 2


def _bits_to_f64(bits):
    return oracle.bf16_bits_to_f64(np.asarray(bits, dtype=np.uint16))


def _torch_bf16_bits(v32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _fp32_sample(rng, n=4000):
    """fp32 values over the whole range: normals, subnormals, edges."""
    exps = rng.integers(-149, 128, n)
    mant = rng.random(n) + 1.0
    v = np.ldexp(mant, exps).astype(np.float32)
    v = v * np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    edges = np.array([0.0, -0.0, np.inf, -np.inf, np.finfo(np.float32).max,
                      -np.finfo(np.float32).max, np.finfo(np.float32).tiny,
                      np.float32(1.4e-45), 3.3895314e38, 3.3961776e38, 1.0, -2.5],
                     dtype=np.float32)
    return np.concatenate([v, edges])


def test_f64_rounding_agrees_with_fp32_rounding_on_fp32_values(orc):
    rng = np.random.default_rng(11)
    v = _fp32_sample(rng)
    got = orc.f64_to_bf16_rne(v.astype(np.float64))
    assert np.array_equal(got, orc.f32_to_bf16_rne(v))
    finite = np.isfinite(v)
    assert np.array_equal(got[finite], _torch_bf16_bits(v[finite]))
    nan = orc.f64_to_bf16_rne(np.array([np.nan, -np.nan]))
    assert all(((b & 0x7F80) == 0x7F80) and (b & 0x7F) for b in nan)


def _midpoint_cases(rng):
    """(value, expected bits): exact midpoints of adjacent bf16 patterns of
    one sign and values a hair (2^-30 relative) either side of them."""
    lo = np.concatenate([rng.integers(0x0001, 0x7F7F, 600), np.arange(0x0000, 0x0080),
                         np.array([0x7F7E, 0x7F7F, 0x0080, 0x007F])]).astype(np.uint32)
    cases = []
    for a in lo:
        b = a + 1
        va = float(_bits_to_f64([a])[0])
        vb = math.inf if b == 0x7F80 else float(_bits_to_f64([b])[0])
        if b == 0x7F80:
            mid = (va + 2.0 ** 128) / 2.0
        else:
            mid = (va + vb) / 2.0
        even = a if a % 2 == 0 else b
        for sign, sbit in ((1.0, 0), (-1.0, 0x8000)):
            cases.append((sign * mid, even | sbit))
            cases.append((sign * mid * (1 + 2.0 ** -30), b | sbit))
            cases.append((sign * mid * (1 - 2.0 ** -30), a | sbit))
    return cases


def test_f64_rounding_on_exact_midpoints(orc):
    rng = np.random.default_rng(12)
    cases = _midpoint_cases(rng)
    vals = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    got = orc.f64_to_bf16_rne(vals)
    assert np.array_equal(got, want)


def test_silu_mul_matches_torch_float64_silu(orc):
    rng = np.random.default_rng(13)
    g = np.concatenate([rng.normal(0, 3, 3000), np.linspace(-800, 800, 1601),
                        np.array([0.0, -0.0, 1e-300, -1e-300, 700.0, -700.0, 40.0, -40.0])])
    u = rng.normal(0, 2, g.shape)
    got = orc.silu_mul_f64(g, u)
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-300)


def test_silu_closed_forms_and_limits(orc):
    # ln 3: exp(-v) = 1/3, so silu(v) = 3v/4
    v = math.log(3.0)
    assert orc.silu_mul_f64(v, 1.0)[()] == pytest.approx(0.75 * v, rel=4e-16)
    assert orc.silu_mul_f64(-v, 1.0)[()] == pytest.approx(-0.25 * v, rel=4e-16)
    # silu(0) = 0; for v >= 40, 1 + exp(-v) rounds to 1 in fp64: silu(v) = v
    big = np.array([40.0, 100.0, 1e6, 1e300])
    assert np.array_equal(orc.silu_mul_f64(big, 1.0), big)
    assert orc.silu_mul_f64(0.0, 5.0)[()] == 0.0
    # very negative v: silu(v) ~ v e^v
    for w in (-40.0, -100.0, -600.0):
        assert orc.silu_mul_f64(w, 1.0)[()] == pytest.approx(w * math.exp(w), rel=1e-13)
    # special values
    h = orc.silu_mul_f64(np.array([np.inf, -np.inf, np.nan, 3.0]),
                         np.array([2.0, 2.0, 1.0, 0.0]))
    assert h[0] == np.inf and np.isnan(h[1]) and np.isnan(h[2]) and h[3] == 0.0


def test_silu_odd_part_identity(orc):
    # v sigmoid(v) - (-v) sigmoid(-v) = v (sigmoid(v) + sigmoid(-v)) = v
    g = np.random.default_rng(14).normal(0, 6, 5000)
    u = np.full_like(g, 1.0)
    d = orc.silu_mul_f64(g, u) - orc.silu_mul_f64(-g, u)
    np.testing.assert_allclose(d, g, rtol=4e-15, atol=1e-300)
    # and u scales the result linearly (exactly, for a power of two)
    np.testing.assert_array_equal(orc.silu_mul_f64(g, 4.0), 4.0 * orc.silu_mul_f64(g, 1.0))


def test_silu_lipschitz_constant(orc):
    # the parity tolerance bounds |silu(a) - silu(b)| by L |a - b|
    g = np.linspace(-30.0, 30.0, 600001)
    s = orc.silu_mul_f64(g, 1.0)
    slope = np.abs(np.diff(s) / np.diff(g))
    assert slope.max() <= oracle.SILU_LIPSCHITZ
    assert slope.max() > 1.099  # and it is tight: silu' peaks at 1.0998 near v = 2.40


def _exact_gate_up_case(seed, half, k, m):
    """Codes of a narrow band (1..4 x 2^j), unit scales and small integer
    activations: every partial sum is an integer far below 2^24, so the
    projection's outputs are exact whatever the summation order."""
    rng = np.random.default_rng(seed)
    mags = np.array([0x38, 0x40, 0x44, 0x48], dtype=np.uint8)  # 1, 2, 3, 4
    w = mags[rng.integers(0, 4, (2 * half, k))] | np.where(rng.random((2 * half, k)) < 0.5,
                                                           0x80, 0).astype(np.uint8)
    xv = rng.integers(-3, 4, (m, k)).astype(np.float32)
    x = _torch_bf16_bits(xv)
    return w, np.ones(2 * half, dtype=np.float32), x


def test_gate_up_silu_mul_is_nearest_bf16_of_exact_result(orc):
    half, k, m = 24, 12, 5
    w, scale, x = _exact_gate_up_case(15, half, k, m)
    h = orc.gate_up_silu_mul(w, DT8, scale, x)
    y = brute.gemv_f64_brute(w, True, scale, x, k)  # exact integers
    assert np.all(np.abs(y) < 256) and np.array_equal(y, np.round(y))
    big_h = (torch.nn.functional.silu(torch.from_numpy(y[:, :half]))
             * torch.from_numpy(y[:, half:])).numpy()
    hv = _bits_to_f64(h)
    # nearest: no bf16 neighbour of h is closer to the exact value
    up = _bits_to_f64(np.where(hv >= 0, h + 1, h - 1).astype(np.uint16))
    dn = _bits_to_f64(np.where(hv > 0, h - 1, np.where(hv < 0, h + 1, h)).astype(np.uint16))
    err = np.abs(hv - big_h)
    assert np.all(err <= np.abs(up - big_h) * (1 + 1e-12))
    assert np.all(err <= np.abs(dn - big_h) * (1 + 1e-12))
    assert np.all(err <= 2.0 ** -8 * np.abs(big_h) + 1e-300)


@pytest.mark.parametrize("fp8", [True, False])
def test_gate_up_silu_mul_against_fp64_brute_force(orc, fp8):
    from fp8_weight_only_w8a16_gb300 import synth

    rng = np.random.default_rng(16 + fp8)
    half, k, m = 40, 96, 7
    plane = synth.weight_plane(rng, 2 * half, k, "e4m3fn" if fp8 else "bf16")
    x = synth.activations(rng, k, m)
    dt = DT8 if fp8 else DT16
    h = orc.gate_up_silu_mul(plane.w, dt, plane.scale, x)
    assert h.shape == (m, half)
    y64 = brute.gemv_f64_brute(plane.w, fp8, plane.scale, x, k)
    _, mag = orc.gemv_f64(plane.w, dt, plane.scale, x)
    ok, worst = oracle.silu_mul_within_tolerance(h, y64[:, :half], mag[:, :half],
                                                 y64[:, half:], mag[:, half:])
    assert ok, worst
    # the gate half and the up half are not interchangeable
    swapped = orc.silu_mul(orc.gemv(plane.w, dt, plane.scale, x)[:, half:],
                           orc.gemv(plane.w, dt, plane.scale, x)[:, :half])
    assert not oracle.silu_mul_within_tolerance(swapped, y64[:, :half], mag[:, :half],
                                                y64[:, half:], mag[:, half:])[0]
