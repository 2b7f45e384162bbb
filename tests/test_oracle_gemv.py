"""Pins for the oracle's GEMV (CPU only).

The oracle computes y[m,n] = bf16_rne(scale[n] * sum_k W[n,k] x[m,k]) with
fp32 accumulation in ascending k (ATOM PR #2980, Summary and Changes: each
E4M3 code has an exact bf16 value, and the fp32 row factor is applied to the
finished row sum ahead of the one conversion to bf16).  These tests pin it to
things it cannot agree with by construction:

* an independent fp64 brute force (torch dtypes + numpy matmul) on tiny
  inputs, within the stated tolerance, and the oracle's own fp64 recompute
  equal to it to fp64 rounding;
* one-hot activations, which must return bf16(scale[n] * W[n,k]) for every
  k and for all 254 finite codes;
* exact-sum inputs, where every order of summation gives the exact rational
  sum, against Fraction arithmetic;
* power-of-two scales, which commute with every rounding away from
  overflow and subnormals;
* the fp32 sequential-sum error bound gamma_K on larger random inputs.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import brute

DT8, DT16 = 1, 2


def _f32(v):
    return np.float32(v)


def _bf16_bits_of(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _random_case(seed, n, k, m, fp8=True, ldw=None, ldx=None):
    from fp8_weight_only_w8a16_gb300 import synth

    rng = np.random.default_rng(seed)
    plane = synth.weight_plane(rng, n, k, "e4m3fn" if fp8 else "bf16", ldw)
    x = synth.activations(rng, k, m, ldx)
    return plane, x


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("seed,n,k,m", [(0, 7, 5, 1), (1, 16, 32, 4), (2, 33, 64, 16),
                                        (3, 64, 48, 3), (4, 1, 1, 1), (5, 40, 63, 9)])
def test_gemv_against_fp64_brute_force(orc, fp8, seed, n, k, m):
    plane, x = _random_case(seed, n, k, m, fp8)
    dt = DT8 if fp8 else DT16
    y = orc.gemv(plane.w, dt, plane.scale, x)
    ref = brute.gemv_f64_brute(plane.w, fp8, plane.scale, x, k)
    y64, mag = orc.gemv_f64(plane.w, dt, plane.scale, x)
    # the oracle's fp64 recompute is the brute force up to fp64 rounding
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-300)
    ok, worst = orc.within_tolerance(y, ref, mag)
    assert ok, worst
    # and it is far tighter than that: fp32 sum error <= k * 2^-24 * mag,
    # then one bf16 rounding (half an ulp, 2^-8 relative)
    yv = orc.bf16_bits_to_f64(y)
    assert np.all(np.abs(yv - ref) <= 2.0 ** -8 * np.abs(ref) * (1 + 2.0 ** -8)
                  + (k + 2) * 2.0 ** -24 * mag * 1.01 + 1e-300)


def test_mag_is_sum_of_absolute_products(orc):
    plane, x = _random_case(7, 9, 20, 3, True)
    _, mag = orc.gemv_f64(plane.w, DT8, plane.scale, x)
    wd = brute.decode_e4m3_lib(plane.w)
    xd = brute.decode_bf16_lib(x)
    want = np.abs(xd) @ np.abs(wd).T * np.abs(plane.scale.astype(np.float64))[None, :]
    assert np.allclose(mag, want, rtol=1e-12)


def _all_finite_codes_plane():
    """[16, 16] plane holding every code except the two NaNs (2 slots get 0)."""
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    codes += [0x00, 0x80]
    return np.array(codes, dtype=np.uint8).reshape(16, 16)


@pytest.mark.parametrize("scale_kind", ["ones", "random"])
def test_one_hot_returns_scaled_code(orc, scale_kind):
    w = _all_finite_codes_plane()
    n, k = w.shape
    rng = np.random.default_rng(11)
    scale = (np.ones(n, np.float32) if scale_kind == "ones"
             else rng.uniform(0.001, 3.0, n).astype(np.float32))
    x = np.zeros((k, k), dtype=np.uint16)
    x[np.arange(k), np.arange(k)] = 0x3F80  # bf16 1.0
    y = orc.gemv(w, DT8, scale, x)          # [k tokens, n rows]
    wd = brute.decode_e4m3_lib(w).astype(np.float32)
    # token j picks column j; the sum starts at +0, so a -0 code sums to +0
    want = _bf16_bits_of(scale[None, :] * (np.float32(0.0) + wd.T))
    assert np.array_equal(y, want)


def test_one_hot_bf16_plane_returns_weight(orc):
    rng = np.random.default_rng(12)
    w = _bf16_bits_of(rng.standard_normal((8, 24)).astype(np.float32))
    x = np.zeros((24, 24), dtype=np.uint16)
    x[np.arange(24), np.arange(24)] = 0x3F80
    y = orc.gemv(w, DT16, None, x)
    assert np.array_equal(y, w.T)


def test_exact_sum_inputs_match_rational_result(orc):
    """Codes from a narrow exponent band and small-integer activations: every
    partial sum is a multiple of 2^-7 below 2^17, so fp32 holds it exactly
    and the result is the exact rational sum, rounded once to fp32 by the
    power-of-two scale (exact) and once to bf16."""
    rng = np.random.default_rng(13)
    n, k, m = 24, 64, 5
    e = rng.integers(5, 10, (n, k))           # exponent field 5..9
    mant = rng.integers(0, 8, (n, k))
    sign = rng.integers(0, 2, (n, k))
    w = ((sign << 7) | (e << 3) | mant).astype(np.uint8)
    xv = rng.integers(-8, 9, (m, k)).astype(np.float32)
    x = _bf16_bits_of(xv)
    scale = (2.0 ** rng.integers(-6, 3, n)).astype(np.float32)
    y = orc.gemv(w, DT8, scale, x)
    for i in range(m):
        for r in range(n):
            s = Fraction(0)
            for j in range(k):
                s += Fraction(orc.e4m3_to_f32(int(w[r, j]))) * Fraction(int(xv[i, j]))
            t = s * Fraction(float(scale[r]))
            assert float(t) == float(np.float32(float(t)))  # exact in fp32
            assert y[i, r] == _bf16_bits_of(np.array([float(t)], np.float32))[0]


def test_scale_multiplies_the_reduced_row_once(orc):
    """Exact-sum rows with arbitrary fp32 scales: the result must be
    bf16(fp32(scale * acc)) with acc the exact row sum -- one fp32 multiply of
    the reduced row, then one bf16 rounding (PR page, Changes: the factor is
    applied to the finished row sum, ahead of the conversion).  Scaling each product, or rounding
    acc to bf16 before scaling, gives other bits on many of these rows."""
    rng = np.random.default_rng(14)
    n, k, m = 32, 48, 4
    e = rng.integers(6, 11, (n, k))
    mant = rng.integers(0, 8, (n, k))
    sign = rng.integers(0, 2, (n, k))
    w = ((sign << 7) | (e << 3) | mant).astype(np.uint8)
    xv = rng.integers(-16, 17, (m, k)).astype(np.float32)
    x = _bf16_bits_of(xv)
    scale = rng.uniform(0.01, 5.0, n).astype(np.float32)
    y = orc.gemv(w, DT8, scale, x)
    wd = brute.decode_e4m3_lib(w)
    acc = xv.astype(np.float64) @ wd.T               # exact: integers * 2^-4 steps
    assert np.array_equal(acc.astype(np.float32).astype(np.float64), acc)
    t = scale[None, :] * acc.astype(np.float32)      # one IEEE fp32 multiply
    assert np.array_equal(y, _bf16_bits_of(t))


@pytest.mark.parametrize("j", [-5, 3])
def test_power_of_two_scale_commutes(orc, j):
    plane, x = _random_case(21, 48, 96, 6, True)
    y1 = orc.gemv(plane.w, DT8, plane.scale, x)
    y2 = orc.gemv(plane.w, DT8, (plane.scale * np.float32(2.0 ** j)).astype(np.float32), x)
    v1 = orc.bf16_bits_to_f64(y1)
    v2 = orc.bf16_bits_to_f64(y2)
    assert np.array_equal(v2, v1 * 2.0 ** j)


def test_padded_row_stride_and_padded_k_agree(orc):
    """Columns past K in a padded plane are ignored (row stride ldw > K), and
    zero pad codes with zero pad activations add exact zeros."""
    plane, x = _random_case(22, 20, 100, 4, True, ldw=100 + 28)
    y_pad = orc.gemv(plane.w, DT8, plane.scale, x[:, :100], k=100)
    dense = np.ascontiguousarray(plane.w[:, :100])
    y_dense = orc.gemv(dense, DT8, plane.scale, x[:, :100])
    assert np.array_equal(y_pad, y_dense)
    xk = np.zeros((4, 128), np.uint16)
    xk[:, :100] = x[:, :100]
    y_kpad = orc.gemv(plane.w, DT8, plane.scale, xk, k=128)
    assert np.array_equal(y_kpad, y_dense)


def test_nan_code_poisons_its_row_only(orc):
    plane, x = _random_case(23, 6, 40, 3, True)
    w = plane.w.copy()
    w[2, 17] = 0x7F
    y = orc.gemv(w, DT8, plane.scale, x)
    v = orc.bf16_bits_to_f64(y)
    assert np.all(np.isnan(v[:, 2]))
    assert not np.any(np.isnan(np.delete(v, 2, axis=1)))


def test_sequential_sum_error_bound_large_k(orc):
    """fp32 ascending-k error stays inside gamma_K * sum|terms| (plus the
    bf16 rounding) at a realistic K, and inside the parity tolerance."""
    plane, x = _random_case(24, 64, 6144, 2, True)
    y = orc.gemv(plane.w, DT8, plane.scale, x)
    y64, mag = orc.gemv_f64(plane.w, DT8, plane.scale, x)
    ok, worst = orc.within_tolerance(y, y64, mag)
    assert ok, worst
    yv = orc.bf16_bits_to_f64(y)
    gamma = 6144 * 2.0 ** -24
    assert np.all(np.abs(yv - y64) <= 2.0 ** -8 * np.abs(y64) * 1.01 + gamma * mag)


def test_threads_do_not_change_the_result(orc):
    plane, x = _random_case(25, 200, 300, 4, True)
    y1 = orc.gemv(plane.w, DT8, plane.scale, x, threads=1)
    y4 = orc.gemv(plane.w, DT8, plane.scale, x, threads=4)
    assert np.array_equal(y1, y4)


def test_workload_inputs_cover_every_token_count():
    # every workload's activations hold as many rows as its largest M, and
    # drawing more rows leaves the first ones unchanged
    from fp8_weight_only_w8a16_gb300 import synth, workloads

    mmax = max(max(p.ms) for p in workloads.ALL)
    _p, x = synth.workload(16, 64, seed=0)
    assert x.shape[0] >= mmax
    _p, x64 = synth.workload(16, 64, seed=0, x_rows=64)
    assert np.array_equal(x[:64], x64)
