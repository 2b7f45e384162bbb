"""Pins for the oracle's w4a16 GEMV on MXFP4 weights (CPU only).

The ATOM Model Support Guide (Model-specific optimizations, DeepSeek V2/V3:
FP4 support) names MXFP4 GEMMs with 16-bit activations, and the GLM-5.2
anatomy page's deployments serve a GLM-5.2-MXFP4 checkpoint.  MXFP4 is the
OCP microscaling format: E2M1 elements (sign, 2 exponent bits with bias 1, 1
mantissa bit, subnormal at exponent 0, no infinity or NaN), 32 consecutive
elements along K sharing an E8M0 scale 2^(e - 127) (255 = NaN).  The oracle
computes y = bf16(sum_k e2m1(W) * scale * x) with fp32 accumulation in
ascending k.  These tests hold it to:

* the 16 E2M1 codes against their closed form, and the E8M0 scales against
  the closed form and torch.float8_e8m0fnu;
* an independent fp64 brute force (numpy decode tables, numpy matmul) on tiny
  inputs, within the GEMV tolerance, and the oracle's fp64 recompute equal
  to it;
* one-hot activations over every code and edge scales (E8M0 0, 1, 127, 254,
  255), the nibble order (even column in the low nibble) and the block
  index (column / 32);
* exact-sum inputs against Fraction arithmetic, and power-of-two scale
  steps that double every output exactly.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _e2m1_closed(code: int) -> float:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = m / 2 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
    return -v if s else v


def test_e2m1_codes_closed_form(orc):
    got = [orc.e2m1_to_f32(c) for c in range(16)]
    assert got == [_e2m1_closed(c) for c in range(16)]
    # the format's value set: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives
    assert got[:8] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.signbit(got[8]) and got[9:] == [-v for v in got[1:8]]


def test_e8m0_scales_closed_form_and_torch(orc):
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for e in range(256):
        v = orc.e8m0_to_f32(e)
        if e == 255:
            assert np.isnan(v) and np.isnan(lib[e].item())
        else:
            assert v == 2.0 ** (e - 127) == lib[e].item()


def _decode_tables():
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    e2m1 = np.concatenate([mags, -mags])
    e8m0 = np.array([2.0 ** (e - 127) for e in range(255)] + [np.nan])
    return e2m1, e8m0


def _brute_f64(w, bs, x, k):
    """numpy decode of the packed plane and an fp64 matmul: [m, n]."""
    e2m1, e8m0 = _decode_tables()
    codes = np.empty((w.shape[0], 2 * w.shape[1]), dtype=np.int64)
    codes[:, 0::2] = w & 15
    codes[:, 1::2] = w >> 4
    wd = e2m1[codes[:, :k]] * np.repeat(e8m0[bs], 32, axis=1)[:, :k]
    xd = oracle.bf16_bits_to_f64(x[:, :k])
    return xd @ wd.T


def _random_plane(rng, n, k, e_lo=115, e_hi=125):
    nb = -(-k // 2)
    w = rng.integers(0, 256, (n, nb), dtype=np.uint8)
    if k % 2:
        w[:, -1] &= 15
    bs = rng.integers(e_lo, e_hi, (n, -(-k // 32)), dtype=np.uint8)
    return w, bs


@pytest.mark.parametrize("seed,n,k,m", [(0, 7, 5, 1), (1, 16, 32, 4), (2, 33, 64, 16),
                                        (3, 40, 100, 3), (4, 1, 1, 1), (5, 24, 257, 9)])
def test_mxfp4_gemv_against_fp64_brute_force(orc, seed, n, k, m):
    rng = np.random.default_rng(seed)
    w, bs = _random_plane(rng, n, k)
    x = oracle.f32_to_bf16_rne(rng.standard_normal((m, k), dtype=np.float32))
    y = orc.gemv_mxfp4(w, bs, x, k)
    ref = _brute_f64(w, bs, x, k)
    y64, mag = orc.gemv_mxfp4_f64(w, bs, x, k)
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-300)
    ok, worst = oracle.within_tolerance(y, ref, mag)
    assert ok, worst


def test_mxfp4_one_hot_codes_scales_and_packing(orc):
    # row r holds code c = r % 16 in every column; block scales vary; one-hot
    # tokens pick one column each: y = bf16(e2m1(c) * 2^(e - 127))
    n, k = 48, 96
    codes = np.arange(n) % 16
    w = np.repeat((codes | (codes << 4)).astype(np.uint8)[:, None], k // 2, axis=1)
    # make the odd columns of block 1 differ, so the nibble order matters
    w[:, 16:32] = (codes | (((codes + 3) % 16) << 4)).astype(np.uint8)[:, None]
    edge = np.array([0, 1, 127, 254, 255, 126, 130, 100, 10, 200, 127, 64], dtype=np.uint8)
    bs = np.stack([np.resize(edge, n), np.resize(edge[::-1], n), np.resize(np.roll(edge, 3), n)],
                  axis=1).astype(np.uint8)
    cols = [0, 1, 33, 34, 65, 95]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    y = orc.gemv_mxfp4(w, bs, x, k)
    # a row holding a weight that is NaN (E8M0 255) or past fp32's range
    # (6 x 2^127) is NaN wherever it meets a zero token (NaN x 0, inf x 0), as
    # the plain fp32 definition gives; every other output is bf16(W[r, c])
    e2m1, e8m0 = _decode_tables()
    codes_all = np.empty((n, k), dtype=np.int64)
    codes_all[:, 0::2] = w & 15
    codes_all[:, 1::2] = w >> 4
    deq = e2m1[codes_all] * np.repeat(e8m0[bs], 32, axis=1)[:, :k]
    poisoned = ~np.all(np.abs(deq) < 2.0 ** 128, axis=1)
    assert poisoned.any() and (~poisoned).any()
    for i, c in enumerate(cols):
        got = oracle.bf16_bits_to_f64(y[i])
        assert np.all(np.isnan(got[poisoned]))
        want = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_rne(deq[~poisoned, c]))
        assert np.array_equal(got[~poisoned], want), c
    # in block 1 the odd columns hold other codes: column 33 reads a high nibble
    assert not oracle.same_values(y[2][~poisoned], y[3][~poisoned])


def _exact_case(rng, n, k, m):
    # codes up to +-6 in halves, scales 2^-1..2^1, integer tokens: every
    # partial sum is a multiple of 1/4 far below 2^22
    w, _ = _random_plane(rng, n, k)
    bs = rng.integers(126, 129, (n, -(-k // 32)), dtype=np.uint8)
    x = oracle.f32_to_bf16_rne(rng.integers(-8, 9, (m, k)).astype(np.float32))
    return w, bs, x


def test_mxfp4_exact_sum_inputs_match_rational_result(orc):
    rng = np.random.default_rng(21)
    n, k, m = 12, 200, 3
    w, bs, x = _exact_case(rng, n, k, m)
    y = orc.gemv_mxfp4(w, bs, x, k)
    for i in range(m):
        for r in range(n):
            acc = Fraction(0)
            for j in range(k):
                code = (int(w[r, j // 2]) >> (4 * (j & 1))) & 15
                acc += (Fraction(_e2m1_closed(code)) * Fraction(2) ** (int(bs[r, j // 32]) - 127)
                        * Fraction(oracle.bf16_to_f32(int(x[i, j]))))
            assert oracle.bf16_bits_to_f64(y[i:i + 1, r])[0] == float(
                oracle.bf16_bits_to_f64(oracle.f64_to_bf16_rne(np.array([float(acc)])))[0])


def test_mxfp4_scale_steps_double_exactly(orc):
    rng = np.random.default_rng(22)
    w, bs, x = _exact_case(rng, 20, 160, 4)
    y1 = oracle.bf16_bits_to_f64(orc.gemv_mxfp4(w, bs, x))
    y2 = oracle.bf16_bits_to_f64(orc.gemv_mxfp4(w, (bs + 1).astype(np.uint8), x))
    np.testing.assert_array_equal(y2, 2 * y1)
