"""Pins for the oracle's GEMV on block-scaled FP8 planes (CPU only).

The GLM-5.2 anatomy page runs fused_qkv_a_proj through AITER's preshuffle
blockscale GEMM, and the ATOM Model Support Guide (Weight loading) loads a
checkpoint's weight_scale_inv tensors as the layers' weight scales.  Reading
taken (the pages fix neither): one fp32 factor per 128 x 128 block of W,
applied, as the PR applies its row factor, to a finished sum -- the sum of
the block's 128 columns.  Per row and token the oracle forms each block's
partial sum in fp32 (ascending k), multiplies it by the block's factor,
adds it to an fp32 total (blocks ascending) and rounds the total to bf16
once.  These tests hold it to:

* an independent fp64 brute force (torch's float8_e4m3fn decode, numpy
  expansion of the factors, numpy matmul) on small ragged inputs;
* one-hot tokens: y = bf16(factor * code) with each block's own factor
  (distinct powers of two per block, so a transposed or wrongly sized block
  index shows);
* exact-sum inputs against Fraction arithmetic;
* a plane of one column block reduces to the row-scaled GEMV of the PR
  (pinned on its own) with scale[n] = the factor of n's row block, bit for
  bit on any inputs;
* factors times 2 double every output exactly.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _decode_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _brute_f64(w, bs, x, k):
    n = w.shape[0]
    f = np.repeat(np.repeat(bs.astype(np.float64), 128, axis=0)[:n], 128, axis=1)[:, :k]
    wd = _decode_table()[w[:, :k]] * f
    return oracle.bf16_bits_to_f64(x[:, :k]) @ wd.T


def _finite_codes(rng, shape, e_lo=1, e_hi=15):
    e = rng.integers(e_lo, e_hi, shape)
    return ((rng.integers(0, 2, shape) << 7) | (e << 3) | rng.integers(0, 8, shape)).astype(np.uint8)


def _factors(rng, n, k, lo=-12, hi=-4):
    shape = (-(-n // 128), -(-k // 128))
    return (rng.uniform(0.5, 1.0, shape) * 2.0 ** rng.integers(lo, hi, shape)).astype(np.float32)


@pytest.mark.parametrize("seed,n,k,m", [(0, 7, 5, 1), (1, 130, 300, 4), (2, 256, 256, 3),
                                        (3, 300, 129, 2), (4, 1, 1, 1), (5, 129, 640, 9)])
def test_b128_gemv_against_fp64_brute_force(orc, seed, n, k, m):
    rng = np.random.default_rng(seed)
    w = _finite_codes(rng, (n, k))
    bs = _factors(rng, n, k)
    x = oracle.f32_to_bf16_rne(rng.standard_normal((m, k), dtype=np.float32))
    ref = _brute_f64(w, bs, x, k)
    y64, mag = orc.gemv_b128_f64(w, bs, x)
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-300)
    ok, worst = oracle.within_tolerance(orc.gemv_b128(w, bs, x), ref, mag)
    assert ok, worst


def test_b128_one_hot_picks_each_blocks_factor(orc):
    n, k = 300, 384  # 3 x 3 blocks, the last row block ragged
    rng = np.random.default_rng(7)
    w = _finite_codes(rng, (n, k), 4, 12)
    # distinct powers of two per block: factor(rb, cb) = 2^(3 rb + cb - 6)
    rb, cb = np.meshgrid(np.arange(3), np.arange(3), indexing="ij")
    bs = (2.0 ** (3 * rb + cb - 6)).astype(np.float32)
    cols = [0, 127, 128, 200, 255, 256, 383]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    y = orc.gemv_b128(w, bs, x)
    table = _decode_table()
    for i, c in enumerate(cols):
        want = np.array([table[w[r, c]] * 2.0 ** (3 * (r // 128) + c // 128 - 6) for r in range(n)])
        got = oracle.bf16_bits_to_f64(y[i])
        np.testing.assert_array_equal(got, oracle.bf16_bits_to_f64(oracle.f64_to_bf16_rne(want)))


def test_b128_exact_sum_inputs_match_rational_result(orc):
    rng = np.random.default_rng(8)
    n, k, m = 140, 300, 3
    w = _finite_codes(rng, (n, k), 6, 10)  # |W| in [2^-1, 2^3)
    bs = (2.0 ** rng.integers(-3, 3, (2, 3))).astype(np.float32)
    x = oracle.f32_to_bf16_rne(rng.integers(-8, 9, (m, k)).astype(np.float32))
    y = orc.gemv_b128(w, bs, x)
    table = _decode_table()
    for i in range(m):
        for r in range(0, n, 7):
            acc = Fraction(0)
            for j in range(k):
                acc += (Fraction(float(bs[r // 128, j // 128])) * Fraction(float(table[w[r, j]]))
                        * Fraction(oracle.bf16_to_f32(int(x[i, j]))))
            want = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_rne(np.array([float(acc)])))[0]
            assert oracle.bf16_bits_to_f64(y[i:i + 1, r])[0] == want, (i, r)


def test_b128_one_column_block_is_the_row_scaled_gemv(orc):
    rng = np.random.default_rng(9)
    n, k, m = 300, 100, 5
    w = _finite_codes(rng, (n, k))
    bs = _factors(rng, n, k)
    x = oracle.f32_to_bf16_rne(rng.standard_normal((m, k), dtype=np.float32))
    scale = np.ascontiguousarray(bs[np.arange(n) // 128, 0])
    assert oracle.same_values(orc.gemv_b128(w, bs, x), orc.gemv(w, oracle.DT_E4M3FN, scale, x))


def test_b128_factor_doubling_doubles_exactly(orc):
    rng = np.random.default_rng(10)
    n, k, m = 200, 400, 4
    w = _finite_codes(rng, (n, k), 5, 12)
    bs = _factors(rng, n, k)
    x = oracle.f32_to_bf16_rne(rng.standard_normal((m, k), dtype=np.float32))
    y1 = oracle.bf16_bits_to_f64(orc.gemv_b128(w, bs, x))
    y2 = oracle.bf16_bits_to_f64(orc.gemv_b128(w, (bs * 2).astype(np.float32), x))
    np.testing.assert_array_equal(y2, 2 * y1)
