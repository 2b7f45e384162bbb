"""GPU parity of the GEMV on block-scaled FP8 planes, through the C ABI.

A block-scaled plane (W8_DT_E4M3FN_B128) holds E4M3fn codes and one fp32
factor per 128 x 128 block (the blockscale GEMM that the GLM-5.2 anatomy page
names for fused_qkv_a_proj; a checkpoint's weight_scale_inv).  w8_gemv sums
each 128-column block of a row, multiplies the block's sum by its factor and
adds it to the row's fp32 total, then rounds once to bf16 (register-ring
kernel, 1..64 tokens).  Checked against the oracle:

* bind copies the factors, sets the row scales to 1 and packs the codes as
  an E4M3FN bind of the same codes does;
* random seeded inputs over ragged N and K -- warp K parts and split-K CTAs
  that begin inside a column block, every token-group count, a plane whose
  warps stream more than 32 column blocks -- within the GEMV tolerance of
  the oracle's fp64 recompute;
* exact-sum inputs (power-of-two factors) and one-hot tokens bit for bit;
* a row holding a NaN code, a zero factor;
* the full-size fused_qkv_a_proj and o_proj shapes on sampled rows;
* the refusals: other entry points, more than 64 tokens.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_weight_only_w8a16_gb300 import synth

from .gpu_util import dev, from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_weight_only_w8a16_gb300 import w8 as lib

    return lib


def _ldw(k):
    return -(-k // 16) * 16


def _bind(w8, w, factors, k):
    w_d = to_dev(w)
    f_d = to_dev(np.ascontiguousarray(factors, dtype=np.float32))
    return w8.bind([w8.Plane.e4m3_b128(w_d, f_d, k=k)]), (w_d, f_d)


def _run(w8, b, x, n, ws=None):
    m, k = x.shape
    xp = torch.zeros((m, -(-k // 8) * 8), dtype=torch.int16, device=dev())
    xp[:, :k] = to_dev(x)
    y = torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev())
    w8.w8_gemv(b, 0, xp[:, :k], y, b.new_workspace() if ws is None else ws)
    torch.cuda.synchronize()
    return from_dev(y)


def _case(seed, n, k, m):
    rng = np.random.default_rng(seed)
    plane = synth.weight_plane(rng, n, k, "e4m3fn_b128", _ldw(k))
    return plane, synth.activations(rng, k, m)


def test_bind_copies_factors_and_packs_like_fp8(w8):
    plane, _ = _case(1, 300, 500, 1)
    b, _src = _bind(w8, plane.w, plane.scale, plane.k)
    info = b.info(0)
    assert info.dtype == w8.DT_E4M3FN_B128 and info.layout == w8.LAYOUT_MMA_16x32
    nf = plane.scale.size
    base = info.block_factors - b.dst.data_ptr()
    got = b.dst[base: base + 4 * nf].cpu().numpy().view(np.float32).reshape(plane.scale.shape)
    assert np.array_equal(got, plane.scale)
    sb = info.scale - b.dst.data_ptr()
    rows = b.dst[sb: sb + 4 * 300].cpu().numpy().view(np.float32)
    assert np.all(rows == 1.0)
    # the codes are packed exactly as a row-scaled bind of the same codes packs them
    b8 = w8.bind([w8.Plane.from_tensor(to_dev(plane.w), to_dev(np.ones(300, np.float32)),
                                       k=plane.k)])
    i8 = b8.info(0)
    assert i8.packed_bytes == info.packed_bytes
    p0 = info.packed - b.dst.data_ptr()
    p8 = i8.packed - b8.dst.data_ptr()
    assert torch.equal(b.dst[p0: p0 + info.packed_bytes].cpu(),
                       b8.dst[p8: p8 + i8.packed_bytes].cpu())


SHAPES = [(256, 512, 1), (300, 500, 4), (37, 77, 8), (1, 1, 1), (129, 3000, 16), (513, 1000, 33),
          (130, 2100, 64), (37, 5000, 3), (2624, 6144, 5), (6144, 2048, 32), (4096, 6144, 64),
          (200, 131, 2)]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_random_inputs_within_tolerance(w8, n, k, m):
    plane, x = _case(n + 3 * k + m, n, k, m)
    b, _src = _bind(w8, plane.w, plane.scale, k)
    assert b.plan(0, m).kernel == 0
    y = _run(w8, b, x, n)
    y64, mag = oracle.gemv_b128_f64(plane.w, plane.scale, x, k=k, threads=8)
    ok, worst = oracle.within_tolerance(y, y64, mag)
    assert ok, worst


def test_warps_past_32_column_blocks(w8):
    # [2432, 49152] at one token: each warp streams 192 K blocks (48 column
    # blocks), so the warp's window of 32 factors moves on once
    n, k = 2432, 49152
    plane, x_all = _case(11, n, k, 4)
    b, _src = _bind(w8, plane.w, plane.scale, k)
    assert b.plan(0, 1).k_blocks_per_warp_max > 128
    rows = np.unique(np.concatenate([np.random.default_rng(3).choice(n, 64, replace=False),
                                     [0, n - 1]]))
    for m in (1, 4):
        x = np.ascontiguousarray(x_all[:m])
        y = _run(w8, b, x, n)
        y64, mag = _oracle_rows_f64(plane, rows, x, k)
        ok, worst = oracle.within_tolerance(y[:, rows], y64, mag)
        assert ok, (m, worst)


def _oracle_rows_f64(plane, rows, x, k):
    """The oracle's fp64 recompute on sampled rows only: the rows of one row
    block at a time, with that block's factor row (so the oracle's row i of
    the group reads factor row 0, the group's own)."""
    y64 = np.zeros((x.shape[0], len(rows)))
    mag = np.zeros_like(y64)
    for rb in np.unique(rows // 128):
        sel = np.nonzero(rows // 128 == rb)[0]
        yg, mg = oracle.gemv_b128_f64(np.ascontiguousarray(plane.w[rows[sel]]),
                                      np.ascontiguousarray(plane.scale[rb:rb + 1]), x, k=k,
                                      threads=8)
        y64[:, sel] = yg
        mag[:, sel] = mg
    return y64, mag


def _exact_case(rng, n, k, m):
    # |W| < 4 in steps of 2^-4, integer |x| <= 4, factors 2^-1 .. 2^1: every
    # block sum is a multiple of 2^-4 below 2^11, every scaled one a multiple
    # of 2^-5, and a row total of up to 48 blocks stays below 2^18 -- all
    # exact in fp32, whatever the order
    e = rng.integers(6, 9, (n, k))
    w = ((rng.integers(0, 2, (n, k)) << 7) | (e << 3) | rng.integers(0, 8, (n, k))).astype(np.uint8)
    wp = np.zeros((n, _ldw(k)), np.uint8)
    wp[:, :k] = w
    f = (2.0 ** rng.integers(-1, 2, (-(-n // 128), -(-k // 128)))).astype(np.float32)
    x = synth.to_bf16_bits(rng.integers(-4, 5, (m, k)).astype(np.float32))
    return wp, f, x


@pytest.mark.parametrize("n,k,m", [(16, 32, 1), (300, 700, 5), (130, 3000, 16), (64, 6144, 8),
                                   (2624, 512, 64), (37, 5000, 2)])
def test_exact_sum_inputs_bit_exact(w8, n, k, m):
    rng = np.random.default_rng(n + k + m)
    w, f, x = _exact_case(rng, n, k, m)
    b, _src = _bind(w8, w, f, k)
    y = _run(w8, b, x, n)
    assert oracle.same_values(y, oracle.gemv_b128(w, f, x, k=k))


def test_one_hot_tokens_pick_each_blocks_factor(w8):
    n, k = 300, 384
    rng = np.random.default_rng(12)
    w, _, _ = _exact_case(rng, n, k, 1)
    rb, cb = np.meshgrid(np.arange(3), np.arange(3), indexing="ij")
    f = (1.5 * 2.0 ** (3 * rb + cb - 6)).astype(np.float32)
    cols = [0, 31, 127, 128, 200, 255, 256, 383]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    b, _src = _bind(w8, w, f, k)
    assert oracle.same_values(_run(w8, b, x, n), oracle.gemv_b128(w, f, x, k=k))


def test_nan_code_row_and_zero_factor(w8):
    n, k, m = 256, 512, 3
    plane, x = _case(13, n, k, m)
    w = plane.w.copy()
    w[5, 300] = 0x7F          # row 5 holds a NaN code
    f = plane.scale.copy()
    f[1, 2] = 0.0             # rows 128.., columns 256..383 contribute nothing
    b, _src = _bind(w8, w, f, k)
    y = _run(w8, b, x, n)
    yv = oracle.bf16_bits_to_f64(y)
    assert np.all(np.isnan(yv[:, 5]))
    want = oracle.gemv_b128(w, f, x, k=k)
    assert np.all(np.isnan(oracle.bf16_bits_to_f64(want)[:, 5]))
    keep = np.ones(n, bool)
    keep[5] = False
    y64, mag = oracle.gemv_b128_f64(w, f, x, k=k)
    ok, worst = oracle.within_tolerance(y[:, keep], y64[:, keep], mag[:, keep])
    assert ok, worst


@pytest.mark.parametrize("n,k,ms", [(2624, 6144, (1, 4, 16)), (6144, 16384, (1, 8, 32))],
                         ids=["fused_qkv_a_proj_b128", "o_proj_b128"])
def test_full_size_sampled(w8, n, k, ms):
    plane, x_all = synth.workload(n, k, "e4m3fn_b128", seed=0)
    b, _src = _bind(w8, plane.w, plane.scale, k)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(n, 96, replace=False), [0, n - 1]]))
    for m in ms:
        x = np.ascontiguousarray(x_all[:m])
        y = _run(w8, b, x, n)
        y64, mag = _oracle_rows_f64(plane, rows, x, k)
        ok, worst = oracle.within_tolerance(y[:, rows], y64, mag)
        assert ok, (m, worst)


def test_refusals(w8):
    plane, x = _case(9, 64, 256, 2)
    b, _src = _bind(w8, plane.w, plane.scale, 256)
    xd = to_dev(x)
    y = torch.zeros((2, 64), dtype=torch.int16, device=dev())
    for fn in (w8.bf16_gemv, w8.mxfp4_gemv):
        with pytest.raises(w8.W8Error) as e:
            fn(b, 0, xd, y)
        assert e.value.name == "W8_ERR_DTYPE"
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_silu_mul(b, 0, xd, y)
    assert e.value.name == "W8_ERR_LAYOUT"
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_noalloc(b, 0, xd, y)
    assert e.value.name == "W8_ERR_DTYPE"
    big = torch.zeros((65, 256), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv(b, 0, big, torch.zeros((65, 64), dtype=torch.int16, device=dev()))
    assert e.value.name == "W8_ERR_SHAPE"
    with pytest.raises(w8.W8Error) as e:
        b.plan(0, 65)
    assert e.value.name == "W8_ERR_SHAPE"
    torch.cuda.synchronize()
    assert torch.all(y == 0)
