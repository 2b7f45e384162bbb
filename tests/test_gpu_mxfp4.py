"""GPU parity of the w4a16 GEMV on MXFP4 weights, through the C ABI.

MXFP4 (the OCP microscaling format that the ATOM Model Support Guide's FP4
GEMMs with 16-bit activations read, and that the GLM-5.2 anatomy page's
deployed GLM-5.2-MXFP4 checkpoint holds): E2M1 codes two a byte, an E8M0
scale per 32 columns.  mxfp4_gemv computes y = bf16(sum_k e2m1(W) 2^(e-127)
x) with fp32 accumulation on the register-ring kernel (1..64 tokens).
Checked against the oracle:

* the repack places every code bit where the host bit map says and writes
  each run's bf16 block-scale words;
* random seeded inputs over ragged N and K, every token-group count and
  split K, within the GEMV tolerance of the oracle's fp64 recompute;
* exact-sum inputs bit for bit; with every scale 1 the result equals the
  bf16 plane of the dequantized codes bit for bit (same summation order);
* one-hot tokens over every code and edge scales (E8M0 0, 1, 254, 255):
  each output exactly the oracle's, NaN rows included -- on a plane whose
  scales reach past 2^1 (two multiplies per code pair) and on one whose
  scales stay at or below it, down to E8M0 0 and up to 128 (2^126 folded
  into the stored factor at bind, one multiply);
* the two forms agree bit for bit on the rows they share;
* the full-size o_proj and q_b planes on sampled rows;
* the refusals: other entry points, other builds, more than 64 tokens.
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
    return -(-k // 32) * 32


def _case(seed, n, k, m):
    rng = np.random.default_rng(seed)
    plane = synth.weight_plane(rng, n, k, "mxfp4", _ldw(k))
    return plane, synth.activations(rng, k, m)


def _bind(w8, plane):
    w_d = to_dev(plane.w)
    s_d = to_dev(np.ascontiguousarray(plane.scale))
    return w8.bind([w8.Plane.mxfp4(w_d, s_d, k=plane.k)]), (w_d, s_d)


def _run(w8, b, x, n, fn=None):
    m, k = x.shape
    xp = torch.zeros((m, -(-k // 8) * 8), dtype=torch.int16, device=dev())
    xp[:, :k] = to_dev(x)
    y = torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev())
    (fn or w8.mxfp4_gemv)(b, 0, xp[:, :k], y, b.new_workspace())
    torch.cuda.synchronize()
    return from_dev(y)


@pytest.mark.parametrize("wide", [False, True], ids=["folded", "wide"])
@pytest.mark.parametrize("n,k", [(37, 77), (16, 32), (100, 300), (5, 1)])
def test_repack_matches_host_bit_map(w8, n, k, wide):
    plane, _ = _case(1, n, k, 1)
    if wide:  # one scale above 2^1: the plane keeps the plain scales
        plane.scale[n // 2, 0] = 131
    b, _src = _bind(w8, plane)
    info = b.info(0)
    assert info.dtype == w8.DT_MXFP4 and info.layout == w8.LAYOUT_MMA_16x32
    assert info.mxfp4_wide_scales == int(wide)
    rt, kb = info.row_tiles, info.k_blocks
    assert info.packed_bytes == rt * kb * 288
    base = info.packed - b.dst.data_ptr()
    packed = b.dst[base: base + info.packed_bytes].cpu().numpy()
    want = np.zeros(info.packed_bytes, dtype=np.uint8)
    for r in range(rt * 16):
        for c in range(kb * 32):
            code = int(plane.w[r, c // 2] >> (4 * (c & 1))) & 15 if (r < n and c < k) else 0
            for i, b in enumerate(w8.mxfp4_code_bits(kb, r, c)):
                want[b // 8] |= np.uint8(((code >> i) & 1) << (b % 8))
    # the scale words for rows g and g+8 of each run: bf16 of 2^126 x 2^(e - 127)
    # on a folded plane, of 2^(e - 127) on a wide one; NaN for e = 255
    def bf16_of(e):
        if e == 255:
            return 0x7FC0
        if not wide:
            return (int(e) + 126) << 7
        return 0x0040 if e == 0 else (int(e) << 7)
    for t in range(rt):
        for blk in range(kb):
            run = (t * kb + blk) * 288
            for g in range(8):
                lo = bf16_of(plane.scale[t * 16 + g, blk]) if t * 16 + g < n else 0
                hi = bf16_of(plane.scale[t * 16 + g + 8, blk]) if t * 16 + g + 8 < n else 0
                want[run + 256 + 4 * g: run + 260 + 4 * g] = np.frombuffer(
                    np.uint32(lo | (hi << 16)).tobytes(), dtype=np.uint8)
    assert np.array_equal(packed, want)


SHAPES = [(256, 512, 1), (100, 200, 4), (37, 77, 8), (1, 1, 1), (16, 32, 16), (513, 1000, 33),
          (130, 2100, 64), (64, 6144, 5), (6144, 2048, 32), (6144, 2048, 64)]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_random_inputs_within_tolerance(w8, n, k, m):
    plane, x = _case(n + k + m, n, k, m)
    b, _src = _bind(w8, plane)
    assert b.plan(0, m).kernel == 0  # MXFP4 runs the register ring
    y = _run(w8, b, x, n)
    y64, mag = oracle.gemv_mxfp4_f64(plane.w, plane.scale, x, k=k, threads=8)
    ok, worst = oracle.within_tolerance(y, y64, mag)
    assert ok, worst


def _exact_case(rng, n, k, m):
    w = rng.integers(0, 256, (n, _ldw(k) // 2), dtype=np.uint8)
    w[:, -(-k // 2):] = 0
    if k % 2:
        w[:, k // 2] &= 15
    bs = rng.integers(126, 129, (n, -(-k // 32)), dtype=np.uint8)
    x = synth.to_bf16_bits(rng.integers(-8, 9, (m, k)).astype(np.float32))
    return synth.Plane("mxfp4", n, k, _ldw(k), w, bs), x


@pytest.mark.parametrize("n,k,m", [(16, 32, 1), (64, 2048, 5), (300, 700, 16), (40, 6144, 8),
                                   (2624, 512, 64)])
def test_exact_sum_inputs_bit_exact(w8, n, k, m):
    rng = np.random.default_rng(n * 11 + k + m)
    plane, x = _exact_case(rng, n, k, m)
    b, _src = _bind(w8, plane)
    y = _run(w8, b, x, n)
    assert oracle.same_values(y, oracle.gemv_mxfp4(plane.w, plane.scale, x, k=k))


# (shapes where the bf16 plane also runs the register ring: same order)
@pytest.mark.parametrize("n,k,m", [(256, 512, 8), (2624, 6144, 16), (640, 2048, 64)])
def test_unit_scales_equal_the_bf16_plane(w8, n, k, m):
    plane, x = _case(3 * n + k, n, k, m)
    plane.scale[:] = 127
    b4, _s4 = _bind(w8, plane)
    # the bf16 plane of the dequantized codes (exact: E2M1 values are bf16)
    vals = np.array([oracle.e2m1_to_f32(c) for c in range(16)], dtype=np.float32)
    codes = np.empty((n, 2 * plane.w.shape[1]), dtype=np.int64)
    codes[:, 0::2] = plane.w & 15
    codes[:, 1::2] = plane.w >> 4
    wb = synth.to_bf16_bits(vals[codes[:, :k]])
    ldw16 = -(-k // 8) * 8
    wpad = np.zeros((n, ldw16), dtype=np.uint16)
    wpad[:, :k] = wb
    w_d = to_dev(wpad)
    b16 = w8.bind([w8.Plane.from_tensor(w_d, None, k=k, dtype=w8.DT_BF16)])
    y4 = _run(w8, b4, x, n)
    y16 = _run(w8, b16, x, n, fn=w8.bf16_gemv)
    assert oracle.same_values(y4, y16)


def test_one_hot_every_code_and_edge_scales(w8):
    n, k = 64, 96
    codes = np.arange(n) % 16
    w = np.repeat((codes | (((codes + 5) % 16) << 4)).astype(np.uint8)[:, None], k // 2, axis=1)
    edge = np.array([0, 1, 127, 254, 126, 130, 100, 10, 200, 127, 64, 120, 133], dtype=np.uint8)
    bs = np.stack([np.resize(edge, n), np.resize(edge[::-1], n), np.resize(np.roll(edge, 4), n)],
                  axis=1).astype(np.uint8)
    bs[5, 2] = 255  # a NaN block: row 5 is NaN everywhere
    plane = synth.Plane("mxfp4", n, k, k, w, bs)
    cols = [0, 1, 33, 34, 64, 95]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0x3F80
    b, _src = _bind(w8, plane)
    y = _run(w8, b, x, n)
    want = oracle.gemv_mxfp4(w, bs, x, k=k)
    assert oracle.same_values(y, want)
    assert np.all(np.isnan(oracle.bf16_bits_to_f64(y[:, 5])))


def test_one_hot_folded_edge_scales(w8):
    """The folded factor's range ends: E8M0 0 (2^-1 stored), 1, 127, 128 (2^127
    stored), with a NaN block; every output exactly the oracle's."""
    n, k = 64, 96
    codes = np.arange(n) % 16
    w = np.repeat((codes | (((codes + 7) % 16) << 4)).astype(np.uint8)[:, None], k // 2, axis=1)
    edge = np.array([0, 1, 127, 128, 126, 2, 100, 10, 120, 64, 125], dtype=np.uint8)
    bs = np.stack([np.resize(edge, n), np.resize(edge[::-1], n), np.resize(np.roll(edge, 3), n)],
                  axis=1).astype(np.uint8)
    bs[9, 1] = 255
    plane = synth.Plane("mxfp4", n, k, k, w, bs)
    cols = [0, 1, 33, 34, 64, 95]
    x = np.zeros((len(cols), k), dtype=np.uint16)
    for i, c in enumerate(cols):
        x[i, c] = 0xBF80  # -1: the signs too
    b, _src = _bind(w8, plane)
    assert b.info(0).mxfp4_wide_scales == 0
    y = _run(w8, b, x, n)
    assert oracle.same_values(y, oracle.gemv_mxfp4(w, bs, x, k=k))
    assert np.all(np.isnan(oracle.bf16_bits_to_f64(y[:, 9])))


@pytest.mark.parametrize("n,k,m", [(256, 512, 8), (300, 2100, 16), (2624, 6144, 1)])
def test_folded_and_wide_planes_agree(w8, n, k, m):
    """One plane bound twice: as drawn (every scale at most 2^1, folded) and
    with one block's scale raised past 2^1 (wide).  Every row but that one is
    the same bit for bit (both multiply exactly, in the same order); all rows
    are within the oracle's tolerance."""
    plane, x = _case(n * 3 + k + m, n, k, m)
    b1, _s1 = _bind(w8, plane)
    wide = synth.Plane("mxfp4", n, k, plane.ldw, plane.w, plane.scale.copy())
    r = n // 3
    wide.scale[r, 1] = 140
    b2, _s2 = _bind(w8, wide)
    assert b1.info(0).mxfp4_wide_scales == 0 and b2.info(0).mxfp4_wide_scales == 1
    y1, y2 = _run(w8, b1, x, n), _run(w8, b2, x, n)
    others = np.arange(n) != r
    assert oracle.same_values(y1[:, others], y2[:, others])
    for pl, y in ((plane, y1), (wide, y2)):
        y64, mag = oracle.gemv_mxfp4_f64(pl.w, pl.scale, x, k=k, threads=8)
        ok, worst = oracle.within_tolerance(y, y64, mag)
        assert ok, worst


@pytest.mark.parametrize("n,k,ms", [(6144, 16384, (1, 2, 8, 32)), (16384, 2048, (1, 8, 64)),
                                    (2624, 6144, (1, 4, 16))],
                         ids=["o_proj_mxfp4", "q_b_proj_mxfp4", "fused_qkv_a_proj_mxfp4"])
def test_full_size_sampled(w8, n, k, ms):
    plane, x_all = synth.workload(n, k, "mxfp4", seed=0, ldw=_ldw(k))
    b, _src = _bind(w8, plane)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(n, 96, replace=False), [0, n - 1]]))
    for m in ms:
        x = np.ascontiguousarray(x_all[:m])
        y = _run(w8, b, x, n)
        y64, mag = oracle.gemv_mxfp4_f64(np.ascontiguousarray(plane.w[rows]),
                                         np.ascontiguousarray(plane.scale[rows]), x, k=k, threads=8)
        ok, worst = oracle.within_tolerance(y[:, rows], y64, mag)
        assert ok, (m, worst)


def test_refusals(w8):
    plane, x = _case(9, 64, 64, 2)
    b, _src = _bind(w8, plane)
    xd = to_dev(x)
    y = torch.zeros((2, 64), dtype=torch.int16, device=dev())
    for fn in (w8.w8_gemv, w8.bf16_gemv):
        with pytest.raises(w8.W8Error) as e:
            fn(b, 0, xd, y)
        assert e.value.name == "W8_ERR_DTYPE"
    big = torch.zeros((65, 64), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.mxfp4_gemv(b, 0, big, torch.zeros((65, 64), dtype=torch.int16, device=dev()))
    assert e.value.name == "W8_ERR_SHAPE"
    with pytest.raises(w8.W8Error) as e:
        b.plan(0, 65)
    assert e.value.name == "W8_ERR_SHAPE"
    fp8, _x = synth.weight_plane(np.random.default_rng(1), 64, 64), None
    b8 = w8.bind([w8.Plane.from_tensor(to_dev(fp8.w), to_dev(fp8.scale))])
    with pytest.raises(w8.W8Error) as e:
        w8.mxfp4_gemv(b8, 0, xd, y)
    assert e.value.name == "W8_ERR_DTYPE"
    torch.cuda.synchronize()
    assert torch.all(y == 0)
