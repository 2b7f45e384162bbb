"""GPU parity of the merged gate_up projection and its fused SiLU-and-multiply.

A gate_up plane is the MLP's merged [2I, K] projection: rows 0..I-1 gate,
I..2I-1 up (ATOM Model Support Guide: Llama MLP, merged gate+up then
SiLU+mul then down; gate_proj is shard 0, up_proj shard 1).  Bound with
W8_SRC_GATE_UP, its packed tiles interleave gate and up rows, and

* w8_gemv / bf16_gemv on it give the plain GEMV in source row order, bit for
  bit what the same plane bound row-major gives (every row is reduced in the
  same order wherever its tile sits) and within the GEMV tolerance of the
  oracle;
* w8_gemv_silu_mul gives h = bf16(silu(g) * u) from the bf16 outputs g, u:
  within the propagated tolerance of the oracle's fp64 recompute on random
  inputs (register-ring and tensor-memory kernels, with and without split K,
  both dtypes); on exact-sum inputs equal to the oracle's one-rounding result
  except where the exact value lies within fp32 evaluation error of a bf16
  rounding midpoint; over all 254 finite gate codes and the special values
  (inf, -inf, NaN, very negative g) as the definition gives;
* the full-size shared expert (gate_up [4096, 6144] at 8 tokens) and the
  dense MLP's gate_up ([24576, 6144], GLM-5.2 anatomy page, layers 0-2) on
  sampled gate rows;
* the refusals: SiLU-and-multiply on a row-major plane, an output stride
  below I, a gate_up plane whose I is not a multiple of 8.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_weight_only_w8a16_gb300 import synth

from .gpu_util import dev, from_dev, padded, to_dev

pytestmark = pytest.mark.gpu

DT8, DT16 = oracle.DT_E4M3FN, oracle.DT_BF16


@pytest.fixture(scope="module")
def w8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_weight_only_w8a16_gb300 import w8 as lib

    return lib


def _bind(w8, plane: synth.Plane, gated: bool):
    plane = padded(plane)
    w_d = to_dev(plane.w)
    s_d = to_dev(plane.scale) if plane.scale is not None else None
    p = w8.Plane.from_tensor(w_d, s_d, k=plane.k,
                             dtype=w8.DT_E4M3FN if plane.dtype == "e4m3fn" else w8.DT_BF16,
                             layout=w8.SRC_GATE_UP if gated else w8.SRC_ROW_MAJOR)
    return w8.bind([p]), (w_d, s_d)


def _x_dev(x: np.ndarray) -> torch.Tensor:
    m, k = x.shape
    ldx = -(-k // 8) * 8
    xp = torch.zeros((m, ldx), dtype=torch.int16, device=dev())
    xp[:, :k] = to_dev(x)
    return xp[:, :k]


def _call(w8, fn, b, x: np.ndarray, cols: int, ws=None):
    xd = _x_dev(x)
    y = torch.full((x.shape[0], cols), 0x7FC1, dtype=torch.int16, device=dev())
    fn(b, 0, xd, y, b.new_workspace() if ws is None else ws)
    torch.cuda.synchronize()
    return from_dev(y)


def _plain_fn(w8, plane):
    return w8.w8_gemv if plane.dtype == "e4m3fn" else w8.bf16_gemv


def _case(seed, n, k, m, dtype="e4m3fn"):
    rng = np.random.default_rng(seed)
    return synth.weight_plane(rng, n, k, dtype), synth.activations(rng, k, m)


# (2I, K, m): register-ring plans with and without split K, tensor-memory
# plans (m >= 17 on >= 48 blocks of 128 rows) with and without a cluster, and
# one whose K splits meet in the workspace (6144 x 8192 at 24 tokens)
GATED_SHAPES = [(16, 32, 1), (64, 96, 3), (160, 1000, 8), (32, 6144, 5), (4096, 6144, 8),
                (512, 3000, 16), (6144, 1024, 32), (6144, 2048, 20), (7168, 512, 64),
                (512, 700, 100), (7168, 512, 256), (6144, 8192, 24)]


@pytest.mark.parametrize("dtype", ["e4m3fn", "bf16"])
@pytest.mark.parametrize("n,k,m", GATED_SHAPES)
def test_gate_up_plain_gemv_keeps_source_order(w8, dtype, n, k, m):
    plane, x = _case(n + 3 * k + m, n, k, m, dtype)
    bg, _sg = _bind(w8, plane, gated=True)
    br, _sr = _bind(w8, plane, gated=False)
    assert bg.info(0).layout == w8.LAYOUT_MMA_16x32_GATE_UP
    assert br.info(0).layout == w8.LAYOUT_MMA_16x32
    fn = _plain_fn(w8, plane)
    yg = _call(w8, fn, bg, x, n)
    yr = _call(w8, fn, br, x, n)
    assert oracle.same_values(yg, yr)
    y64, mag = oracle.gemv_f64(plane.w, DT8 if dtype == "e4m3fn" else DT16, plane.scale, x,
                               k=k, threads=8)
    ok, worst = oracle.within_tolerance(yg, y64, mag)
    assert ok, worst


@pytest.mark.parametrize("dtype", ["e4m3fn", "bf16"])
@pytest.mark.parametrize("n,k,m", GATED_SHAPES)
def test_silu_mul_within_propagated_tolerance(w8, dtype, n, k, m):
    plane, x = _case(7 * n + k + m, n, k, m, dtype)
    b, _src = _bind(w8, plane, gated=True)
    half = n // 2
    h = _call(w8, w8.w8_gemv_silu_mul, b, x, half + 3)  # 3 columns past I stay untouched
    assert np.all(h[:, half:] == 0x7FC1)
    h = h[:, :half]
    y64, mag = oracle.gemv_f64(plane.w, DT8 if dtype == "e4m3fn" else DT16, plane.scale, x,
                               k=k, threads=8)
    ok, worst = oracle.silu_mul_within_tolerance(h, y64[:, :half], mag[:, :half],
                                                 y64[:, half:], mag[:, half:])
    assert ok, worst
    assert not np.any(np.isnan(oracle.bf16_bits_to_f64(h)))


def _exact_gate_up(rng, n, k, m):
    """Codes of exponents 5..9, power-of-two scales, small integer tokens:
    every partial sum is exact, so g and u are the oracle's bit for bit."""
    e = rng.integers(5, 10, (n, k))
    codes = ((rng.integers(0, 2, (n, k)) << 7) | (e << 3) | rng.integers(0, 8, (n, k)))
    scale = (2.0 ** rng.integers(-9, -4, n)).astype(np.float32)
    x = synth.to_bf16_bits(rng.integers(-8, 9, (m, k)).astype(np.float32))
    return synth.Plane("e4m3fn", n, k, k, codes.astype(np.uint8), scale), x


def _agrees_up_to_midpoints(h_gpu, h_orc, g_bits, u_bits):
    """Bits equal, except (a) where the exact silu(g) u lies within 2^-20
    (relative) of the midpoint between the two results, which must be
    adjacent, and (b) where fp32 exp(-g) overflows (g below about -87) and the
    kernel's SiLU is zero while |silu(g) u| < 2^-120 (|u| + 1)."""
    if oracle.same_values(h_gpu, h_orc):
        return True, 0
    uv = oracle.bf16_bits_to_f64(u_bits)
    big = oracle.silu_mul_f64(oracle.bf16_bits_to_f64(g_bits), uv)
    a, b = oracle.bf16_bits_to_f64(h_gpu), oracle.bf16_bits_to_f64(h_orc)
    diff = ~((a == b) | (np.isnan(a) & np.isnan(b)))
    flips = 0  # case (a); case (b) is not counted
    for i in zip(*np.nonzero(diff)):
        if a[i] == 0 and abs(big[i]) < 2.0 ** -120 * (abs(uv[i]) + 1):
            continue
        mid = (a[i] + b[i]) / 2
        adjacent = abs(int(h_gpu[i]) - int(h_orc[i])) == 1
        if not adjacent or abs(big[i] - mid) > 2.0 ** -20 * abs(big[i]):
            return False, int(diff.sum())
        flips += 1
    return True, flips


@pytest.mark.parametrize("n,k", [(16, 32), (64, 2048), (320, 700), (32, 6144), (6144, 256),
                                 (6144, 2048)])
@pytest.mark.parametrize("m", [1, 5, 16, 33, 64])
def test_silu_mul_exact_sum_inputs(w8, n, k, m):
    rng = np.random.default_rng(n * 5 + k + m)
    plane, x = _exact_gate_up(rng, n, k, m)
    b, _src = _bind(w8, plane, gated=True)
    half = n // 2
    h = _call(w8, w8.w8_gemv_silu_mul, b, x, half)
    y = oracle.gemv(plane.w, DT8, plane.scale, x)
    h_orc = oracle.silu_mul(y[:, :half], y[:, half:])
    ok, flips = _agrees_up_to_midpoints(h, h_orc, y[:, :half], y[:, half:])
    assert ok, "outputs differ beyond a rounding midpoint"
    # a flip needs the exact value within ~2^-21 of a midpoint: rare
    assert flips <= max(2, h.size // 1000)


def test_silu_mul_all_gate_codes_and_special_values(w8):
    """One-hot tokens read one column: g_j = bf16(scale_j * code), u_j likewise.
    The gate column holds all 254 finite codes over 16 scales (g from -inf to
    +inf through very negative values, zeros and subnormals) plus a NaN row."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    half = 512
    k = 32
    rng = np.random.default_rng(41)
    w = rng.integers(0, 0x7E, (2 * half, k)).astype(np.uint8)
    w[:half, 0] = np.resize(codes, half)
    w[half:, 0] = rng.integers(0x30, 0x50, half) | (rng.integers(0, 2, half) << 7).astype(np.uint8)
    scales = np.array([1.0, 1e-3, 0.25, 3.0, 50.0, 3e38, 1e-30, 0.9, 2.0, 7.0, 0.5, 100.0,
                       0.125, 1e-40, 1.5, 0.3], np.float32)
    scale = np.ones(2 * half, np.float32)
    scale[:half] = np.repeat(scales, half // 16)[:half]
    scale[half:] = rng.uniform(0.01, 2.0, half).astype(np.float32)
    w[7, 0] = 0x7F  # a NaN gate
    w[half + 9, 0] = 0xFF  # a NaN up
    x = np.zeros((4, k), np.uint16)
    x[:, 0] = [0x3F80, 0xBF80, 0x4000, 0x3F00]  # 1, -1, 2, 0.5
    plane = synth.Plane("e4m3fn", 2 * half, k, k, w, scale)
    b, _src = _bind(w8, plane, gated=True)
    h = _call(w8, w8.w8_gemv_silu_mul, b, x, half)
    y = oracle.gemv(w, DT8, scale, x)
    g, u = y[:, :half], y[:, half:]
    h_orc = oracle.silu_mul(g, u)
    gv, uv = oracle.bf16_bits_to_f64(g), oracle.bf16_bits_to_f64(u)
    assert np.any(np.isinf(gv)) and np.any(gv < -100) and np.any(np.isnan(gv))
    big = oracle.silu_mul_f64(gv, uv)
    a, want = oracle.bf16_bits_to_f64(h), oracle.bf16_bits_to_f64(h_orc)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(a), nan)
    inf = np.isinf(want)  # g = +-inf, or silu(g) u past the largest bf16
    assert np.any(inf) and np.array_equal(a[inf], want[inf])
    fin = ~(nan | inf)
    # fp32 SiLU: a few fp32 roundings, the final bf16 rounding, and exp
    # overflow for g below about -87 (then |silu(g) u| < 2^-120 (|u| + 1))
    err = np.abs(a[fin] - big[fin])
    assert np.all(err <= (2.0 ** -8 + 2.0 ** -20) * np.abs(big[fin])
                  + 2.0 ** -120 * (np.abs(uv[fin]) + 1.0))
    ok, _nd = _agrees_up_to_midpoints(h, h_orc, g, u)
    assert ok


def test_silu_mul_refusals(w8):
    plane, x = _case(5, 64, 64, 2)
    b_row, _s1 = _bind(w8, plane, gated=False)
    xd = _x_dev(x)
    y = torch.zeros((2, 64), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_silu_mul(b_row, 0, xd, y)
    assert e.value.name == "W8_ERR_LAYOUT"
    b_g, _s2 = _bind(w8, plane, gated=True)
    narrow = torch.zeros((2, 31), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv_silu_mul(b_g, 0, xd, narrow)
    assert e.value.name == "W8_ERR_SHAPE"
    # ldy == I is enough for SiLU-and-multiply, not for the plain GEMV
    exact = torch.zeros((2, 32), dtype=torch.int16, device=dev())
    w8.w8_gemv_silu_mul(b_g, 0, xd, exact)
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv(b_g, 0, xd, exact)
    assert e.value.name == "W8_ERR_SHAPE"
    # m = 0 is a no-op
    w8.w8_gemv_silu_mul(b_g, 0, xd, exact, m=0)
    # I not a multiple of 8
    bad, _x = _case(6, 40, 64, 1)
    with pytest.raises(w8.W8Error) as e:
        _bind(w8, bad, gated=True)
    assert e.value.name == "W8_ERR_SHAPE"
    torch.cuda.synchronize()


@pytest.mark.parametrize("n,k,ms", [(4096, 6144, (8,)), (24576, 6144, (1, 8, 32, 64))],
                         ids=["shared_expert_gate_up", "dense_mlp_gate_up"])
def test_full_size_gate_up_silu_sampled(w8, n, k, ms):
    plane, x_all = synth.workload(n, k, "e4m3fn", seed=0)
    b, _src = _bind(w8, plane, gated=True)
    ws = b.new_workspace()
    half = n // 2
    rng = np.random.default_rng(3)
    j = np.unique(np.concatenate([rng.choice(half, 64, replace=False), [0, 7, 8, half - 1]]))
    rows = np.concatenate([j, half + j])
    sub = synth.Plane("e4m3fn", rows.size, k, k, np.ascontiguousarray(plane.w[rows]),
                      plane.scale[rows])
    for m in ms:
        x = np.ascontiguousarray(x_all[:m])
        h = _call(w8, w8.w8_gemv_silu_mul, b, x, half, ws)
        y64, mag = oracle.gemv_f64(sub.w, DT8, sub.scale, x, k=k, threads=8)
        ok, worst = oracle.silu_mul_within_tolerance(h[:, j], y64[:, :j.size], mag[:, :j.size],
                                                     y64[:, j.size:], mag[:, j.size:])
        assert ok, (m, worst)
    assert w8.device_status() == 0
