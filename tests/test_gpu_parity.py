"""GPU parity of the w8a16 / bf16 GEMV against the CPU oracle, through the C ABI.

What is checked (ATOM PR #2980, Testing: the PR compares its kernels with the
dequantized product, bit-identical for token counts 1, 5 and 16, and checks that
every finite E4M3 code is read without error; its served outputs are held to
the fp32 rounding bound against an fp64 recomputation):

* random seeded inputs, many shapes with ragged N and K tails and every
  token-count regime, within |y - y64| <= 2^-7 |y64| + 2^-12 sum|scale W x|
  of the oracle's fp64 recompute;
* exact-sum inputs (every order of summation exact): bit for bit equal to the
  oracle's fp32 ascending-k result, including split-K plans;
* one-hot activations over all 254 finite codes: y = bf16(scale * W[n,k]);
* unit scales: the FP8 path equals the bf16 path on the widened plane bit
  for bit, at every size (same summation order by construction);
* power-of-two scales commute; NaN codes poison exactly their row;
* the repack places every element where the documented address map says;
* padded planes, strided / misaligned activations, strided outputs, m = 0,
  workspace reuse, CUDA-graph replay and the error returns of the gemv calls;
* every full-size workload (the shapes the bench times, with the same plans)
  on sampled rows that the oracle computes one by one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_weight_only_w8a16_gb300 import synth, workloads

from .gpu_util import bind_plane, dev, from_dev, run_gemv, to_dev

pytestmark = pytest.mark.gpu

DT8, DT16 = oracle.DT_E4M3FN, oracle.DT_BF16


@pytest.fixture(scope="module")
def w8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_weight_only_w8a16_gb300 import w8 as lib

    return lib


def _case(seed, n, k, m, dtype="e4m3fn", ldw=None):
    """A seeded plane whose rows are padded to 16 bytes (bind refuses unpadded
    planes) and m tokens."""
    if ldw is None:
        step = 16 if dtype == "e4m3fn" else 8
        ldw = -(-k // step) * step
    rng = np.random.default_rng(seed)
    plane = synth.weight_plane(rng, n, k, dtype, ldw)
    x = synth.activations(rng, k, m)
    return plane, x


def _oracle_dt(plane):
    return DT8 if plane.dtype == "e4m3fn" else DT16


def _check_tol(plane, x, y, rows=None):
    w = plane.w if rows is None else np.ascontiguousarray(plane.w[rows])
    sc = plane.scale if (rows is None or plane.scale is None) else plane.scale[rows]
    y64, mag = oracle.gemv_f64(w, _oracle_dt(plane), sc, x, k=plane.k, threads=8)
    yy = y if rows is None else y[:, rows]
    ok, worst = oracle.within_tolerance(yy, y64, mag)
    assert ok, f"outside tolerance: worst ratio {worst:.3g}"
    return worst


# ---------------------------------------------------------------------------
# layout
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["e4m3fn", "bf16"])
@pytest.mark.parametrize("n,k,ldw", [(37, 77, 80), (16, 32, 32), (100, 300, 320), (5, 1, 16)])
def test_repack_matches_host_address_map(w8, dtype, n, k, ldw):
    plane, _ = _case(1, n, k, 1, dtype, ldw)
    b, _src = bind_plane(w8, plane)
    info = b.info(0)
    elt = 1 if dtype == "e4m3fn" else 2
    assert info.layout == w8.LAYOUT_MMA_16x32
    assert info.row_tiles == -(-n // 16) and info.k_blocks == -(-k // 32)
    nbytes = info.packed_bytes
    base = info.packed - b.dst.data_ptr()
    packed = b.dst[base: base + nbytes].cpu().numpy()
    rt, kb = info.row_tiles, info.k_blocks
    want = np.zeros(nbytes, dtype=np.uint8)
    src = plane.w.view(np.uint8).reshape(n, ldw * elt)
    for r in range(rt * 16):
        for c in range(kb * 32):
            o = w8.packed_offset(w8.DT_E4M3FN if elt == 1 else w8.DT_BF16, kb, r, c)
            if r < n and c < k:
                want[o: o + elt] = src[r, c * elt: c * elt + elt]
    assert np.array_equal(packed, want)
    if dtype == "e4m3fn":
        sbase = info.scale - b.dst.data_ptr()
        sc = b.dst[sbase: sbase + 4 * rt * 16].cpu().numpy().view(np.float32)
        assert np.array_equal(sc[:n], plane.scale) and np.all(sc[n:] == 0)


# ---------------------------------------------------------------------------
# random inputs within tolerance
# ---------------------------------------------------------------------------

# (6200, 700) has 49 row blocks of 128: from 17 tokens on, the tensor-memory kernel
SHAPES = [(256, 512), (100, 200), (37, 77), (1, 1), (16, 32), (513, 1000), (130, 2100),
          (48, 4096), (2624, 640), (6200, 700)]
MS = [1, 2, 3, 5, 8, 9, 16, 17, 31, 33, 64]


@pytest.mark.parametrize("dtype", ["e4m3fn", "bf16"])
@pytest.mark.parametrize("n,k", SHAPES)
def test_random_inputs_within_tolerance(w8, dtype, n, k):
    plane, x_all = _case(hash((n, k)) & 0xFFFF, n, k, 64, dtype)
    b, _src = bind_plane(w8, plane)
    ws = b.new_workspace()
    for m in MS:
        x = np.ascontiguousarray(x_all[:m])
        y = run_gemv(w8, b, 0, x, n, ws=ws, fp8=(dtype == "e4m3fn"))
        _check_tol(plane, x, y)


# ---------------------------------------------------------------------------
# bit-exact cases
# ---------------------------------------------------------------------------

def _exact_sum_case(rng, n, k, m, e_lo=5, e_hi=10):
    e = rng.integers(e_lo, e_hi, (n, k))
    codes = ((rng.integers(0, 2, (n, k)) << 7) | (e << 3) | rng.integers(0, 8, (n, k)))
    codes = codes.astype(np.uint8)
    scale = (2.0 ** rng.integers(-6, 3, n)).astype(np.float32)
    x = synth.to_bf16_bits(rng.integers(-8, 9, (m, k)).astype(np.float32))
    return synth.Plane("e4m3fn", n, k, k, codes, scale), x


@pytest.mark.parametrize("n,k", [(16, 32), (64, 2048), (300, 700), (2624, 256), (40, 6144),
                                 (6144, 256)])
@pytest.mark.parametrize("m", [1, 5, 16, 33, 64])
def test_exact_sum_inputs_bit_exact(w8, n, k, m):
    rng = np.random.default_rng(n * 7 + k + m)
    plane, x = _exact_sum_case(rng, n, k, m)
    b, _src = bind_plane(w8, plane)
    y = run_gemv(w8, b, 0, x, n)
    want = oracle.gemv(plane.w, DT8, plane.scale, x)
    assert oracle.same_values(y, want)


def test_one_hot_reads_all_254_codes(w8):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)] + [0, 0x80], np.uint8)
    w = codes.reshape(16, 16)
    rng = np.random.default_rng(31)
    scale = rng.uniform(0.001, 3.0, 16).astype(np.float32)
    x = np.zeros((16, 16), np.uint16)
    x[np.arange(16), np.arange(16)] = 0x3F80
    b, _src = bind_plane(w8, synth.Plane("e4m3fn", 16, 16, 16, w, scale))
    y = run_gemv(w8, b, 0, x, 16)
    assert oracle.same_values(y, oracle.gemv(w, DT8, scale, x))


def test_one_hot_codes_across_tiles_and_blocks(w8):
    """All 254 codes spread over several row tiles and K blocks; each token
    picks one column, so y[m, n] is the scaled code at (n, k_m)."""
    rng = np.random.default_rng(32)
    n, k, m = 70, 200, 64
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    w = rng.choice(finite, (n, k))
    w.flat[:254] = finite
    scale = rng.uniform(0.01, 2.0, n).astype(np.float32)
    cols = rng.choice(k, m, replace=False)
    cols[:4] = [0, 31, 32, k - 1]
    x = np.zeros((m, k), np.uint16)
    x[np.arange(m), cols] = 0x3F80
    b, _src = bind_plane(w8, synth.Plane("e4m3fn", n, k, k, w, scale))
    y = run_gemv(w8, b, 0, x, n)
    assert oracle.same_values(y, oracle.gemv(w, DT8, scale, x))


def _widened_bf16_plane(plane):
    """The bf16 plane holding exactly the widened codes (through torch)."""
    t = torch.from_numpy(np.ascontiguousarray(plane.w[:, :plane.k]))
    wb = t.view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return synth.Plane("bf16", plane.n, plane.k, plane.k, np.ascontiguousarray(wb), None)


@pytest.mark.parametrize("n,k", [(256, 512), (2624, 6144), (333, 16384), (6144, 2048)])
@pytest.mark.parametrize("m", [1, 4, 8, 16, 32, 64])
def test_unit_scale_fp8_equals_bf16_path(w8, n, k, m):
    plane, x_all = _case(n + k, n, k, m)
    plane.scale = np.ones(n, np.float32)
    x = np.ascontiguousarray(x_all[:m])
    b8, _s8 = bind_plane(w8, plane)
    b16, _s16 = bind_plane(w8, _widened_bf16_plane(plane))
    y8 = run_gemv(w8, b8, 0, x, n, fp8=True)
    y16 = run_gemv(w8, b16, 0, x, n, fp8=False)
    assert np.array_equal(y8, y16)


@pytest.mark.parametrize("n,k,m", [(6144, 8192, 64), (16384, 512, 50)])
def test_unit_scale_fp8_equals_bf16_path_one_cta_per_sm(w8, n, k, m):
    """The one-CTA-per-SM tensor-memory instance (49..64 tokens) of both
    weight formats: an FP8 plane with unit scales gives the bits of the bf16
    plane of its decoded values, and the bf16 path is within tolerance."""
    plane, x_all = _case(n + k + m, n, k, m)
    plane.scale = np.ones(n, np.float32)
    x = np.ascontiguousarray(x_all[:m])
    b8, _s8 = bind_plane(w8, plane)
    wide = _widened_bf16_plane(plane)
    b16, _s16 = bind_plane(w8, wide)
    if torch.cuda.get_device_properties(dev()).multi_processor_count == 152:
        assert b8.plan(0, m).ctas_per_sm == 1 and b16.plan(0, m).ctas_per_sm == 1
    w8.device_status(reset=True)
    y8 = run_gemv(w8, b8, 0, x, n, fp8=True)
    y16 = run_gemv(w8, b16, 0, x, n, fp8=False)
    assert np.array_equal(y8, y16)
    _check_tol(wide, x, y16)
    assert w8.device_status() == 0


@pytest.mark.parametrize("j", [-4, 5])
@pytest.mark.parametrize("n,k,m", [(300, 3000, 8), (6144, 1000, 40)])
def test_power_of_two_scale_commutes(w8, j, n, k, m):
    plane, x_all = _case(77, n, k, m)
    x = np.ascontiguousarray(x_all[:m])
    b1, _s1 = bind_plane(w8, plane)
    y1 = run_gemv(w8, b1, 0, x, n)
    plane2 = synth.Plane("e4m3fn", n, k, plane.ldw, plane.w,
                         (plane.scale * np.float32(2.0 ** j)).astype(np.float32))
    b2, _s2 = bind_plane(w8, plane2)
    y2 = run_gemv(w8, b2, 0, x, n)
    assert np.array_equal(oracle.bf16_bits_to_f64(y2), oracle.bf16_bits_to_f64(y1) * 2.0 ** j)


@pytest.mark.parametrize("n,k,m", [(50, 500, 4), (6144, 500, 20)])
def test_nan_code_poisons_its_row(w8, n, k, m):
    plane, x_all = _case(78, n, k, m)
    plane.w[7, 123] = 0x7F
    plane.w[40, 499] = 0xFF
    x = np.ascontiguousarray(x_all[:m])
    b, _src = bind_plane(w8, plane)
    y = run_gemv(w8, b, 0, x, n)
    v = oracle.bf16_bits_to_f64(y)
    assert np.all(np.isnan(v[:, [7, 40]]))
    assert not np.any(np.isnan(np.delete(v, [7, 40], axis=1)))
    _check_tol(plane, x, y)


# ---------------------------------------------------------------------------
# strides, padding, edge cases
# ---------------------------------------------------------------------------

def test_padded_row_stride_equals_dense_plane(w8):
    """The K-padding workload: W [4096, 6144 + 128 pad] with zero pad columns
    gives exactly the dense [4096, 6144] result."""
    plane, x_all = _case(40, 4096, 6144, 8, ldw=6144 + 128)
    x = np.ascontiguousarray(x_all[:8])
    b_pad, _s1 = bind_plane(w8, plane)
    dense = synth.Plane("e4m3fn", 4096, 6144, 6144, np.ascontiguousarray(plane.w[:, :6144]),
                        plane.scale)
    b_dense, _s2 = bind_plane(w8, dense)
    y_pad = run_gemv(w8, b_pad, 0, x, 4096)
    y_dense = run_gemv(w8, b_dense, 0, x, 4096)
    assert np.array_equal(y_pad, y_dense)
    # the pad columns read as part of K (zero codes, finite activations) add
    # exact zeros; the plan differs (more K blocks), so compare within tolerance
    kpad = synth.Plane("e4m3fn", 4096, 6272, 6272, plane.w, plane.scale)
    b_k, _s3 = bind_plane(w8, kpad)
    xk = np.ascontiguousarray(synth.activations(np.random.default_rng(9), 6272, 8))
    xk[:, :6144] = x
    y_k = run_gemv(w8, b_k, 0, xk, 4096)
    _check_tol(dense, x, y_k)


def test_strided_and_misaligned_activations(w8):
    plane, x_all = _case(41, 200, 1000, 9)
    x = np.ascontiguousarray(x_all[:9])
    b, _src = bind_plane(w8, plane)
    ws = b.new_workspace()
    y_ref = run_gemv(w8, b, 0, x, 200, ws=ws)
    # a wider row stride (ldx = K + 24, still a multiple of 8)
    big = torch.zeros((9, 1024), dtype=torch.int16, device=dev())
    big[:, :1000] = to_dev(x)
    y1 = run_gemv(w8, b, 0, x, 200, ws=ws, x_dev=big[:, :1000])
    assert np.array_equal(y1, y_ref)
    # rows that are not 16-byte aligned are refused before any launch
    odd = torch.zeros((9, 1003), dtype=torch.int16, device=dev())
    flat = torch.zeros(9 * 1000 + 8, dtype=torch.int16, device=dev())
    yd = torch.zeros((9, 200), dtype=torch.int16, device=dev())
    for xd in (odd[:, :1000], flat[1:9001].view(9, 1000)):
        with pytest.raises(w8.W8Error) as e:
            w8.w8_gemv(b, 0, xd, yd, ws)
        assert e.value.name == "W8_ERR_ALIGN"
    torch.cuda.synchronize()
    assert torch.all(yd == 0)


def test_strided_output_leaves_gap_untouched(w8):
    plane, x_all = _case(42, 100, 256, 3)
    x = np.ascontiguousarray(x_all[:3])
    b, _src = bind_plane(w8, plane)
    y = torch.full((3, 130), 0x1234, dtype=torch.int16, device=dev())
    w8.w8_gemv(b, 0, to_dev(x), y, b.new_workspace())
    torch.cuda.synchronize()
    yy = from_dev(y)
    assert np.all(yy[:, 100:] == 0x1234)
    _check_tol(plane, x, np.ascontiguousarray(yy[:, :100]))


def test_zero_tokens_is_a_no_op(w8):
    plane, _ = _case(43, 64, 64, 1)
    b, _src = bind_plane(w8, plane)
    y = torch.full((1, 64), 7, dtype=torch.int16, device=dev())
    x = torch.zeros((1, 64), dtype=torch.int16, device=dev())
    w8.w8_gemv(b, 0, x, y, None, m=0)
    torch.cuda.synchronize()
    assert torch.all(y == 7)


def test_workspace_reuse_graph_replay_and_errors(w8):
    # m = 8: the register-ring kernel, whose split-K plans use the workspace
    plane, x_all = _case(44, 128, 6144, 8)
    x = np.ascontiguousarray(x_all[:8])
    b, _src = bind_plane(w8, plane)
    assert b.plan(0, 8).kernel == 0 and b.plan(0, 8).splits > 1
    ws = b.new_workspace(0, 8)
    y1 = run_gemv(w8, b, 0, x, 128, ws=ws)
    y2 = run_gemv(w8, b, 0, x, 128, ws=ws)
    assert np.array_equal(y1, y2)
    _check_tol(plane, x, y1)
    # CUDA-graph capture and replay of the same call
    xd = to_dev(x)
    yd = torch.zeros((8, 128), dtype=torch.int16, device=dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w8.w8_gemv(b, 0, xd, yd, ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w8.w8_gemv(b, 0, xd, yd, ws)
    yd.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(yd), y1)
    # error returns
    yd2 = torch.zeros((8, 128), dtype=torch.int16, device=dev())
    for kw, name in [(dict(workspace=None), "W8_ERR_NULL"),
                     (dict(workspace=ws[:256]), "W8_ERR_CAPACITY"),
                     (dict(workspace=ws[8:]), "W8_ERR_ALIGN")]:
        with pytest.raises(w8.W8Error) as e:
            w8.w8_gemv(b, 0, xd, yd2, **kw)
        assert e.value.name == name
    with pytest.raises(w8.W8Error) as e:
        w8.bf16_gemv(b, 0, xd, yd2, ws)
    assert e.value.name == "W8_ERR_DTYPE"
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv(b, 1, xd, yd2, ws)
    assert e.value.name == "W8_ERR_PLANE"
    big = torch.zeros((257, 6144), dtype=torch.int16, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.w8_gemv(b, 0, big, torch.zeros((257, 128), dtype=torch.int16, device=dev()), ws)
    assert e.value.name == "W8_ERR_SHAPE"
    with pytest.raises(w8.W8Error) as e:   # output row stride shorter than N
        w8.w8_gemv(b, 0, xd, torch.zeros((8, 100), dtype=torch.int16, device=dev()), ws)
    assert e.value.name == "W8_ERR_SHAPE"
    torch.cuda.synchronize()
    assert torch.all(yd2 == 0)  # no refused call wrote anything


@pytest.mark.parametrize("n,k,m,kind", [(6144, 2048, 32, "cluster"), (6200, 1000, 17, "cluster"),
                                        (7000, 512, 64, "cluster"), (28672, 512, 64, "cluster"),
                                        (6144, 1000, 64, "cluster"),
                                        (6144, 8192, 48, "ws"), (6144, 8192, 33, "ws"),
                                        (6160, 8192, 20, "ws"),
                                        (6144, 8192, 64, "deep_ws"), (6160, 8192, 57, "deep_ws"),
                                        (16384, 512, 50, "deep")])
def test_tensor_memory_kernel_clusters_and_graph_replay(w8, n, k, m, kind):
    """Planes of >= 48 row blocks with >= 17 tokens run the tensor-memory
    kernel; with split K its CTAs form a cluster (up to 8 splits) and add
    their partial tiles on chip (28672 rows: no split), or, on planes of few
    row blocks and long K (48-49 row blocks x 8192: 6 splits), add them
    through the workspace (a ragged last row block included).  At 49..64
    tokens, where one wave of unclustered CTAs covers 3/4 of the SMs, the
    instance with one CTA per SM and the deeper ring runs (48-49 row blocks
    x 3 K ranges through the workspace; 128 row blocks with no split).
    Repeated calls and a CUDA-graph replay give identical bits, within
    tolerance, and every bounded wait of the kernel ended normally (device
    status 0)."""
    plane, x_all = _case(45, n, k, m)
    x = np.ascontiguousarray(x_all[:m])
    b, _src = bind_plane(w8, plane)
    p = b.plan(0, m)
    assert p.kernel == 1
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    if kind == "ws":
        assert p.cluster == 1 and p.splits == 6 and p.workspace_bytes > 0
    elif kind == "cluster":
        assert p.cluster == p.splits and p.workspace_bytes == 0 and p.ctas_per_sm == 2
    elif sms == 152:  # the deep instance: its choice depends on the SM count
        assert p.ctas_per_sm == 1 and p.cluster == 1 and p.smem_bytes > 150 * 1024
        assert p.splits == (3 if kind == "deep_ws" else 1)
        assert (p.workspace_bytes > 0) == (kind == "deep_ws")
    ws = b.new_workspace()
    w8.device_status(reset=True)
    y1 = run_gemv(w8, b, 0, x, n)
    y2 = run_gemv(w8, b, 0, x, n)
    assert np.array_equal(y1, y2)
    _check_tol(plane, x, y1)
    xd = to_dev(x)
    yd = torch.zeros((m, n), dtype=torch.int16, device=dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w8.w8_gemv(b, 0, xd, yd, ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w8.w8_gemv(b, 0, xd, yd, ws)
    yd.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(yd), y1)
    assert w8.device_status() == 0


def test_plan_info_of_a_bf16_tensor_memory_plan(w8):
    # a bf16 build's plan reports the bf16 ring depth: for the tensor-memory
    # kernel its weight stages (2 of 4 blocks at 17..32 tokens), not an entry
    # of the register-ring instance table
    plane, _x = _case(9, 6144, 256, 1, "bf16")
    b, _src = bind_plane(w8, plane)
    p = b.plan(0, 32)
    assert p.kernel == 1 and p.n_tiles == 4
    assert p.depth == 2 * 4
    assert b.plan(0, 8).kernel == 0


def test_bind_refusals_on_device(w8):
    n, k = 32, 64
    codes = to_dev(np.zeros((n, k), np.uint8))
    sc = to_dev(np.ones(n, np.float32))
    bf = torch.zeros((n, k), dtype=torch.bfloat16, device=dev())
    cases = [
        ([w8.Plane.from_tensor(codes.view(torch.float8_e4m3fnuz), sc)], "W8_ERR_DTYPE"),
        ([w8.Plane.from_tensor(codes.view(torch.float8_e5m2), sc)], "W8_ERR_DTYPE"),
        ([w8.Plane.from_tensor(bf.view(torch.float16))], "W8_ERR_DTYPE"),
        ([w8.Plane.from_tensor(codes, sc), w8.Plane.from_tensor(bf)], "W8_ERR_MIXED"),
        ([w8.Plane.from_tensor(codes)], "W8_ERR_SCALE"),
        ([w8.Plane.from_tensor(bf, sc)], "W8_ERR_SCALE"),
        ([w8.Plane.from_tensor(codes[:, 1:], sc[:n])], "W8_ERR_UNPADDED"),
    ]
    p_bias = w8.Plane.from_tensor(codes, sc)
    p_bias.bias = sc
    cases.append(([p_bias], "W8_ERR_BIAS"))
    for planes, name in cases:
        with pytest.raises(w8.W8Error) as e:
            w8.bind(planes)
        assert e.value.name == name
    # too small / misaligned packed buffer
    good = [w8.Plane.from_tensor(codes, sc)]
    need = w8.packed_bytes(good)
    with pytest.raises(w8.W8Error) as e:
        w8.bind(good, torch.empty(need - 256, dtype=torch.uint8, device=dev()))
    assert e.value.name == "W8_ERR_CAPACITY"
    buf = torch.empty(need + 512, dtype=torch.uint8, device=dev())
    with pytest.raises(w8.W8Error) as e:
        w8.bind(good, buf[16:])
    assert e.value.name == "W8_ERR_ALIGN"


def test_multi_plane_build(w8):
    """gate+up then down of the shared expert in one build."""
    rng = np.random.default_rng(45)
    gu = synth.weight_plane(rng, 4096, 6144)
    dn = synth.weight_plane(rng, 6144, 2048)
    x1 = synth.activations(rng, 6144, 8)
    x2 = synth.activations(rng, 2048, 8)
    srcs = [(to_dev(p.w), to_dev(p.scale)) for p in (gu, dn)]
    b = w8.bind([w8.Plane.from_tensor(w, s) for w, s in srcs])
    assert b.n_planes == 2
    ws = b.new_workspace()
    y1 = run_gemv(w8, b, 0, x1, 4096, ws=ws)
    y2 = run_gemv(w8, b, 1, x2, 6144, ws=ws)
    rows = np.arange(0, 4096, 37)
    _check_tol(gu, x1, y1, rows)
    _check_tol(dn, x2, y2, np.arange(0, 6144, 41))


# ---------------------------------------------------------------------------
# full-size workloads, sampled rows
# ---------------------------------------------------------------------------

# (gate_up planes with SiLU-and-multiply: tests/test_gpu_gate_up.py; MXFP4
# planes: tests/test_gpu_mxfp4.py; block-scaled FP8 planes: tests/test_gpu_b128.py)
FULL = [p for p in workloads.ALL
        if p.name != "lm_head" and not p.act and p.dtype in ("e4m3fn", "bf16")]


@pytest.mark.parametrize("proj", FULL, ids=[p.name for p in FULL])
def test_full_size_workloads_sampled(w8, proj):
    plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0, ldw=proj.ldw)
    b, _src = bind_plane(w8, plane)
    ws = b.new_workspace()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(proj.n, min(proj.n, 96), replace=False),
                                     [0, proj.n - 1]]))
    for m in proj.ms:
        x = np.ascontiguousarray(x_all[:m])
        y = run_gemv(w8, b, 0, x, proj.n, ws=ws, fp8=(proj.dtype == "e4m3fn"))
        assert not np.any(np.isnan(oracle.bf16_bits_to_f64(y)))
        _check_tol(plane, x, y, rows)


def test_lm_head_full_size_sampled(w8):
    proj = workloads.LM_HEAD
    plane, x_all = synth.workload(proj.n, proj.k, proj.dtype, seed=0)
    b, _src = bind_plane(w8, plane)
    del _src
    x = np.ascontiguousarray(x_all[:1])
    y = run_gemv(w8, b, 0, x, proj.n, fp8=False)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(proj.n, 128, replace=False), [0, proj.n - 1]]))
    _check_tol(plane, x, y, rows)


# ---------------------------------------------------------------------------
# 65..256 tokens: draft rows and prefill chunks, tensor-memory kernel only
# ---------------------------------------------------------------------------

LARGE_M = [(300, 700, 100), (100, 64, 200), (256, 512, 65), (6144, 2048, 128),
           (6144, 1000, 192), (2624, 6144, 256), (28672, 512, 256), (6144, 4096, 96)]


@pytest.mark.parametrize("dtype", ["e4m3fn", "bf16"])
@pytest.mark.parametrize("n,k,m", LARGE_M)
def test_large_token_counts_within_tolerance(w8, dtype, n, k, m):
    """Above 64 tokens every call runs the tensor-memory kernel with the
    tokens padded to 96, 128, 192 or 256 (one CTA per SM, 512 TMEM columns),
    split K in clusters (the workspace splits serve 17..64 tokens only);
    ragged N, K and token counts; sampled rows on the large planes."""
    plane, x = _case(n + k + m, n, k, m, dtype)
    b, _src = bind_plane(w8, plane)
    p = b.plan(0, m)
    assert p.kernel == 1 and p.workspace_bytes == 0 and p.cluster == p.splits
    w8.device_status(reset=True)
    y = run_gemv(w8, b, 0, x, n, fp8=(dtype == "e4m3fn"))
    rows = None
    if n >= 2000:
        rng = np.random.default_rng(5)
        rows = np.unique(np.concatenate([rng.choice(n, 96, replace=False), [0, 127, 128, n - 1]]))
    _check_tol(plane, x, y, rows)
    assert w8.device_status() == 0


@pytest.mark.parametrize("n,k,m", [(6144, 256, 128), (6144, 256, 256), (300, 700, 97),
                                   (2624, 512, 200)])
def test_large_token_counts_exact_sums_bit_exact(w8, n, k, m):
    rng = np.random.default_rng(n * 3 + k + m)
    plane, x = _exact_sum_case(rng, n, k, m)
    b, _src = bind_plane(w8, plane)
    y = run_gemv(w8, b, 0, x, n)
    assert oracle.same_values(y, oracle.gemv(plane.w, DT8, plane.scale, x))


@pytest.mark.parametrize("m", [128, 256])
def test_large_token_counts_unit_scale_fp8_equals_bf16(w8, m):
    plane, x = _case(77, 6144, 2048, m)
    unit = synth.Plane("e4m3fn", plane.n, plane.k, plane.ldw, plane.w,
                       np.ones(plane.n, dtype=np.float32))
    wide = _widened_bf16_plane(unit)
    b8, _s8 = bind_plane(w8, unit)
    b16, _s16 = bind_plane(w8, wide)
    y8 = run_gemv(w8, b8, 0, x, plane.n)
    y16 = run_gemv(w8, b16, 0, x, plane.n, fp8=False)
    assert oracle.same_values(y8, y16)


def test_large_token_counts_graph_replay(w8):
    n, k, m = 6144, 1024, 256
    plane, x = _case(91, n, k, m)
    b, _src = bind_plane(w8, plane)
    ws = b.new_workspace()
    w8.device_status(reset=True)
    y1 = run_gemv(w8, b, 0, x, n)
    xd = to_dev(x)
    yd = torch.zeros((m, n), dtype=torch.int16, device=dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w8.w8_gemv(b, 0, xd, yd, ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w8.w8_gemv(b, 0, xd, yd, ws)
    yd.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(yd), y1)
    assert w8.device_status() == 0


def test_one_workspace_across_planes_of_a_build(w8):
    """Split-K calls on planes of different sizes in one build share one
    workspace, back to back.  The counter head sits in the same place for
    every call of the build, so one call's partial sums never land on another
    call's arrival counters: here the second plane (1040 rows, 65 row groups
    at one token) counts past the 64 counters that fill the first 256 bytes,
    where the first plane's partial sums would otherwise start."""
    rng = np.random.default_rng(92)
    shapes = [(128, 6144), (1040, 2048)]
    planes = [synth.weight_plane(rng, n, k) for n, k in shapes]
    b = w8.bind([w8.Plane.from_tensor(to_dev(p.w), to_dev(p.scale)) for p in planes])
    ws = b.new_workspace()
    calls = [(0, 8), (1, 1), (0, 24), (1, 1), (1, 8), (0, 1)]
    p1 = b.plan(1, 1)
    assert p1.kernel == 0 and p1.splits > 1 and p1.row_groups > 64
    assert all(b.plan(i, m).splits > 1 for i, m in calls)
    xs = {k: synth.activations(rng, k, 24) for k in (2048, 6144)}
    outs = []
    for i, m in calls:
        n, k = shapes[i]
        outs.append(run_gemv(w8, b, i, np.ascontiguousarray(xs[k][:m]), n, ws=ws))
    for (i, m), y in zip(calls, outs):
        n, k = shapes[i]
        own, _src = bind_plane(w8, planes[i])
        x = np.ascontiguousarray(xs[k][:m])
        assert np.array_equal(y, run_gemv(w8, own, 0, x, n))
        _check_tol(planes[i], x, y)
