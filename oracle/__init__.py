"""CPU oracle for the FP8 weight-only (w8a16) decode GEMV.

TEST INFRASTRUCTURE ONLY: the product path (the C-ABI library and its Python
binding) never imports this package.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.

The arithmetic lives in ``w8_oracle.c`` (plain C, fp32 ascending-k
accumulation, one fp32 scale multiply, one bf16 round to nearest even), which
follows ATOM pull request #2980, sections Summary and
Changes: every E4M3 code has an exact bf16 value, and the fp32 row factor is
applied to the finished row sum, ahead of the one conversion to bf16.  ``brute.py`` is an
independent numpy fp64 recompute used to pin it.  It also holds the MLP
activation that follows a merged gate_up projection (ATOM Model Support
Guide, Model architecture details, Llama MLP): h = silu(g) * u in fp64 with
one bf16 rounding, the w4a16 GEMV on MXFP4 weights (E2M1 elements, E8M0
scales per 32 along K), and the GEMV on block-scaled FP8 planes (one fp32
factor per 128 x 128 block, applied to each block's finished partial sum).

Every function here is pinned by a ``-m "not gpu"`` test
(tests/test_oracle_codecs.py, tests/test_oracle_gemv.py,
tests/test_oracle_silu.py, tests/test_oracle_mxfp4.py,
tests/test_oracle_b128.py).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .build import build_oracle, ORACLE_SO

DT_E4M3FN = 1
DT_BF16 = 2

_default = None
_lock = threading.Lock()


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.c_void_p)


def _declare(lib):
    c_i64 = ctypes.c_int64
    vp = ctypes.c_void_p
    lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_f32.restype = ctypes.c_float
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f32.restype = ctypes.c_float
    lib.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.orc_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
    lib.orc_f32_to_e4m3_sat.restype = ctypes.c_uint8
    lib.orc_quantize_rows.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp]
    lib.orc_quantize_rows.restype = None
    lib.orc_gemv.argtypes = [vp, ctypes.c_int, c_i64, c_i64, c_i64, vp, vp, c_i64, c_i64,
                             vp, c_i64, ctypes.c_int]
    lib.orc_gemv.restype = ctypes.c_int
    lib.orc_gemv_f64.argtypes = [vp, ctypes.c_int, c_i64, c_i64, c_i64, vp, vp, c_i64,
                                 c_i64, vp, vp, ctypes.c_int]
    lib.orc_gemv_f64.restype = ctypes.c_int
    lib.orc_max_threads.argtypes = []
    lib.orc_max_threads.restype = ctypes.c_int
    lib.orc_f64_to_bf16_rne.argtypes = [ctypes.c_double]
    lib.orc_f64_to_bf16_rne.restype = ctypes.c_uint16
    lib.orc_silu_mul_f64.argtypes = [vp, vp, c_i64, vp]
    lib.orc_silu_mul_f64.restype = ctypes.c_int
    lib.orc_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_to_f32.restype = ctypes.c_float
    lib.orc_e8m0_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e8m0_to_f32.restype = ctypes.c_float
    lib.orc_gemv_mxfp4.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp, c_i64, c_i64, vp,
                                   c_i64, ctypes.c_int]
    lib.orc_gemv_mxfp4.restype = ctypes.c_int
    lib.orc_gemv_mxfp4_f64.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp, c_i64, c_i64,
                                       vp, vp, ctypes.c_int]
    lib.orc_gemv_mxfp4_f64.restype = ctypes.c_int
    lib.orc_gemv_e4m3_b128.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp, c_i64, c_i64,
                                       vp, c_i64, ctypes.c_int]
    lib.orc_gemv_e4m3_b128.restype = ctypes.c_int
    lib.orc_gemv_e4m3_b128_f64.argtypes = [vp, c_i64, c_i64, c_i64, vp, c_i64, vp, c_i64,
                                           c_i64, vp, vp, ctypes.c_int]
    lib.orc_gemv_e4m3_b128_f64.restype = ctypes.c_int
    return lib


def _check_plane(w: np.ndarray, dtype: int, k: int | None):
    if dtype == DT_E4M3FN:
        assert w.dtype == np.uint8, "E4M3 planes are uint8 codes"
    elif dtype == DT_BF16:
        assert w.dtype == np.uint16, "bf16 planes are uint16 bit patterns"
    else:
        raise ValueError(f"unknown dtype {dtype}")
    assert w.ndim == 2 and w.strides[1] == w.itemsize
    n, ldw = w.shape[0], w.strides[0] // w.itemsize
    kk = w.shape[1] if k is None else k
    return n, kk, ldw


class Oracle:
    """The oracle's functions bound to one compiled copy of w8_oracle.c."""

    DT_E4M3FN = DT_E4M3FN
    DT_BF16 = DT_BF16

    def __init__(self, lib):
        self.lib = _declare(lib)

    # ---- codecs -------------------------------------------------------
    def e4m3_to_f32(self, code: int) -> float:
        return float(self.lib.orc_e4m3_to_f32(int(code) & 0xFF))

    def bf16_to_f32(self, bits: int) -> float:
        return float(self.lib.orc_bf16_to_f32(int(bits) & 0xFFFF))

    def f32_to_bf16_rne(self, values) -> np.ndarray:
        """fp32 values -> bf16 bit patterns (uint16), round to nearest even."""
        v = np.ascontiguousarray(values, dtype=np.float32).ravel()
        out = np.empty(v.shape, dtype=np.uint16)
        f = self.lib.orc_f32_to_bf16_rne
        for i, x in enumerate(v):
            out[i] = f(ctypes.c_float(x))
        return out.reshape(np.shape(values))

    def f32_to_e4m3_sat(self, values) -> np.ndarray:
        """fp32 values -> E4M3fn codes (uint8), RNE, saturating at +-448."""
        v = np.ascontiguousarray(values, dtype=np.float32).ravel()
        out = np.empty(v.shape, dtype=np.uint8)
        f = self.lib.orc_f32_to_e4m3_sat
        for i, x in enumerate(v):
            out[i] = f(ctypes.c_float(x))
        return out.reshape(np.shape(values))

    def quantize_rows(self, w: np.ndarray):
        """ptpc_fp8 row quantizer: returns (codes uint8 [n,k], scale fp32 [n])."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        n, k = w.shape
        q = np.empty((n, k), dtype=np.uint8)
        s = np.empty((n,), dtype=np.float32)
        self.lib.orc_quantize_rows(_ptr(w), n, k, k, _ptr(q), k, _ptr(s))
        return q, s

    # ---- the GEMV -----------------------------------------------------
    def gemv(self, w: np.ndarray, dtype: int, scale: np.ndarray | None, x: np.ndarray,
             k: int | None = None, threads: int = 1) -> np.ndarray:
        """y = bf16(scale * sum_k W x) in fp32, ascending k.  Returns uint16 [m, n].

        ``w``: [n, >=k] codes (uint8) or bf16 bits (uint16); its row stride is
        taken from the array.  ``x``: [m, >=k] bf16 bits (uint16).
        """
        n, k, ldw = _check_plane(w, dtype, k)
        assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
        m, ldx = x.shape[0], x.strides[0] // 2
        sc = None
        if dtype == DT_E4M3FN:
            sc = np.ascontiguousarray(scale, dtype=np.float32)
            assert sc.shape == (n,)
        y = np.zeros((m, n), dtype=np.uint16)
        rc = self.lib.orc_gemv(_ptr(w), dtype, n, k, ldw, _ptr(sc), _ptr(x), ldx, m, _ptr(y),
                               n, int(threads))
        if rc != 0:
            raise ValueError("orc_gemv rejected its arguments")
        return y

    def gemv_f64(self, w: np.ndarray, dtype: int, scale: np.ndarray | None, x: np.ndarray,
                 k: int | None = None, threads: int = 1):
        """fp64 recompute: (y64 [m,n] float64, mag64 [m,n] = sum|scale*W*x|)."""
        n, k, ldw = _check_plane(w, dtype, k)
        assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
        m, ldx = x.shape[0], x.strides[0] // 2
        sc = None
        if dtype == DT_E4M3FN:
            sc = np.ascontiguousarray(scale, dtype=np.float32)
        y64 = np.zeros((m, n), dtype=np.float64)
        mag = np.zeros((m, n), dtype=np.float64)
        rc = self.lib.orc_gemv_f64(_ptr(w), dtype, n, k, ldw, _ptr(sc), _ptr(x), ldx, m,
                                   _ptr(y64), _ptr(mag), int(threads))
        if rc != 0:
            raise ValueError("orc_gemv_f64 rejected its arguments")
        return y64, mag

    # ---- SiLU-and-multiply of a merged gate_up plane -------------------
    def f64_to_bf16_rne(self, values) -> np.ndarray:
        """fp64 values -> bf16 bit patterns (uint16), one round to nearest even."""
        v = np.ascontiguousarray(values, dtype=np.float64).ravel()
        out = np.empty(v.shape, dtype=np.uint16)
        f = self.lib.orc_f64_to_bf16_rne
        for i, x in enumerate(v):
            out[i] = f(ctypes.c_double(x))
        return out.reshape(np.shape(values))

    def silu_mul_f64(self, g, u) -> np.ndarray:
        """h = silu(g) * u elementwise in fp64 (unrounded); g and u broadcast."""
        g, u = np.broadcast_arrays(np.asarray(g, dtype=np.float64),
                                   np.asarray(u, dtype=np.float64))
        g = np.ascontiguousarray(g)
        u = np.ascontiguousarray(u)
        h = np.empty(g.shape, dtype=np.float64)
        if self.lib.orc_silu_mul_f64(_ptr(g), _ptr(u), g.size, _ptr(h)) != 0:
            raise ValueError("orc_silu_mul_f64 rejected its arguments")
        return h

    def silu_mul(self, g_bits: np.ndarray, u_bits: np.ndarray) -> np.ndarray:
        """bf16(silu(g) * u) from bf16 g and u: fp64 inside, one bf16 rounding."""
        h = self.silu_mul_f64(bf16_bits_to_f64(g_bits), bf16_bits_to_f64(u_bits))
        return self.f64_to_bf16_rne(h)

    def gate_up_silu_mul(self, w: np.ndarray, dtype: int, scale: np.ndarray | None,
                         x: np.ndarray, k: int | None = None, threads: int = 1) -> np.ndarray:
        """The merged gate_up projection followed by SiLU-and-multiply.

        ``w`` is the merged [2I, >=k] plane (rows 0..I-1 gate, I..2I-1 up),
        ``scale`` its [2I] row scales (FP8).  The projection is the GEMV
        above (its bf16 outputs g and u); returns bf16 bits [m, I] of
        silu(g) * u.
        """
        n = w.shape[0]
        assert n % 2 == 0
        y = self.gemv(w, dtype, scale, x, k, threads)
        return self.silu_mul(y[:, : n // 2], y[:, n // 2:])

    # ---- w4a16: MXFP4 weights -------------------------------------------
    def e2m1_to_f32(self, code: int) -> float:
        return float(self.lib.orc_e2m1_to_f32(int(code) & 0xF))

    def e8m0_to_f32(self, code: int) -> float:
        return float(self.lib.orc_e8m0_to_f32(int(code) & 0xFF))

    @staticmethod
    def _mxfp4_args(w, bs, x, k):
        assert w.dtype == np.uint8 and w.ndim == 2 and w.strides[1] == 1
        assert bs.dtype == np.uint8 and bs.ndim == 2 and bs.strides[1] == 1
        assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
        n, ldw_bytes = w.shape[0], w.strides[0]
        k = 2 * w.shape[1] if k is None else k
        assert k <= 2 * w.shape[1] and bs.shape[0] == n and 32 * bs.shape[1] >= k
        return n, k, ldw_bytes, bs.strides[0], x.shape[0], x.strides[0] // 2

    def gemv_mxfp4(self, w: np.ndarray, bs: np.ndarray, x: np.ndarray, k: int | None = None,
                   threads: int = 1) -> np.ndarray:
        """y = bf16(sum_k e2m1(W) * 2^(bs - 127) * x) in fp32, ascending k; uint16 [m, n].

        ``w``: [n, >=k/2] bytes, two codes each (even column in the low
        nibble); ``bs``: [n, >=ceil(k/32)] E8M0 block scales; ``x``: [m, >=k].
        """
        n, k, ldw, ldb, m, ldx = self._mxfp4_args(w, bs, x, k)
        y = np.zeros((m, n), dtype=np.uint16)
        if self.lib.orc_gemv_mxfp4(_ptr(w), n, k, ldw, _ptr(bs), ldb, _ptr(x), ldx, m, _ptr(y), n,
                                   int(threads)) != 0:
            raise ValueError("orc_gemv_mxfp4 rejected its arguments")
        return y

    def gemv_mxfp4_f64(self, w: np.ndarray, bs: np.ndarray, x: np.ndarray, k: int | None = None,
                       threads: int = 1):
        """fp64 recompute: (y64 [m,n], mag64 [m,n] = sum|W x|)."""
        n, k, ldw, ldb, m, ldx = self._mxfp4_args(w, bs, x, k)
        y64 = np.zeros((m, n), dtype=np.float64)
        mag = np.zeros((m, n), dtype=np.float64)
        if self.lib.orc_gemv_mxfp4_f64(_ptr(w), n, k, ldw, _ptr(bs), ldb, _ptr(x), ldx, m,
                                       _ptr(y64), _ptr(mag), int(threads)) != 0:
            raise ValueError("orc_gemv_mxfp4_f64 rejected its arguments")
        return y64, mag

    # ---- block-scaled FP8: one fp32 factor per 128 x 128 block -----------
    @staticmethod
    def _b128_args(w, bs, x, k):
        assert w.dtype == np.uint8 and w.ndim == 2 and w.strides[1] == 1
        assert bs.dtype == np.float32 and bs.ndim == 2 and bs.strides[1] == 4
        assert x.dtype == np.uint16 and x.ndim == 2 and x.strides[1] == 2
        n, ldw = w.shape[0], w.strides[0]
        k = w.shape[1] if k is None else k
        assert k <= w.shape[1] and bs.shape[0] == -(-n // 128) and 128 * bs.shape[1] >= k
        return n, k, ldw, bs.strides[0] // 4, x.shape[0], x.strides[0] // 2

    def gemv_b128(self, w: np.ndarray, bs: np.ndarray, x: np.ndarray, k: int | None = None,
                  threads: int = 1) -> np.ndarray:
        """y = bf16(sum over 128-column blocks of bs * (sum_k W x)) in fp32; uint16 [m, n].

        ``w``: [n, >=k] E4M3 codes; ``bs``: [ceil(n/128), >=ceil(k/128)] fp32
        block factors; ``x``: [m, >=k] bf16 bits.
        """
        n, k, ldw, ldb, m, ldx = self._b128_args(w, bs, x, k)
        y = np.zeros((m, n), dtype=np.uint16)
        if self.lib.orc_gemv_e4m3_b128(_ptr(w), n, k, ldw, _ptr(bs), ldb, _ptr(x), ldx, m,
                                       _ptr(y), n, int(threads)) != 0:
            raise ValueError("orc_gemv_e4m3_b128 rejected its arguments")
        return y

    def gemv_b128_f64(self, w: np.ndarray, bs: np.ndarray, x: np.ndarray,
                      k: int | None = None, threads: int = 1):
        """fp64 recompute: (y64 [m,n], mag64 [m,n] = sum|bs * W * x|)."""
        n, k, ldw, ldb, m, ldx = self._b128_args(w, bs, x, k)
        y64 = np.zeros((m, n), dtype=np.float64)
        mag = np.zeros((m, n), dtype=np.float64)
        if self.lib.orc_gemv_e4m3_b128_f64(_ptr(w), n, k, ldw, _ptr(bs), ldb, _ptr(x), ldx, m,
                                           _ptr(y64), _ptr(mag), int(threads)) != 0:
            raise ValueError("orc_gemv_e4m3_b128_f64 rejected its arguments")
        return y64, mag

    def max_threads(self) -> int:
        return int(self.lib.orc_max_threads())

    # ---- helpers that hold no method arithmetic ------------------------
    bf16_bits_to_f64 = staticmethod(lambda bits: bf16_bits_to_f64(bits))
    within_tolerance = staticmethod(lambda y, y64, mag: within_tolerance(y, y64, mag))


def _load() -> Oracle:
    global _default
    with _lock:
        if _default is not None:
            return _default
        src = os.path.join(os.path.dirname(__file__), "w8_oracle.c")
        if not os.path.exists(ORACLE_SO) or os.path.getmtime(ORACLE_SO) < os.path.getmtime(src):
            build_oracle()
        _default = Oracle(ctypes.CDLL(ORACLE_SO))
        return _default


def load_variant(so_path: str) -> Oracle:
    """Bind the API to another compiled copy (the mutation tests use this)."""
    return Oracle(ctypes.CDLL(so_path))


def e4m3_to_f32(code):
    return _load().e4m3_to_f32(code)


def bf16_to_f32(bits):
    return _load().bf16_to_f32(bits)


def f32_to_bf16_rne(values):
    return _load().f32_to_bf16_rne(values)


def f32_to_e4m3_sat(values):
    return _load().f32_to_e4m3_sat(values)


def quantize_rows(w):
    return _load().quantize_rows(w)


def gemv(w, dtype, scale, x, k=None, threads=1):
    return _load().gemv(w, dtype, scale, x, k, threads)


def gemv_f64(w, dtype, scale, x, k=None, threads=1):
    return _load().gemv_f64(w, dtype, scale, x, k, threads)


def max_threads():
    return _load().max_threads()


def f64_to_bf16_rne(values):
    return _load().f64_to_bf16_rne(values)


def e2m1_to_f32(code):
    return _load().e2m1_to_f32(code)


def e8m0_to_f32(code):
    return _load().e8m0_to_f32(code)


def gemv_mxfp4(w, bs, x, k=None, threads=1):
    return _load().gemv_mxfp4(w, bs, x, k, threads)


def gemv_mxfp4_f64(w, bs, x, k=None, threads=1):
    return _load().gemv_mxfp4_f64(w, bs, x, k, threads)


def gemv_b128(w, bs, x, k=None, threads=1):
    return _load().gemv_b128(w, bs, x, k, threads)


def gemv_b128_f64(w, bs, x, k=None, threads=1):
    return _load().gemv_b128_f64(w, bs, x, k, threads)


def silu_mul_f64(g, u):
    return _load().silu_mul_f64(g, u)


def silu_mul(g_bits, u_bits):
    return _load().silu_mul(g_bits, u_bits)


def gate_up_silu_mul(w, dtype, scale, x, k=None, threads=1):
    return _load().gate_up_silu_mul(w, dtype, scale, x, k, threads)


# --------------------------------------------------------------------------
# the tolerance of the parity tests
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def within_tolerance(y_bits: np.ndarray, y64: np.ndarray, mag64: np.ndarray):
    """|y - y64| <= 2^-7 |y64| + 2^-12 sum|scale W x|, NaN matching NaN.

    This is the stated parity tolerance for the w8a16 GEMV: twice the bf16
    half-ulp for the final rounding plus 2^-12 of the absolute sum for the
    fp32 accumulation.  Returns (ok: bool, worst ratio |err|/bound).
    """
    y = bf16_bits_to_f64(y_bits)
    nan_ref = np.isnan(y64)
    nan_y = np.isnan(y)
    if not np.array_equal(nan_ref, nan_y):
        return False, float("inf")
    fin = ~nan_ref
    err = np.abs(y[fin] - y64[fin])
    bound = 2.0 ** -7 * np.abs(y64[fin]) + 2.0 ** -12 * mag64[fin]
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(worst <= 1.0), worst


# sup |silu'(v)| over the reals (attained near v = 2.40: 1.0998...); the
# tolerance below uses it as the Lipschitz constant of silu, and a CPU test
# checks it on a fine grid.
SILU_LIPSCHITZ = 1.1


def silu_mul_within_tolerance(h_bits: np.ndarray, g64: np.ndarray, mag_g: np.ndarray,
                              u64: np.ndarray, mag_u: np.ndarray):
    """Parity bound for h = bf16(silu(g) * u) computed from GEMV outputs g, u.

    g64 / u64 are the fp64 recomputes of the two projections and mag_g /
    mag_u their absolute sums (gemv_f64).  The GEMV's own bound gives
    |g - g64| <= Eg = 2^-7 |g64| + 2^-12 mag_g (and Eu for u).  Then

      |silu(g) u - silu(g64) u64| <= L Eg (|u64| + Eu) + |silu(g64)| Eu =: D

    with L = SILU_LIPSCHITZ, and the fp32 evaluation (a few fp32 roundings,
    2^-20 relative) plus the final bf16 rounding (2^-8 relative) add
    (2^-8 + 2^-20)(|H| + D), H = silu(g64) u64.  A floor of
    2^-120 (|u64| + Eu + 1) covers fp32 underflow of silu at very negative
    g.  NaN must match NaN.  Returns (ok, worst ratio |err| / bound).
    """
    h = bf16_bits_to_f64(h_bits)
    big_h = silu_mul_f64(g64, u64)
    s = np.abs(silu_mul_f64(g64, 1.0))
    eg = 2.0 ** -7 * np.abs(g64) + 2.0 ** -12 * mag_g
    eu = 2.0 ** -7 * np.abs(u64) + 2.0 ** -12 * mag_u
    d = SILU_LIPSCHITZ * eg * (np.abs(u64) + eu) + s * eu
    nan_ref = np.isnan(big_h)
    if not np.array_equal(nan_ref, np.isnan(h)):
        return False, float("inf")
    fin = ~nan_ref
    bound = (d + (2.0 ** -8 + 2.0 ** -20) * (np.abs(big_h) + d)
             + 2.0 ** -120 * (np.abs(u64) + eu + 1.0))[fin]
    err = np.abs(h[fin] - big_h[fin])
    ratio = err / bound
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(worst <= 1.0), worst


def same_values(a_bits: np.ndarray, b_bits: np.ndarray) -> bool:
    """Bit-for-bit equality of bf16 results, with +0 == -0 and NaN == NaN.

    The sign of an exact zero depends on where a sum starts, and a NaN's
    payload is not part of the method; every other pattern must match.
    """
    a = np.ascontiguousarray(a_bits, dtype=np.uint16)
    b = np.ascontiguousarray(b_bits, dtype=np.uint16)
    if a.shape != b.shape:
        return False
    za = (a & 0x7FFF) == 0
    zb = (b & 0x7FFF) == 0
    na = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nb = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    if not np.array_equal(za, zb) or not np.array_equal(na, nb):
        return False
    rest = ~(za | na)
    return bool(np.array_equal(a[rest], b[rest]))


__all__ = [
    "DT_E4M3FN", "DT_BF16", "Oracle", "load_variant", "e4m3_to_f32", "bf16_to_f32",
    "f32_to_bf16_rne", "f32_to_e4m3_sat", "quantize_rows", "gemv", "gemv_f64",
    "max_threads", "bf16_bits_to_f64", "within_tolerance", "same_values", "build_oracle",
    "f64_to_bf16_rne", "silu_mul_f64", "silu_mul", "gate_up_silu_mul", "SILU_LIPSCHITZ",
    "silu_mul_within_tolerance", "e2m1_to_f32", "e8m0_to_f32", "gemv_mxfp4", "gemv_mxfp4_f64",
    "gemv_b128", "gemv_b128_f64",
]
