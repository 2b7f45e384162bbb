"""Seeded synthetic inputs for the w8a16 GEMV: weight planes and activations.

This module is the one piece both sides share: the tests feed the same bytes
to the CPU oracle and to the CUDA path.  It holds none of the GEMV's
arithmetic (no widening, no accumulation, no scaling of a reduced row, no
output rounding).  Its only numeric steps are input preparation, done with
library routines:

* draws: numpy PCG64 (``default_rng(seed)``), standard normal in fp32; the
  weights are N(0, 0.02) and the activations N(0, 1);
* activations: fp32 -> bf16 through ``torch.Tensor.to(torch.bfloat16)``;
* FP8 planes: the ptpc_fp8 weight format of ATOM PR #2980 (Summary: E4M3
  codes with one fp32 factor for each row): scale[n] = amax_n / 448 in fp32 (an all-zero row
  gets scale 1), codes = E4M3(W / scale) clamped to +-448 and rounded through
  ``torch.float8_e4m3fn`` (round to nearest even);
* block-scaled FP8 planes (the blockscale GEMM's weights; a checkpoint's
  weight_scale_inv): one fp32 factor per 128 x 128 block, amax_block / 448
  (an all-zero block gets 1), codes = E4M3(W / factor) clamped to +-448 and
  rounded through ``torch.float8_e4m3fn``;
* bf16 planes: fp32 -> bf16 through torch;
* MXFP4 planes (w4a16; the OCP microscaling format the Model Support Guide's
  FP4 GEMMs use): per row and 32-column block, the shared exponent is
  floor(log2(amax)) - 2 (E2M1's largest exponent), stored as E8M0 (bias 127;
  an all-zero block gets 127); elements = W / 2^exponent rounded to the
  nearest E2M1 value (ties to the even code), saturating at +-6; two codes per
  byte, the even column in the low nibble.

Draw order per workload: the weight plane first, then a [256, K] activation
block whose first M rows are the M decode tokens, so every M of one workload
sees the same prefix of tokens.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

E4M3_MAX = 448.0
X_ROWS = 256  # largest token count of the workloads (rows are drawn row-major, so
              # the first rows do not depend on how many are drawn)


@dataclass
class Plane:
    """A source weight plane as a checkpoint would hold it (row-major)."""

    dtype: str            # "e4m3fn", "e4m3fn_b128", "bf16" or "mxfp4"
    n: int
    k: int                # logical columns
    ldw: int              # row stride in elements (>= k); columns k..ldw-1 are zero
    w: np.ndarray         # [n, ldw] uint8 codes or uint16 bf16 bits; MXFP4: [n, ldw / 2]
                          # bytes of two codes (even column in the low nibble)
    scale: np.ndarray | None  # [n] fp32 row scales (FP8); MXFP4: [n, ceil(k / 32)]
                              # E8M0 block scales (uint8); block-scaled FP8:
                              # [ceil(n / 128), ceil(k / 128)] fp32; None for bf16


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    z = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return z


def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def quantize_ptpc_fp8(w: np.ndarray):
    """fp32 [n, k] -> (E4M3fn codes uint8 [n, k], fp32 row scales [n])."""
    t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))
    amax = t.abs().amax(dim=1) if t.shape[1] > 0 else torch.zeros(t.shape[0])
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (t / scale[:, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy().copy(), scale.numpy().astype(np.float32)


def quantize_fp8_b128(w: np.ndarray, block: int = 128):
    """fp32 [n, k] -> (E4M3fn codes uint8 [n, k], fp32 factors [ceil(n/128), ceil(k/128)])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    nbr, nbc = -(-n // block), -(-k // block)
    t = torch.zeros((nbr * block, nbc * block), dtype=torch.float32)
    t[:n, :k] = torch.from_numpy(w)
    blocks = t.view(nbr, block, nbc, block)
    amax = blocks.abs().amax(dim=(1, 3))
    factor = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (blocks / factor[:, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = q.reshape(nbr * block, nbc * block)[:n, :k].contiguous()
    codes = codes.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy().copy(), factor.numpy().astype(np.float32)


# E2M1 magnitudes by code (sign in bit 3): the values an MXFP4 element takes.
_E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def quantize_mxfp4(w: np.ndarray, block: int = 32):
    """fp32 [n, k] -> (packed codes uint8 [n, ceil(k/2)], E8M0 scales uint8 [n, ceil(k/32)])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    nb = -(-k // block)
    wp = np.zeros((n, nb * block), dtype=np.float64)
    wp[:, :k] = w
    blocks = wp.reshape(n, nb, block)
    amax = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, 0)
    ex = np.clip(ex, -127, 127).astype(np.int64)
    scales = (ex + 127).astype(np.uint8)
    v = blocks / np.ldexp(1.0, ex)[:, :, None]
    mag = np.minimum(np.abs(v), 6.0)
    dist = np.abs(mag[..., None] - _E2M1_MAGNITUDES)
    # nearest magnitude; on a tie the even code (an exact midpoint sits between
    # an even and an odd code)
    best = np.argmin(dist * 4 + (np.arange(8) & 1) * 1e-9, axis=-1)
    codes = (best | np.where(v < 0, 8, 0)).astype(np.uint8).reshape(n, nb * block)[:, :k]
    if k % 2:
        codes = np.concatenate([codes, np.zeros((n, 1), np.uint8)], axis=1)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales


def weight_plane(rng: np.random.Generator, n: int, k: int, dtype: str = "e4m3fn",
                 ldw: int | None = None, std: float = 0.02) -> Plane:
    ldw = k if ldw is None else ldw
    assert ldw >= k
    w32 = _normal(rng, (n, k), std)
    if dtype == "e4m3fn":
        codes, scale = quantize_ptpc_fp8(w32)
        w = np.zeros((n, ldw), dtype=np.uint8)
        w[:, :k] = codes
        return Plane("e4m3fn", n, k, ldw, w, scale)
    if dtype == "e4m3fn_b128":
        codes, factor = quantize_fp8_b128(w32)
        w = np.zeros((n, ldw), dtype=np.uint8)
        w[:, :k] = codes
        return Plane("e4m3fn_b128", n, k, ldw, w, factor)
    if dtype == "bf16":
        w = np.zeros((n, ldw), dtype=np.uint16)
        w[:, :k] = to_bf16_bits(w32)
        return Plane("bf16", n, k, ldw, w, None)
    if dtype == "mxfp4":
        assert ldw % 2 == 0
        packed, scales = quantize_mxfp4(w32)
        w = np.zeros((n, ldw // 2), dtype=np.uint8)
        w[:, :packed.shape[1]] = packed
        return Plane("mxfp4", n, k, ldw, w, scales)
    raise ValueError(dtype)


def activations(rng: np.random.Generator, k: int, rows: int = X_ROWS,
                ldx: int | None = None) -> np.ndarray:
    """[rows, ldx] bf16 bits ~ N(0, 1); columns k..ldx-1 (if any) are drawn too."""
    ldx = k if ldx is None else ldx
    return to_bf16_bits(_normal(rng, (rows, ldx), 1.0))


def workload(n: int, k: int, dtype: str = "e4m3fn", seed: int = 0, ldw: int | None = None,
             x_rows: int = X_ROWS):
    """(plane, x_all) for one workload: the plane is drawn before the tokens."""
    rng = np.random.default_rng(seed)
    plane = weight_plane(rng, n, k, dtype, ldw)
    x = activations(rng, k, x_rows)
    return plane, x


def plane_rows(n: int, k: int, dtype: str = "e4m3fn", seed: int = 0, rows: int | None = None,
               ldw: int | None = None) -> Plane:
    """The first `rows` rows (all when None) of the [n, k] plane that
    ``weight_plane(default_rng(seed), n, k, dtype, ldw)`` draws.  The draw
    fills row-major and every supported format quantises each row on its own,
    so a prefix of rows is exactly those rows of the whole plane (block-scaled
    planes only in whole 128-row blocks)."""
    rows = n if rows is None else min(rows, n)
    if dtype == "e4m3fn_b128":
        assert rows == n or rows % 128 == 0, "block-scaled planes: whole row blocks"
    return weight_plane(np.random.default_rng(seed), rows, k, dtype, ldw)


def tokens(k: int, rows: int, seed: int = 0) -> np.ndarray:
    """[rows, k] bf16 bits ~ N(0, 1) drawn from their own stream
    (``default_rng([seed, 1])``), so that they do not depend on a plane's
    draw: the bench's decode tokens."""
    return activations(np.random.default_rng([seed, 1]), k, rows)
