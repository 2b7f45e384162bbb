"""Independent fp64 brute force for tiny inputs (test infrastructure only).

It decodes E4M3 codes and bf16 bits through torch's own dtypes
(``torch.float8_e4m3fn`` and ``torch.bfloat16`` viewed as bytes), not through
the C oracle, and contracts with a numpy float64 matmul.  It therefore shares
no arithmetic with ``w8_oracle.c`` and can pin it: a dropped term, a wrong
sign, a swapped index or a transposed operand in the oracle shows up as a
disagreement far above the fp32 rounding bound.

The method being pinned is the w8a16 GEMV of ATOM PR #2980 (Summary,
Changes): y = bf16(scale[n] * sum_k W[n,k] x[m,k]).
"""
from __future__ import annotations

import numpy as np
import torch


def decode_e4m3_lib(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def decode_bf16_lib(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def gemv_f64_brute(w: np.ndarray, is_fp8: bool, scale, x: np.ndarray, k: int) -> np.ndarray:
    """scale[n] * (W[:, :k] @ x[:, :k]^T)^T in float64, shape [m, n]."""
    wd = decode_e4m3_lib(w[:, :k]) if is_fp8 else decode_bf16_lib(w[:, :k])
    xd = decode_bf16_lib(x[:, :k])
    y = xd @ wd.T
    if is_fp8:
        y = y * np.asarray(scale, dtype=np.float64)[None, :]
    return y
