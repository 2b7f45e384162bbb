"""Shared helpers of the GPU tests: move seeded inputs to the device, bind,
call the C ABI, read results back.  No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np
import torch

from fp8_weight_only_w8a16_gb300 import synth


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev())


def from_dev(t: torch.Tensor) -> np.ndarray:
    a = t.cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a


def padded(plane: synth.Plane) -> synth.Plane:
    """The same plane with its rows padded with zeros to a multiple of 16 bytes
    (bind refuses unpadded planes; the pad columns lie past K)."""
    elt = plane.w.itemsize
    step = 16 // elt
    if plane.ldw % step == 0:
        return plane
    ldw = -(-plane.ldw // step) * step
    w = np.zeros((plane.n, ldw), dtype=plane.w.dtype)
    w[:, :plane.ldw] = plane.w
    return synth.Plane(plane.dtype, plane.n, plane.k, ldw, w, plane.scale)


def bind_plane(w8, plane: synth.Plane):
    """Bind one source plane (rows padded to 16 bytes if needed) and return
    (build, source tensors)."""
    plane = padded(plane)
    w_d = to_dev(plane.w)
    s_d = to_dev(plane.scale) if plane.scale is not None else None
    p = w8.Plane.from_tensor(w_d, s_d, k=plane.k,
                             dtype=w8.DT_E4M3FN if plane.dtype == "e4m3fn" else w8.DT_BF16)
    b = w8.bind([p])
    return b, (w_d, s_d)


def run_gemv(w8, build, plane_idx: int, x: np.ndarray, n: int, ldy: int | None = None,
             ws: torch.Tensor | None = None, fp8: bool = True, x_dev: torch.Tensor | None = None):
    """y [m, n] (uint16) = the library's GEMV of x (uint16 [m, >=k])."""
    m = x.shape[0] if x_dev is None else x_dev.shape[0]
    ldy = n if ldy is None else ldy
    if x_dev is None:
        # rows padded to 8 elements (the ABI reads x with 16-byte loads)
        k = x.shape[1]
        ldx = -(-k // 8) * 8
        xp = torch.zeros((m, ldx), dtype=torch.int16, device=dev())
        xp[:, :k] = to_dev(x)
        xd = xp[:, :k]
    else:
        xd = x_dev
    y = torch.zeros((m, ldy), dtype=torch.int16, device=dev())
    if ws is None:
        ws = build.new_workspace()
    fn = w8.w8_gemv if fp8 else w8.bf16_gemv
    fn(build, plane_idx, xd, y, ws)
    torch.cuda.synchronize()
    return from_dev(y)[:, :n]
