"""Thin ctypes binding of libw8 (include/w8.h): argument marshalling only.

Every step of the GEMV runs in the library's CUDA kernels; this module turns
torch tensors into pointers, sizes and a stream handle and turns status codes
into exceptions.  PyTorch provides device memory and streams only.  There is
no fallback: if libw8.so is missing, importing this module raises.

Names follow the C ABI: ``validate``, ``packed_bytes``, ``bind`` (w8_bind),
``w8_gemv``, ``bf16_gemv``, ``mxfp4_gemv``, ``w8_gemv_silu_mul``, ``w8_mlp``, ``workspace_bytes``,
``plan_info``, ``packed_offset``, ``gate_up_packed_row``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build_lib

LIB_PATH = build_lib.LIB

DT_E4M3FN, DT_BF16, DT_E4M3FNUZ, DT_E5M2, DT_FP16, DT_MXFP4 = 1, 2, 3, 4, 5, 6
DT_E4M3FN_B128 = 7  # FP8 codes with one fp32 factor per 128 x 128 block
SRC_ROW_MAJOR, SRC_GATE_UP = 0, 1
LAYOUT_MMA_16x32, LAYOUT_MMA_16x32_GATE_UP = 1, 2
MAX_M = 256
ABI_VERSION = 8  # W8_ABI_VERSION of include/w8.h (the structs below follow it)

STATUS = {
    0: "W8_OK", 1: "W8_ERR_NULL", 2: "W8_ERR_DTYPE", 3: "W8_ERR_UNPADDED", 4: "W8_ERR_BIAS",
    5: "W8_ERR_MIXED", 6: "W8_ERR_SHAPE", 7: "W8_ERR_SCALE", 8: "W8_ERR_LAYOUT",
    9: "W8_ERR_CAPACITY", 10: "W8_ERR_ALIGN", 11: "W8_ERR_PLANE", 12: "W8_ERR_DEVICE",
    13: "W8_ERR_CUDA", 14: "W8_ERR_SCRATCH",
}


class W8Error(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"{STATUS.get(status, status)}: {text}")
        self.status = status
        self.name = STATUS.get(status, str(status))


class PlaneDesc(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("block_scale", ctypes.c_void_p), ("ldb", ctypes.c_int64)]


class PlaneInfo(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("layout", ctypes.c_int32), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64), ("row_tiles", ctypes.c_int64),
                ("k_blocks", ctypes.c_int64), ("packed", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("packed_bytes", ctypes.c_size_t),
                ("block_factors", ctypes.c_void_p), ("mxfp4_wide_scales", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("n_tiles", ctypes.c_int32),
                ("row_tiles_per_warp", ctypes.c_int32), ("warps_k", ctypes.c_int32),
                ("depth", ctypes.c_int32), ("row_groups", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("k_blocks_per_warp_max", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("cluster", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libw8.so is not built ({LIB_PATH}); run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` first -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    lib.w8_status_str.argtypes = [st]
    lib.w8_status_str.restype = ctypes.c_char_p
    lib.w8_abi_version.argtypes = []
    lib.w8_abi_version.restype = i32
    lib.w8_validate.argtypes = [ctypes.POINTER(PlaneDesc), i32]
    lib.w8_validate.restype = st
    lib.w8_packed_bytes.argtypes = [ctypes.POINTER(PlaneDesc), i32, ctypes.POINTER(sz)]
    lib.w8_packed_bytes.restype = st
    lib.w8_bind.argtypes = [ctypes.POINTER(PlaneDesc), i32, vp, sz, vp, ctypes.POINTER(vp)]
    lib.w8_bind.restype = st
    lib.w8_release.argtypes = [vp]
    lib.w8_release.restype = None
    lib.w8_build_planes.argtypes = [vp]
    lib.w8_build_planes.restype = i32
    lib.w8_build_info.argtypes = [vp, i32, ctypes.POINTER(PlaneInfo)]
    lib.w8_build_info.restype = st
    lib.w8_plan_info.argtypes = [vp, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.w8_plan_info.restype = st
    lib.w8_plan_shape.argtypes = [i64, i64, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.w8_plan_shape.restype = st
    lib.w8_plan_shape_dtype.argtypes = [i64, i64, i32, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.w8_plan_shape_dtype.restype = st
    lib.w8_workspace_bytes.argtypes = [vp, i32, i32, ctypes.POINTER(sz)]
    lib.w8_workspace_bytes.restype = st
    for name in ("w8_gemv", "bf16_gemv", "w8_gemv_silu_mul", "mxfp4_gemv"):
        f = getattr(lib, name)
        f.argtypes = [vp, i32, vp, i64, i32, vp, i64, vp, sz, vp]
        f.restype = st
    lib.w8_gemv_noalloc.argtypes = [vp, i32, vp, i64, i32, vp, i64, vp]
    lib.w8_gemv_noalloc.restype = st
    lib.w8_mlp.argtypes = [vp, i32, i32, vp, i64, i32, vp, i64, vp, i64, vp, sz, vp]
    lib.w8_mlp.restype = st
    lib.w8_mlp_workspace_bytes.argtypes = [vp, i32, i32, i32, ctypes.POINTER(sz)]
    lib.w8_mlp_workspace_bytes.restype = st
    lib.w8_packed_offset.argtypes = [i32, i64, i64, i64]
    lib.w8_packed_offset.restype = i64
    lib.w8_mxfp4_code_bits.argtypes = [i64, i64, i64, ctypes.POINTER(i64)]
    lib.w8_mxfp4_code_bits.restype = st
    lib.w8_gate_up_packed_row.argtypes = [i64, i64]
    lib.w8_gate_up_packed_row.restype = i64
    lib.w8_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), i32]
    lib.w8_device_status.restype = st
    if lib.w8_abi_version() != ABI_VERSION:
        raise ImportError(f"{LIB_PATH} has ABI {lib.w8_abi_version()}, this binding "
                          f"{ABI_VERSION}: rebuild it")
    return lib


lib = _load()

# every symbol include/w8.h declares
EXPORTS = ("w8_status_str", "w8_abi_version", "w8_validate", "w8_packed_bytes", "w8_bind",
           "w8_release", "w8_build_planes", "w8_build_info", "w8_plan_info", "w8_plan_shape",
           "w8_plan_shape_dtype",
           "w8_workspace_bytes", "w8_gemv", "bf16_gemv", "w8_gemv_silu_mul", "mxfp4_gemv",
           "w8_gemv_noalloc", "w8_mlp", "w8_mlp_workspace_bytes",
           "w8_packed_offset", "w8_mxfp4_code_bits", "w8_gate_up_packed_row", "w8_device_status")


def _check(status: int):
    if status != 0:
        raise W8Error(status, lib.w8_status_str(status).decode())


def status_str(status: int) -> str:
    return lib.w8_status_str(status).decode()


# ---------------------------------------------------------------------------
# plane descriptors
# ---------------------------------------------------------------------------

@dataclass
class Plane:
    """A source plane on the device: w [n, ldw] (uint8 codes or bf16), scale [n] fp32."""

    w: torch.Tensor
    dtype: int
    n: int
    k: int
    ldw: int
    scale: torch.Tensor | None = None
    bias: torch.Tensor | None = None
    layout: int = SRC_ROW_MAJOR
    block_scale: torch.Tensor | None = None  # MXFP4: [n, ldb] uint8 E8M0 scales
    ldb: int | None = None  # block-scaled FP8: row stride of scale in floats

    @staticmethod
    def from_tensor(w: torch.Tensor, scale: torch.Tensor | None = None, k: int | None = None,
                    dtype: int | None = None, layout: int = SRC_ROW_MAJOR) -> "Plane":
        """w: 2-D with unit column stride; uint8 -> E4M3FN codes, bfloat16/int16/uint16 -> bf16.
        layout SRC_GATE_UP: a merged [2I, K] projection, gate rows first, then up."""
        assert w.dim() == 2 and w.stride(1) == 1, "plane must be row-major with unit column stride"
        if dtype is None:
            if w.dtype in (torch.uint8, torch.float8_e4m3fn):
                dtype = DT_E4M3FN
            elif w.dtype in (torch.bfloat16, torch.int16, torch.uint16):
                dtype = DT_BF16
            elif w.dtype == torch.float8_e5m2:
                dtype = DT_E5M2
            elif w.dtype == torch.float8_e4m3fnuz:
                dtype = DT_E4M3FNUZ
            elif w.dtype == torch.float16:
                dtype = DT_FP16
            else:
                raise TypeError(f"no w8 dtype for {w.dtype}")
        return Plane(w=w, dtype=dtype, n=w.shape[0], k=w.shape[1] if k is None else k,
                     ldw=w.stride(0), scale=scale, layout=layout)

    @staticmethod
    def mxfp4(w: torch.Tensor, block_scale: torch.Tensor, k: int | None = None,
              layout: int = SRC_ROW_MAJOR) -> "Plane":
        """An MXFP4 plane: w [n, ldw/2] uint8 (two codes a byte, the even
        column in the low nibble), block_scale [n, ldb] uint8 E8M0."""
        assert w.dim() == 2 and w.stride(1) == 1 and w.element_size() == 1
        assert block_scale.dim() == 2 and block_scale.stride(1) == 1
        ldw = 2 * w.stride(0)
        return Plane(w=w, dtype=DT_MXFP4, n=w.shape[0], k=2 * w.shape[1] if k is None else k,
                     ldw=ldw, layout=layout, block_scale=block_scale)

    @staticmethod
    def e4m3_b128(w: torch.Tensor, factors: torch.Tensor, k: int | None = None) -> "Plane":
        """A block-scaled FP8 plane: w [n, ldw] uint8 E4M3fn codes, factors
        [ceil(n/128), ldb] fp32, entry (i, j) covering rows 128i.. and columns
        128j.. of W."""
        assert w.dim() == 2 and w.stride(1) == 1 and w.element_size() == 1
        assert factors.dim() == 2 and factors.stride(1) == 1 and factors.dtype == torch.float32
        return Plane(w=w, dtype=DT_E4M3FN_B128, n=w.shape[0], k=w.shape[1] if k is None else k,
                     ldw=w.stride(0), scale=factors, ldb=factors.stride(0))

    def desc(self) -> PlaneDesc:
        bs = self.block_scale
        ldb = bs.stride(0) if bs is not None else (self.ldb or 0)
        return PlaneDesc(self.w.data_ptr() if self.w is not None else None, self.dtype,
                         self.layout, self.n, self.k, self.ldw,
                         self.scale.data_ptr() if self.scale is not None else None,
                         self.bias.data_ptr() if self.bias is not None else None,
                         bs.data_ptr() if bs is not None else None, ldb)


def _descs(planes):
    arr = (PlaneDesc * len(planes))()
    for i, p in enumerate(planes):
        arr[i] = p.desc() if isinstance(p, Plane) else p
    return arr


def validate(planes) -> None:
    arr = _descs(planes)
    _check(lib.w8_validate(arr, len(planes)))


def packed_bytes(planes) -> int:
    arr = _descs(planes)
    out = ctypes.c_size_t(0)
    _check(lib.w8_packed_bytes(arr, len(planes), ctypes.byref(out)))
    return int(out.value)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class Build:
    """A bound build: owns the library handle and keeps the packed buffer alive."""

    def __init__(self, handle: int, dst: torch.Tensor, planes):
        self._h = ctypes.c_void_p(handle)
        self.dst = dst
        self.n_planes = lib.w8_build_planes(self._h)

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("build was released")
        return self._h

    def info(self, plane: int = 0) -> PlaneInfo:
        out = PlaneInfo()
        _check(lib.w8_build_info(self.handle, plane, ctypes.byref(out)))
        return out

    def plan(self, plane: int, m: int) -> PlanInfo:
        out = PlanInfo()
        _check(lib.w8_plan_info(self.handle, plane, m, ctypes.byref(out)))
        return out

    def workspace_bytes(self, plane: int = -1, m: int = 0) -> int:
        out = ctypes.c_size_t(0)
        _check(lib.w8_workspace_bytes(self.handle, plane, m, ctypes.byref(out)))
        return int(out.value)

    def new_workspace(self, plane: int = -1, m: int = 0, device=None) -> torch.Tensor:
        """A zero-filled workspace (its counter head must start at zero)."""
        nbytes = max(self.workspace_bytes(plane, m), 256)
        return torch.zeros(nbytes, dtype=torch.uint8, device=device or self.dst.device)

    def mlp_workspace_bytes(self, gate_up: int, down: int, m: int = 0) -> int:
        out = ctypes.c_size_t(0)
        _check(lib.w8_mlp_workspace_bytes(self.handle, gate_up, down, m, ctypes.byref(out)))
        return int(out.value)

    def new_mlp_workspace(self, gate_up: int, down: int, m: int = 0, device=None) -> torch.Tensor:
        """A zero-filled workspace for w8_mlp on (gate_up, down), large enough
        for every gemv call of the build as well."""
        nbytes = max(self.mlp_workspace_bytes(gate_up, down, m), self.workspace_bytes(), 256)
        return torch.zeros(nbytes, dtype=torch.uint8, device=device or self.dst.device)

    def release(self):
        if self._h:
            lib.w8_release(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.release()
        except Exception:
            pass


def bind(planes, dst: torch.Tensor | None = None, stream=None) -> Build:
    """w8_bind: validate and repack planes into dst (allocated here when None)."""
    arr = _descs(planes)
    need = packed_bytes(planes)
    if dst is None:
        dev = planes[0].w.device if isinstance(planes[0], Plane) else torch.device("cuda")
        dst = torch.empty(need, dtype=torch.uint8, device=dev)
    out = ctypes.c_void_p(None)
    _check(lib.w8_bind(arr, len(planes), ctypes.c_void_p(dst.data_ptr()),
                       dst.numel() * dst.element_size(), _stream_ptr(stream), ctypes.byref(out)))
    return Build(out.value, dst, planes)


def _gemv(fn, build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
          workspace: torch.Tensor | None, m: int | None, stream):
    assert x.dim() == 2 and x.stride(1) == 1 and x.element_size() == 2
    assert y.dim() == 2 and y.stride(1) == 1 and y.element_size() == 2
    m = x.shape[0] if m is None else m
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(fn(build.handle, plane, ctypes.c_void_p(x.data_ptr()), x.stride(0), m,
              ctypes.c_void_p(y.data_ptr()), y.stride(0), ws_ptr, ws_bytes, _stream_ptr(stream)))
    return y


def w8_gemv(build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
            workspace: torch.Tensor | None = None, m: int | None = None, stream=None):
    """y[:m, :N] = bf16(scale * W x^T)^T on an E4M3FN build (one kernel launch)."""
    return _gemv(lib.w8_gemv, build, plane, x, y, workspace, m, stream)


def bf16_gemv(build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
              workspace: torch.Tensor | None = None, m: int | None = None, stream=None):
    """y[:m, :N] = bf16(W x^T)^T on a BF16 build (one kernel launch)."""
    return _gemv(lib.bf16_gemv, build, plane, x, y, workspace, m, stream)


def mxfp4_gemv(build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
               workspace: torch.Tensor | None = None, m: int | None = None, stream=None):
    """y[:m, :N] = bf16(dequant(W) x^T)^T on an MXFP4 build (one kernel launch)."""
    return _gemv(lib.mxfp4_gemv, build, plane, x, y, workspace, m, stream)


def w8_gemv_silu_mul(build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
                     workspace: torch.Tensor | None = None, m: int | None = None, stream=None):
    """y[:m, :I] = bf16(silu(g) * u) on a gate_up plane of either dtype (one kernel launch)."""
    return _gemv(lib.w8_gemv_silu_mul, build, plane, x, y, workspace, m, stream)


def w8_mlp(build: Build, gate_up: int, down: int, x: torch.Tensor, h: torch.Tensor,
           y: torch.Tensor, workspace: torch.Tensor | None = None, m: int | None = None,
           stream=None):
    """h[:m, :I] = silu(g) * u on the gate_up plane, then y[:m, :N] = the down
    plane's GEMV on h (two kernel launches, the second dependent on the first)."""
    for t in (x, h, y):
        assert t.dim() == 2 and t.stride(1) == 1 and t.element_size() == 2
    m = x.shape[0] if m is None else m
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.w8_mlp(build.handle, gate_up, down, ctypes.c_void_p(x.data_ptr()), x.stride(0), m,
                      ctypes.c_void_p(h.data_ptr()), h.stride(0),
                      ctypes.c_void_p(y.data_ptr()), y.stride(0),
                      ctypes.c_void_p(ws_ptr), ws_bytes, _stream_ptr(stream)))
    return y


def plan_shape(n: int, k: int, m: int, sm_count: int) -> PlanInfo:
    out = PlanInfo()
    _check(lib.w8_plan_shape(n, k, m, sm_count, ctypes.byref(out)))
    return out


def plan_shape_dtype(n: int, k: int, m: int, sm_count: int, dtype: int) -> PlanInfo:
    """The plan a bound plane of this dtype and shape gets (w8_plan_shape_dtype)."""
    out = PlanInfo()
    _check(lib.w8_plan_shape_dtype(n, k, m, sm_count, dtype, ctypes.byref(out)))
    return out


def w8_gemv_noalloc(build: Build, plane: int, x: torch.Tensor, y: torch.Tensor,
                    m: int | None = None, stream=None):
    """w8_gemv without a workspace: scratch from the library's fixed array."""
    assert x.dim() == 2 and x.stride(1) == 1 and x.element_size() == 2
    assert y.dim() == 2 and y.stride(1) == 1 and y.element_size() == 2
    m = x.shape[0] if m is None else m
    _check(lib.w8_gemv_noalloc(build.handle, plane, ctypes.c_void_p(x.data_ptr()), x.stride(0),
                               m, ctypes.c_void_p(y.data_ptr()), y.stride(0),
                               _stream_ptr(stream)))
    return y


def device_status(reset: bool = False) -> int:
    """The tensor-memory kernel's status word on the current device (0: every
    bounded wait ended normally).  Synchronous."""
    out = ctypes.c_int(0)
    _check(lib.w8_device_status(ctypes.byref(out), 1 if reset else 0))
    return int(out.value)


def packed_offset(dtype: int, k_blocks: int, row: int, col: int) -> int:
    return int(lib.w8_packed_offset(dtype, k_blocks, row, col))


def mxfp4_code_bits(k_blocks: int, row: int, col: int) -> tuple:
    """Bit offsets of an MXFP4 element's (mantissa, exponent low, exponent
    high, sign) bits in the packed runs."""
    out = (ctypes.c_int64 * 4)()
    _check(lib.w8_mxfp4_code_bits(k_blocks, row, col, out))
    return tuple(out)


def gate_up_packed_row(n: int, row: int) -> int:
    return int(lib.w8_gate_up_packed_row(n, row))
