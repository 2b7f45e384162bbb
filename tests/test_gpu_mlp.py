"""GPU parity of the MLP call (w8_mlp): gate_up with SiLU-and-multiply, then
the down projection, in one call (two dependent kernel launches).

The MLP is the Llama MLP of the ATOM Model Support Guide (Model architecture
details): a merged [2I, K] gate and up projection, h = silu(gate) * up, then
the down projection [N, I] on h.  The call is defined as the two calls in
sequence (and equals them bit for bit), so each output is checked against
the oracle on its own inputs:

* h within the propagated SiLU-and-multiply tolerance of the oracle's fp64
  recompute of the gate_up projection on x;
* y within the GEMV tolerance of the oracle's fp64 recompute of the down
  projection on the h the GPU wrote (the GPU's h, so that the check of y
  does not inherit h's rounding);

for E4M3FN, BF16 and MXFP4 builds, on shapes that give 1 to 64 tokens, split
K in either projection, ragged row and K tails, the tensor-memory kernel for
the down projection (E4M3FN, 100 tokens), and the full-size GLM-5.2 shared
expert (gate_up [4096, 6144], down [6144, 2048]) on every row.  Also: the
result equals the two calls made one after the other, bit for bit;
back-to-back calls and gemv calls sharing one workspace leave its counter
head at zero; and the host refusals, which enqueue nothing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_weight_only_w8a16_gb300 import synth

from .gpu_util import dev, from_dev, padded, to_dev

pytestmark = pytest.mark.gpu

DTYPES = ["e4m3fn", "bf16", "mxfp4"]


@pytest.fixture(scope="module")
def w8():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_weight_only_w8a16_gb300 import w8 as lib

    return lib


def _plane(w8, p: synth.Plane, gated: bool):
    layout = w8.SRC_GATE_UP if gated else w8.SRC_ROW_MAJOR
    if p.dtype == "mxfp4":
        return w8.Plane.mxfp4(to_dev(p.w), to_dev(np.ascontiguousarray(p.scale)), k=p.k,
                              layout=layout)
    p = padded(p)
    return w8.Plane.from_tensor(to_dev(p.w), to_dev(p.scale) if p.scale is not None else None,
                                k=p.k, dtype=w8.DT_E4M3FN if p.dtype == "e4m3fn" else w8.DT_BF16,
                                layout=layout)


def _gemv64(p: synth.Plane, x: np.ndarray, threads: int = 16):
    if p.dtype == "mxfp4":
        return oracle.gemv_mxfp4_f64(p.w, p.scale, x, k=p.k, threads=threads)
    dt = oracle.DT_E4M3FN if p.dtype == "e4m3fn" else oracle.DT_BF16
    return oracle.gemv_f64(p.w, dt, p.scale, x, k=p.k, threads=threads)


def _rows(m: int, k: int) -> torch.Tensor:
    """A [m, k] bf16 view with rows padded to 8 elements (16-byte loads)."""
    ld = -(-k // 8) * 8
    return torch.full((m, ld), 0x7FC1, dtype=torch.int16, device=dev())[:, :k]


class Mlp:
    def __init__(self, w8, n2: int, k: int, n: int, dtype: str, seed: int):
        rng = np.random.default_rng(seed)

        def ldw(kk):  # MXFP4 rows padded to 16 bytes (the others pad on binding)
            return -(-kk // 32) * 32 if dtype == "mxfp4" else None

        self.up = synth.weight_plane(rng, n2, k, dtype, ldw(k))
        self.down = synth.weight_plane(rng, n, n2 // 2, dtype, ldw(n2 // 2))
        self.b = w8.bind([_plane(w8, self.up, True), _plane(w8, self.down, False)])
        self.n2, self.k, self.n, self.i = n2, k, n, n2 // 2
        self.rng = rng

    def run(self, w8, x: np.ndarray, ws: torch.Tensor):
        m = x.shape[0]
        xd = _rows(m, self.k)
        xd.copy_(to_dev(x))
        h = _rows(m, self.i)
        y = torch.full((m, self.n + 3), 0x7FC1, dtype=torch.int16, device=dev())
        w8.w8_mlp(self.b, 0, 1, xd, h, y, ws)
        torch.cuda.synchronize()
        y = from_dev(y)
        assert np.all(y[:, self.n:] == 0x7FC1), "a column past N was written"
        return from_dev(h), y[:, :self.n]

    def check(self, x: np.ndarray, h: np.ndarray, y: np.ndarray):
        assert not np.any(h == 0x7FC1) and not np.any(y == 0x7FC1), "an output was never written"
        g64, mag = _gemv64(self.up, x)
        i = self.i
        ok, worst = oracle.silu_mul_within_tolerance(h, g64[:, :i], mag[:, :i], g64[:, i:],
                                                     mag[:, i:])
        assert ok, f"h outside tolerance: worst ratio {worst:.3g}"
        y64, magy = _gemv64(self.down, np.ascontiguousarray(h))
        ok, worst = oracle.within_tolerance(y, y64, magy)
        assert ok, f"y outside tolerance: worst ratio {worst:.3g}"


# (2I, K, N, m): one to eight token groups; a gate_up plane of two row tiles
# and long K (its items split K); ragged I (K tail of down) and N
SHAPES = [(16, 32, 16, 1), (80, 100, 37, 3), (32, 6144, 64, 5), (512, 3000, 700, 16),
          (256, 1024, 300, 24), (1024, 2048, 512, 33), (160, 704, 1000, 64), (4096, 6144, 6144, 8)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n2,k,n,m", SHAPES)
def test_mlp_matches_oracle(w8, dtype, n2, k, n, m):
    mlp = Mlp(w8, n2, k, n, dtype, seed=n2 + 7 * k + n + m)
    x = synth.activations(mlp.rng, k, m)
    ws = mlp.b.new_mlp_workspace(0, 1)
    w8.device_status(reset=True)
    h, y = mlp.run(w8, x, ws)
    mlp.check(x, h, y)
    assert w8.device_status() == 0


def test_mlp_equals_the_two_calls(w8):
    """w8_mlp gives w8_gemv_silu_mul's h and then w8_gemv's y on it, bit for bit."""
    mlp = Mlp(w8, 512, 3000, 700, "e4m3fn", seed=3)
    ws = mlp.b.new_mlp_workspace(0, 1)
    for m in (1, 8, 16, 40):
        x = synth.activations(mlp.rng, 3000, m)
        h, y = mlp.run(w8, x, ws)
        xd = _rows(m, 3000)
        xd.copy_(to_dev(x))
        h2 = _rows(m, 256)
        y2 = torch.zeros((m, 700), dtype=torch.int16, device=dev())
        w8.w8_gemv_silu_mul(mlp.b, 0, xd, h2, ws)
        w8.w8_gemv(mlp.b, 1, h2, y2, ws)
        torch.cuda.synchronize()
        assert oracle.same_values(h, from_dev(h2)) and oracle.same_values(y, from_dev(y2)), m


def test_mlp_down_on_the_tensor_memory_kernel(w8):
    """100 tokens on an E4M3FN build: the down projection [6144, 256] runs the
    tensor-memory kernel (at least 17 tokens on 48 blocks of 128 rows)."""
    mlp = Mlp(w8, 512, 1024, 6144, "e4m3fn", seed=17)
    assert mlp.b.plan(1, 100).kernel == 1
    x = synth.activations(mlp.rng, 1024, 100)
    h, y = mlp.run(w8, x, mlp.b.new_mlp_workspace(0, 1))
    mlp.check(x, h, y)


@pytest.mark.parametrize("m", [1, 8, 16])
def test_shared_expert_every_row(w8, m):
    """GLM-5.2's shared expert at full size: gate_up [4096, 6144] and down
    [6144, 2048] (E4M3FN), every h and y of the call."""
    mlp = Mlp(w8, 4096, 6144, 6144, "e4m3fn", seed=21)
    x = synth.activations(mlp.rng, 6144, m)
    ws = mlp.b.new_mlp_workspace(0, 1)
    h, y = mlp.run(w8, x, ws)
    mlp.check(x, h, y)


def test_calls_share_the_workspace(w8):
    """Back-to-back MLP calls and gemv calls on one workspace: every result
    right, and the counter head zero after each."""
    mlp = Mlp(w8, 64, 6144, 96, "e4m3fn", seed=5)  # phase 1 splits K
    other = synth.weight_plane(mlp.rng, 48, 6144, "e4m3fn")
    b = w8.bind([_plane(w8, mlp.up, True), _plane(w8, mlp.down, False), _plane(w8, other, False)])
    mlp.b = b
    ws = torch.zeros(max(b.mlp_workspace_bytes(0, 1), b.workspace_bytes()), dtype=torch.uint8,
                     device=dev())
    head = 4 * (-(-max(64, 96, 48) // 16))  # the arrival counters of the largest plane
    for step in range(3):
        x = synth.activations(mlp.rng, 6144, 4 + step)
        h, y = mlp.run(w8, x, ws)
        mlp.check(x, h, y)
        assert not torch.any(ws[:head]).item(), "the workspace head was left non-zero"
        yo = torch.zeros((x.shape[0], 48), dtype=torch.int16, device=dev())
        w8.w8_gemv(b, 2, to_dev(x), yo, ws)
        torch.cuda.synchronize()
        y64, mag = _gemv64(other, x)
        ok, worst = oracle.within_tolerance(from_dev(yo), y64, mag)
        assert ok, worst
        assert not torch.any(ws[:head]).item()
    assert w8.device_status() == 0


def test_mlp_refusals(w8):
    """Refused calls return their status and enqueue nothing (h keeps its
    contents)."""
    mlp = Mlp(w8, 64, 6144, 40, "e4m3fn", seed=9)  # gate_up splits K: a workspace is needed
    need = mlp.b.mlp_workspace_bytes(0, 1, 2)
    assert need > 0
    ws = mlp.b.new_mlp_workspace(0, 1)
    x = _rows(2, 6144)
    x.zero_()
    h = _rows(2, 32)
    y = torch.zeros((2, 40), dtype=torch.int16, device=dev())

    def status(fn):
        with pytest.raises(w8.W8Error) as e:
            fn()
        torch.cuda.synchronize()
        assert np.all(from_dev(h) == 0x7FC1), "a refused call wrote h"
        return e.value.name

    assert status(lambda: w8.w8_mlp(mlp.b, 1, 0, x, h, y, ws)) == "W8_ERR_LAYOUT"
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 0, x, h, y, ws)) == "W8_ERR_LAYOUT"
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 2, x, h, y, ws)) == "W8_ERR_PLANE"
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 1, x, h, y, ws, m=257)) == "W8_ERR_SHAPE"
    y39 = torch.zeros((2, 39), dtype=torch.int16, device=dev())  # ldy < N
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 1, x, h, y39, ws)) == "W8_ERR_SHAPE"
    hb = torch.zeros((2, 36), dtype=torch.int16, device=dev())[:, :33]  # ldh % 8 != 0
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 1, x, hb, y, ws)) == "W8_ERR_ALIGN"
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 1, x, h, y, ws[:need - 1])) == "W8_ERR_CAPACITY"
    assert status(lambda: w8.w8_mlp(mlp.b, 0, 1, x, h, y, None)) == "W8_ERR_NULL"
    # a down plane whose K is not I
    rng = np.random.default_rng(1)
    bad = synth.weight_plane(rng, 40, 48, "e4m3fn")
    b2 = w8.bind([_plane(w8, mlp.up, True), _plane(w8, bad, False)])
    assert status(lambda: w8.w8_mlp(b2, 0, 1, x, h, y, b2.new_workspace())) == "W8_ERR_SHAPE"
    # m = 0 is a no-op
    w8.w8_mlp(mlp.b, 0, 1, x, h, y, ws, m=0)
    torch.cuda.synchronize()
    assert np.all(from_dev(h) == 0x7FC1)
