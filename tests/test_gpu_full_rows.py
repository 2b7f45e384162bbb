"""Every row of full-size GLM-5.2 planes against the oracle, once per kernel path.

The other GPU tests compare full-size planes on sampled rows; here every
output of one full-size call per kernel path is compared with the oracle's
fp64 recompute (16 threads) within |y - y64| <= 2^-7 |y64| + 2^-12
sum|scale W x| (ATOM PR #2980, Testing: served outputs held to the fp32
rounding bound of an fp64 recomputation), in the launch configuration the
bench uses (the plan of this GPU's SM count):

* o_proj E4M3 [6144, 16384] at 8 tokens: the register ring, 3 CTAs per SM;
* fused_qkv_a_proj E4M3 [2624, 6144] at 16 tokens: the register ring with
  two token groups;
* q_b_proj E4M3 [16384, 2048] at 48 tokens: the tensor-memory kernel with
  split-K clusters;
* o_proj E4M3 [6144, 16384] at 64 tokens: the tensor-memory kernel with one
  CTA per SM and the deeper ring, 3 K ranges meeting in the workspace;
* kv_b_proj E4M3 [28672, 512] at 256 tokens: the tensor-memory kernel, one
  CTA per SM over two waves;
* o_proj MXFP4 [6144, 16384] at 8 tokens and fused_qkv_a_proj block-scaled
  FP8 [2624, 6144] at 16 tokens: the register ring on the other weight formats.
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


def _call(w8, fn, b, x, n):
    m = x.shape[0]
    y = torch.full((m, n), 0x7FC1, dtype=torch.int16, device=dev())
    fn(b, 0, to_dev(x), y, b.new_workspace())
    torch.cuda.synchronize()
    return from_dev(y)


def _assert_within(y, y64, mag):
    assert not np.any(y == 0x7FC1), "an output was never written"
    ok, worst = oracle.within_tolerance(y, y64, mag)
    assert ok, f"outside tolerance: worst ratio {worst:.3g}"


@pytest.mark.parametrize("n,k,m,kernel", [(6144, 16384, 8, 0), (2624, 6144, 16, 0),
                                          (16384, 2048, 48, 1), (6144, 16384, 64, 1),
                                          (28672, 512, 256, 1)],
                         ids=["o_proj_m8", "fused_qkv_a_m16", "q_b_m48", "o_proj_m64",
                              "kv_b_m256"])
def test_every_row_e4m3(w8, n, k, m, kernel):
    plane, x_all = synth.workload(n, k, "e4m3fn", seed=11)
    x = np.ascontiguousarray(x_all[:m])
    b = w8.bind([w8.Plane.from_tensor(to_dev(plane.w), to_dev(plane.scale))])
    p = b.plan(0, m)
    assert p.kernel == kernel
    sms = torch.cuda.get_device_properties(dev()).multi_processor_count
    if kernel == 1 and m == 48:
        assert p.splits > 1 and p.cluster == p.splits  # a cluster adds its split partial tiles
    if kernel == 1 and m == 64 and sms == 152:
        assert p.ctas_per_sm == 1 and p.splits == 3 and p.cluster == 1
    if kernel == 1 and m == 256:
        assert p.grid > torch.cuda.get_device_properties(dev()).multi_processor_count
    w8.device_status(reset=True)
    y = _call(w8, w8.w8_gemv, b, x, n)
    assert w8.device_status() == 0
    y64, mag = oracle.gemv_f64(plane.w, oracle.DT_E4M3FN, plane.scale, x, threads=16)
    _assert_within(y, y64, mag)


def test_every_row_mxfp4_o_proj(w8):
    n, k, m = 6144, 16384, 8
    plane, x_all = synth.workload(n, k, "mxfp4", seed=12)
    x = np.ascontiguousarray(x_all[:m])
    b = w8.bind([w8.Plane.mxfp4(to_dev(plane.w), to_dev(np.ascontiguousarray(plane.scale)), k=k)])
    assert b.plan(0, m).kernel == 0
    y = _call(w8, w8.mxfp4_gemv, b, x, n)
    y64, mag = oracle.gemv_mxfp4_f64(plane.w, plane.scale, x, k=k, threads=16)
    _assert_within(y, y64, mag)


def test_every_row_block_scaled_fused_qkv_a(w8):
    n, k, m = 2624, 6144, 16
    plane, x_all = synth.workload(n, k, "e4m3fn_b128", seed=13)
    x = np.ascontiguousarray(x_all[:m])
    b = w8.bind([w8.Plane.e4m3_b128(to_dev(plane.w),
                                    to_dev(np.ascontiguousarray(plane.scale, dtype=np.float32)),
                                    k=k)])
    assert b.plan(0, m).kernel == 0
    y = _call(w8, w8.w8_gemv, b, x, n)
    y64, mag = oracle.gemv_b128_f64(plane.w, plane.scale, x, k=k, threads=16)
    _assert_within(y, y64, mag)
