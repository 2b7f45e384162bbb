"""Pins for the oracle's codecs (CPU only).

Each check holds the C oracle to something other than itself: closed-form
values of the E4M3fn format (tests/golden/e4m3_special_codes.txt), torch's own
float8_e4m3fn and bfloat16 conversions, and structural invariants of the
format (ordering, uniform spacing within a binade).  The method depends on
every E4M3 code having an exact bf16 value (ATOM PR #2980, Summary), and the
GPU tests cover each of the format's finite codes (same page, Testing).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_special_codes.txt")


def _golden_codes():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, value = line.split()[:2]
            rows.append((int(code, 16), value))
    return rows


def test_golden_special_codes(orc):
    rows = _golden_codes()
    assert len(rows) >= 12
    for code, value in rows:
        got = orc.e4m3_to_f32(code)
        if value == "nan":
            assert math.isnan(got), hex(code)
            continue
        want = float(Fraction(value))
        assert got == want, (hex(code), got, want)
        if value.startswith("-"):
            assert math.copysign(1.0, got) < 0, hex(code)
        else:
            assert math.copysign(1.0, got) > 0, hex(code)


def test_all_256_codes_match_torch_float8(orc):
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = orc.e4m3_to_f32(c)
        if math.isnan(lib[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == lib[c] and math.copysign(1, got) == math.copysign(1, lib[c]), hex(c)


def test_exactly_254_finite_codes_and_nan_codes(orc):
    vals = [orc.e4m3_to_f32(c) for c in range(256)]
    nan_codes = [c for c, v in enumerate(vals) if math.isnan(v)]
    assert nan_codes == [0x7F, 0xFF]
    assert sum(1 for v in vals if math.isfinite(v)) == 254
    assert not any(math.isinf(v) for v in vals)
    assert max(v for v in vals if math.isfinite(v)) == 448.0


def test_finite_codes_widen_exactly_to_bf16(orc):
    """Every finite E4M3 value is a bf16 value (checked in fp64, by torch)."""
    for c in range(256):
        v = orc.e4m3_to_f32(c)
        if math.isnan(v):
            continue
        as_bf16 = torch.tensor([v], dtype=torch.float64).to(torch.bfloat16).to(torch.float64)
        assert as_bf16.item() == v, hex(c)
        bits = int(orc.f32_to_bf16_rne(np.float32(v)))
        assert orc.bf16_to_f32(bits) == v, hex(c)


def test_codes_are_ordered_and_binades_evenly_spaced(orc):
    pos = [orc.e4m3_to_f32(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    for c in range(0x7F):
        assert orc.e4m3_to_f32(c | 0x80) == -pos[c]
    # subnormals and the first normal binade share one spacing; every later
    # binade of 8 codes doubles it
    steps = [Fraction(b) - Fraction(a) for a, b in zip(pos, pos[1:])]
    assert len(set(steps[:16])) == 1
    for e in range(2, 16):
        binade = steps[8 * e: min(8 * e + 7, len(steps))]
        assert len(set(binade)) == 1
        assert binade[0] == 2 * steps[8 * (e - 1)]


def test_bf16_roundtrip_all_patterns(orc):
    for bits in range(0, 1 << 16, 1):
        f = orc.bf16_to_f32(bits)
        back = int(orc.f32_to_bf16_rne(np.float32(f)))
        if math.isnan(f):
            assert (back & 0x7F80) == 0x7F80 and (back & 0x7F) != 0
        else:
            assert back == bits, hex(bits)


def _torch_bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(1)
    parts = [
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  np.float32(3.4028235e38)], dtype=np.float32),
    ]
    # exact ties: a bf16 value plus half its ulp, both parities of the kept bit
    base = rng.integers(0x0080, 0x7F00, 3000, dtype=np.uint32)
    ties = ((base << 16) | 0x8000).view(np.float32)
    near = ((base << 16) | 0x7FFF).view(np.float32)
    above = ((base << 16) | 0x8001).view(np.float32)
    v = np.concatenate(parts + [ties, -ties, near, above])
    got = orc.f32_to_bf16_rne(v)
    want = _torch_bf16_bits(v)
    assert np.array_equal(got, want)
    nan = np.array([np.nan], dtype=np.float32)
    nb = int(orc.f32_to_bf16_rne(nan)[0])
    assert (nb & 0x7F80) == 0x7F80 and (nb & 0x7F) != 0


def test_e4m3_encoder_matches_torch_rne(orc):
    rng = np.random.default_rng(2)
    vals = [rng.uniform(-448, 448, 3000), rng.standard_normal(3000) * 0.05,
            rng.standard_normal(1000) * 1e-3]
    # exact midpoints between neighbouring codes (ties to even mantissa)
    pos = np.array([orc.e4m3_to_f32(c) for c in range(0x7F)], dtype=np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    v = np.concatenate(vals + [mids, -mids]).astype(np.float32)
    got = orc.f32_to_e4m3_sat(v)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)
    # saturation instead of NaN beyond the largest code
    big = np.array([448.0, 460.0, 500.0, 1e6, -1e6, np.inf, -np.inf], dtype=np.float32)
    assert list(orc.f32_to_e4m3_sat(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_decode_encode_identity_on_finite_codes(orc):
    for c in range(256):
        v = orc.e4m3_to_f32(c)
        if math.isnan(v):
            continue
        assert int(orc.f32_to_e4m3_sat(np.float32(v))) == c, hex(c)


def test_quantizer_matches_input_generator(orc):
    """The oracle's ptpc_fp8 quantizer (brute-force nearest code) and the
    generator's torch-based one give the same codes and scales."""
    from fp8_weight_only_w8a16_gb300 import synth

    rng = np.random.default_rng(3)
    w = (rng.standard_normal((24, 200)) * 0.02).astype(np.float32)
    w[5] = 0.0  # an all-zero row gets scale 1
    q1, s1 = orc.quantize_rows(w)
    q2, s2 = synth.quantize_ptpc_fp8(w)
    assert np.array_equal(s1, s2)
    assert s1[5] == 1.0
    assert np.array_equal(q1, q2)
    # every row reaches the largest code (amax maps to 448)
    nz = [r for r in range(24) if r != 5]
    assert all(np.any((q1[r] & 0x7F) == 0x7E) for r in nz)
