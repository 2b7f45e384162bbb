"""Negative controls for the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/w8_oracle.c,
compiles the copy to a temporary library and reruns the pins against it: at
least one pin must fail.  This is how the pins show they would catch a
dropped term, a wrong sign, index or exponent, a misplaced scale or a wrong
rounding in the oracle (the PR page, Testing, makes the same demand of its
kernel tests: a broken row factor or a wrong dword order must make them
fail).  The
committed oracle is never modified; mistakes are planted only on the CPU.
"""
from __future__ import annotations

import os

import pytest

import oracle
from oracle.build import ORACLE_SRC, build_oracle

from . import test_oracle_b128 as b128_pins
from . import test_oracle_codecs as codecs
from . import test_oracle_gemv as gemv_pins
from . import test_oracle_mxfp4 as mxfp4_pins
from . import test_oracle_silu as silu_pins

MUTATIONS = {
    "scale_dropped": ("float t = (dtype == ORC_DT_E4M3FN) ? scale[r] * acc : acc;",
                      "float t = acc;"),
    "scale_of_wrong_row": ("? scale[r] * acc : acc;", "? scale[(r + 1) % n] * acc : acc;"),
    "scale_after_bf16_rounding": (
        "float t = (dtype == ORC_DT_E4M3FN) ? scale[r] * acc : acc;",
        "float t = (dtype == ORC_DT_E4M3FN) ? scale[r] * orc_bf16_to_f32("
        "orc_f32_to_bf16_rne(acc)) : acc;"),
    "first_term_dropped": ("for (int64_t j = 0; j < k; ++j) {\n                float wv",
                           "for (int64_t j = 1; j < k; ++j) {\n                float wv"),
    "x_index_reversed": ("float xv = orc_bf16_to_f32(x[i * ldx + j]);\n                float p = wv * xv; /* exact: 4",
                         "float xv = orc_bf16_to_f32(x[i * ldx + (k - 1 - j)]);\n                float p = wv * xv; /* exact: 4"),
    "sign_ignored": ("        v = ldexpf(1.0f + (float)m / 8.0f, e - 7); /* 1.m * 2^(e-7) */\n"
                     "    return s ? -v : v;",
                     "        v = ldexpf(1.0f + (float)m / 8.0f, e - 7); /* 1.m * 2^(e-7) */\n"
                     "    return v;"),
    "exponent_bias_off_by_one": ("e - 7); /* 1.m", "e - 8); /* 1.m"),
    "subnormal_scale_wrong": ("ldexpf((float)m, -9)", "ldexpf((float)m, -10)"),
    "mantissa_over_4": ("1.0f + (float)m / 8.0f", "1.0f + (float)m / 4.0f"),
    "rounding_ties_away": ("up = (int)(kept & 1u);", "up = 1;"),
    "rounding_truncates": ("if (dropped > 0x8000u)\n        up = 1;",
                           "if (dropped > 0x8000u)\n        up = 0;"),
    "bf16_widening_shift_wrong": ("(uint32_t)u << 16;", "(uint32_t)u << 15;"),
    "accumulate_in_bf16": ("float p = wv * xv; /* exact: 4 x 8 significant bits */\n                acc = acc + p;",
                           "float p = wv * xv;\n                acc = orc_bf16_to_f32(orc_f32_to_bf16_rne(acc + p));"),
    "mxfp4_accumulate_in_bf16": (
        "* orc_bf16_to_f32(x[i * ldx + j]);\n                acc = acc + p;",
        "* orc_bf16_to_f32(x[i * ldx + j]);\n                acc = orc_bf16_to_f32(orc_f32_to_bf16_rne(acc + p));"),
    # SiLU-and-multiply and its one-step fp64 -> bf16 rounding
    "silu_exponent_sign": ("double s = g[i] / (1.0 + exp(-g[i]));",
                           "double s = g[i] / (1.0 + exp(g[i]));"),
    "silu_of_up_not_gate": ("double s = g[i] / (1.0 + exp(-g[i]));\n        h[i] = s * u[i];",
                            "double s = u[i] / (1.0 + exp(-u[i]));\n        h[i] = s * g[i];"),
    "silu_multiply_dropped": ("h[i] = s * u[i];", "h[i] = s;"),
    "f64_rounding_through_fp32": ("double r = nearbyint(a / q) * q;",
                                  "double r = (double)orc_bf16_to_f32(orc_f32_to_bf16_rne("
                                  "(float)a));"),
    "f64_rounding_ties_away": ("nearbyint(a / q)", "round(a / q)"),
    "f64_subnormal_spacing": ("if (e < -125)\n        e = -125;", "if (e < -126)\n        e = -126;"),
    # MXFP4 (w4a16)
    "e2m1_exponent_bias": ("ldexpf(1.0f + 0.5f * (float)m, e - 1)", "ldexpf(1.0f + 0.5f * (float)m, e - 2)"),
    "e2m1_mantissa_weight": ("ldexpf(1.0f + 0.5f * (float)m, e - 1)", "ldexpf(1.0f + 0.25f * (float)m, e - 1)"),
    "e2m1_subnormal_dropped": ("float v = (e == 0) ? 0.5f * (float)m :", "float v = (e == 0) ? 0.0f :"),
    "e8m0_bias": ("return ldexpf(1.0f, (int)e - 127);", "return ldexpf(1.0f, (int)e - 128);"),
    "nibble_order_swapped": ("uint8_t code = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);",
                             "uint8_t code = (j & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);"),
    "mxfp4_block_of_16": ("orc_e8m0_to_f32(bs[r * ldb + j / 32])", "orc_e8m0_to_f32(bs[r * ldb + j / 16])"),
    # block-scaled FP8 (indexes kept in bounds so that a mutant reads no stray memory)
    "b128_factor_dropped": ("float scaled = row_factors[j0 / ORC_BLOCK] * part;",
                            "float scaled = part;"),
    "b128_block_index_transposed": (
        "float scaled = row_factors[j0 / ORC_BLOCK] * part;",
        "float scaled = bs[((j0 / ORC_BLOCK) % ((n + ORC_BLOCK - 1) / ORC_BLOCK)) * ldb +"
        " (r / ORC_BLOCK) % ldb] * part;"),
    "b128_row_blocks_of_64": (
        "const float *row_factors = bs + (r / ORC_BLOCK) * ldb;\n        for (int64_t i = 0; i < m; ++i) {\n            float acc = 0.0f;",
        "const float *row_factors = bs + ((r / 64) % ((n + ORC_BLOCK - 1) / ORC_BLOCK)) * ldb;\n        for (int64_t i = 0; i < m; ++i) {\n            float acc = 0.0f;"),
    "b128_first_block_dropped": ("for (int64_t j0 = 0; j0 < k; j0 += ORC_BLOCK) {",
                                 "for (int64_t j0 = ORC_BLOCK; j0 < k; j0 += ORC_BLOCK) {"),
    "b128_total_in_bf16": ("acc = acc + scaled;",
                           "acc = orc_bf16_to_f32(orc_f32_to_bf16_rne(acc + scaled));"),
}

# pins rerun against each mutated copy (test functions that take the oracle)
PINS = [
    lambda o: codecs.test_golden_special_codes(o),
    lambda o: codecs.test_all_256_codes_match_torch_float8(o),
    lambda o: codecs.test_bf16_rne_matches_torch(o),
    lambda o: codecs.test_finite_codes_widen_exactly_to_bf16(o),
    lambda o: gemv_pins.test_one_hot_returns_scaled_code(o, "random"),
    lambda o: gemv_pins.test_one_hot_bf16_plane_returns_weight(o),
    lambda o: gemv_pins.test_exact_sum_inputs_match_rational_result(o),
    lambda o: gemv_pins.test_scale_multiplies_the_reduced_row_once(o),
    lambda o: gemv_pins.test_gemv_against_fp64_brute_force(o, True, 2, 33, 64, 16),
    lambda o: gemv_pins.test_gemv_against_fp64_brute_force(o, False, 5, 40, 63, 9),
    lambda o: silu_pins.test_f64_rounding_agrees_with_fp32_rounding_on_fp32_values(o),
    lambda o: silu_pins.test_f64_rounding_on_exact_midpoints(o),
    lambda o: silu_pins.test_silu_mul_matches_torch_float64_silu(o),
    lambda o: silu_pins.test_silu_closed_forms_and_limits(o),
    lambda o: silu_pins.test_silu_odd_part_identity(o),
    lambda o: silu_pins.test_gate_up_silu_mul_is_nearest_bf16_of_exact_result(o),
    lambda o: mxfp4_pins.test_e2m1_codes_closed_form(o),
    lambda o: mxfp4_pins.test_e8m0_scales_closed_form_and_torch(o),
    lambda o: mxfp4_pins.test_mxfp4_gemv_against_fp64_brute_force(o, 3, 40, 100, 3),
    lambda o: mxfp4_pins.test_mxfp4_one_hot_codes_scales_and_packing(o),
    lambda o: mxfp4_pins.test_mxfp4_exact_sum_inputs_match_rational_result(o),
    lambda o: b128_pins.test_b128_gemv_against_fp64_brute_force(o, 1, 130, 300, 4),
    lambda o: b128_pins.test_b128_one_hot_picks_each_blocks_factor(o),
    lambda o: b128_pins.test_b128_exact_sum_inputs_match_rational_result(o),
    lambda o: b128_pins.test_b128_one_column_block_is_the_row_scaled_gemv(o),
]


def _mutant(tmp_path, name):
    find, repl = MUTATIONS[name]
    src = open(ORACLE_SRC).read()
    assert src.count(find) == 1, f"mutation {name} no longer applies"
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(find, repl))
    so = build_oracle(src=path, out=os.path.join(tmp_path, f"libmut_{name}.so"))
    return oracle.load_variant(so)


# (a mutant may produce garbage bit patterns whose numpy casts warn)
@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    mut = _mutant(str(tmp_path), name)
    caught = []
    for i, pin in enumerate(PINS):
        try:
            pin(mut)
        except AssertionError:
            caught.append(i)
    assert caught, f"no pin caught the mutation {name}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    path = os.path.join(str(tmp_path), "copy.c")
    with open(path, "w") as f:
        f.write(open(ORACLE_SRC).read())
    same = oracle.load_variant(build_oracle(src=path, out=os.path.join(str(tmp_path), "c.so")))
    for pin in PINS:
        pin(same)
