"""Plant plausible mistakes in a copy of the oracle and require that the pins
catch every one of them (no GPU).

Each mutation is a textual edit of fp8q_oracle.c that must apply exactly
once; the edited copy is compiled into a temporary library and the pins are
run against it until one fails.  A mutation that survives every pin means
the pins cannot tell that mistake from the correct oracle.
"""

import pytest

import oracle
import pins

MUTATIONS = {
    "mx_tile_rows_not_interleaved": (
        "int64_t at = (rb * G + cb) * 512 + (r % 32) * 16 + (r / 32) * 4 + cc;",
        "int64_t at = (rb * G + cb) * 512 + r * 4 + cc;",
    ),
    "mx_group_byte_on_one_block_only": (
        "for (int64_t c = 4 * g; c < 4 * g + 4; ++c) {",
        "for (int64_t c = 4 * g; c < 4 * g + 1; ++c) {",
    ),
    "rope_sign_of_sine_term_flipped": (
        "x[ia] = oracle_f32_to_bf16(ac - bs);",
        "x[ia] = oracle_f32_to_bf16(ac + bs);",
    ),
    "rope_cos_and_sin_swapped": (
        "float c = oracle_bf16_to_f32(cs[j]);\n                float sn = oracle_bf16_to_f32(cs[half + j]);",
        "float c = oracle_bf16_to_f32(cs[half + j]);\n                float sn = oracle_bf16_to_f32(cs[j]);",
    ),
    "rope_neox_partner_adjacent": (
        "const int64_t ib = is_neox ? j + half : 2 * j + 1;",
        "const int64_t ib = is_neox ? 2 * j + 1 : 2 * j + 1;",
    ),
    "qk_norm_query_weight_on_key_heads": (
        "const uint16_t *w = h < Hq ? q_w : k_w;",
        "const uint16_t *w = q_w;",
    ),
    "qk_norm_mean_over_half_head": (
        "float inv = oracle_rms_inv((float)acc, D, eps);",
        "float inv = oracle_rms_inv((float)acc, D / 2, eps);",
    ),
    "rope_first_token_position_for_all": (
        "const uint16_t *cs = cos_sin + positions[t] * D;",
        "const uint16_t *cs = cos_sin + positions[0] * D;",
    ),
    "amax_over_first_128_values_only": (
        "for (int64_t i = 0; i < gs; ++i) {\n        float a = fabsf(v[i]);",
        "for (int64_t i = 0; i < (gs < 128 ? gs : 128); ++i) {\n        float a = fabsf(v[i]);",
    ),
    "ties_away_from_zero": (
        "r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;",
        "r = fl + 1.0f;",
    ),
    "ties_to_odd": (
        "r = (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;",
        "r = (fmodf(fl, 2.0f) == 0.0f) ? fl + 1.0f : fl;",
    ),
    "subnormal_binade_off_by_one": (
        "if (k < -6)\n        k = -6;",
        "if (k < -7)\n        k = -7;",
    ),
    "no_subnormals_flush_to_zero": (
        "if (k < -6)\n        k = -6;",
        "if (k < -6)\n        return sign;",
    ),
    "saturation_threshold_480": ("if (a >= 448.0f)\n        return (uint8_t)(sign | 0x7E);",
                                 "if (a >= 480.0f)\n        return (uint8_t)(sign | 0x7E);"),
    "scale_by_reciprocal_of_448": (
        "float s = fmaxf(amax, eps) / 448.0f;",
        "float s = fmaxf(amax, eps) * (1.0f / 448.0f);",
    ),
    "floor_applied_after_division": (
        "float s = fmaxf(amax, eps) / 448.0f;",
        "float s = fmaxf(amax / 448.0f, eps);",
    ),
    "fp8_max_240": (
        "float s = fmaxf(amax, eps) / 448.0f;",
        "float s = fmaxf(amax, eps) / 240.0f;",
    ),
    "quotient_by_reciprocal": (
        "float p = v[i] / s; /* RN32 quotient */",
        "float p = v[i] * (1.0f / s);",
    ),
    "ue8m0_floor_instead_of_ceil": ("return ldexpf(1.0f, e);", "return ldexpf(1.0f, e - 1);"),
    "ue8m0_always_bumps": ("if (f == 0.5f)\n        return s;\n    return ldexpf(1.0f, e);",
                           "return ldexpf(1.0f, e);"),
    "col_major_index_wrong": ("return col_major ? g * T + t : t * G + g;",
                              "return col_major ? t * T + g : t * G + g;"),
    "layout_flag_inverted": ("return col_major ? g * T + t : t * G + g;",
                             "return col_major ? t * G + g : g * T + t;"),
    "amax_signed": ("float a = fabsf(v[i]);\n        if (a > m)", "float a = v[i];\n        if (a > m)"),
    "rms_no_eps": ("float var = mean + eps;", "float var = mean;"),
    "rms_mean_over_h_minus_1": ("float mean = ss / (float)H;", "float mean = ss / (float)(H - 1);"),
    "rms_no_sqrt": ("float rstd = sqrtf(var);", "float rstd = var;"),
    "rms_weight_ignored": ("v[h] = n * oracle_bf16_to_f32(w[h]);", "v[h] = n;"),
    "rms_weight_added": ("v[h] = n * oracle_bf16_to_f32(w[h]);", "v[h] = n + oracle_bf16_to_f32(w[h]);"),
    "rms_residual_not_written": ("rr[h] = zb;", "(void)zb;"),
    "rms_residual_not_added": (
        "float sum = oracle_bf16_to_f32(xr[h]) + oracle_bf16_to_f32(rr[h]);",
        "float sum = oracle_bf16_to_f32(xr[h]);",
    ),
    "rms_norm_on_unrounded_sum": ("z[h] = oracle_bf16_to_f32(zb);", "z[h] = sum;"),
    "bf16_truncates": ("if (low > 0x8000u || (low == 0x8000u && (high & 1u)))",
                       "if (0)"),
    "bf16_ties_away": ("if (low > 0x8000u || (low == 0x8000u && (high & 1u)))",
                       "if (low >= 0x8000u)"),
    "silu_exp_sign": ("float d = 1.0f + expf(-a);", "float d = 1.0f + expf(a);"),
    "silu_missing_one": ("float d = 1.0f + expf(-a);", "float d = expf(-a);"),
    "silu_no_up_factor": ("return sg * b;", "return sg;"),
    "silu_gate_up_swapped": (
        "float a = oracle_bf16_to_f32(xr[g * gs + i]);\n                float b = oracle_bf16_to_f32(xr[I + g * gs + i]);",
        "float b = oracle_bf16_to_f32(xr[g * gs + i]);\n                float a = oracle_bf16_to_f32(xr[I + g * gs + i]);",
    ),
    "silu_up_row_stride_wrong": ("const uint16_t *xr = x + t * 2 * I;", "const uint16_t *xr = x + t * I;"),
    "packed_byte_order_reversed": ("out[word * 4 + (g % 4)] = (uint8_t)(e - 1 + 127);",
                                   "out[word * 4 + (3 - g % 4)] = (uint8_t)(e - 1 + 127);"),
    "packed_stride_unpadded": ("int64_t word = (g / 4) * T_pad + t;", "int64_t word = (g / 4) * T + t;"),
    "packed_exponent_unbiased_off_by_one": ("out[word * 4 + (g % 4)] = (uint8_t)(e - 1 + 127);",
                                            "out[word * 4 + (g % 4)] = (uint8_t)(e + 127);"),
    "packed_groups_fast": ("int64_t word = (g / 4) * T_pad + t;", "int64_t word = t * K + (g / 4);"),
    "rms_sumsq_missing_last": ("for (int64_t h = 0; h < H; ++h)\n            acc += ",
                               "for (int64_t h = 0; h < H - 1; ++h)\n            acc += "),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation {name!r} does not apply exactly once"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / "liboracle_mut.so"))
    caught = None
    with oracle.use_library(lib):
        for pin in pins.ALL_PINS:
            try:
                pin()
            except Exception as e:  # AssertionError, or the oracle rejecting/crashing
                caught = (pin.__name__, type(e).__name__)
                break
    assert caught is not None, f"no pin catches the planted mistake {name!r}"
