"""Each plausible slip planted in a copy of the oracle's C source must fail
at least one pin of tests/pins.py.  The copies are built into a temporary
directory; the real oracle source is never touched."""
import pytest

import oracle
import pins

S = oracle.SOURCE.read_text()

MUTANTS = {
    "add_becomes_subtract": (
        "acc[i] = oracle_bf16_to_f32(x[i]) + oracle_bf16_to_f32(residual[i]);",
        "acc[i] = oracle_bf16_to_f32(x[i]) - oracle_bf16_to_f32(residual[i]);"),
    "eps_dropped": ("float var_eps = mean + eps;", "float var_eps = mean;"),
    "mean_over_padded_length": ("float mean = sum_sq / (float)hidden;",
                                "float mean = sum_sq / (float)padded;"),
    "mean_by_reciprocal": ("float mean = sum_sq / (float)hidden;",
                           "float mean = sum_sq * (1.0f / (float)hidden);"),
    "weight_index_reversed": ("y[i] = normed * oracle_bf16_to_f32(weight[i]);",
                              "y[i] = normed * oracle_bf16_to_f32(weight[hidden - 1 - i]);"),
    "last_square_dropped": ("sq[i] = acc[i] * acc[i];",
                            "sq[i] = (i + 1 < hidden) ? acc[i] * acc[i] : 0.0f;"),
    "sequential_sum": ("float sum_sq = pairwise_pow2(sq, padded);",
                       "float sum_sq = 0.0f; for (int64_t k = 0; k < padded; ++k) sum_sq += sq[k];"),
    "multiply_reassociated": (
        "float normed = acc[i] * inv_rms;\n        y[i] = normed * oracle_bf16_to_f32(weight[i]);",
        "y[i] = acc[i] * (inv_rms * oracle_bf16_to_f32(weight[i]));"),
    "rsqrt_rounded_once": ("float inv_rms = 1.0f / root;",
                           "inv_rms_unused: ; float inv_rms = (float)(1.0 / sqrt((double)var_eps)); (void)root;"),
    "ties_toward_zero": ("return (lo & 1u) ? (uint16_t)(lo + 1u) : lo;", "return lo;"),
    "ties_to_odd": ("return (lo & 1u) ? (uint16_t)(lo + 1u) : lo;",
                    "return (lo & 1u) ? lo : (uint16_t)(lo + 1u);"),
    "ties_away_in_rne": ("if (discarded > 0x8000u)", "if (discarded >= 0x8000u)"),
    "widen_wrong_shift": ("return f32_from_bits((uint32_t)b << 16);",
                          "return f32_from_bits((uint32_t)b << 15);"),
    "out_store_truncates": ("out[base + i] = store_bf16(y[i], store_mode);",
                            "out[base + i] = store_bf16(y[i], ORACLE_STORE_TRUNC);"),
    "residual_out_from_x": ("residual_out[i] = store_bf16(acc[i], store_mode);",
                            "residual_out[i] = store_bf16(oracle_bf16_to_f32(x[i]), store_mode);"),
    "quant_scale_128": ("float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    "quant_truncating_round": ("q = round_half_even_to_int(y[i] / s);", "q = (int32_t)(y[i] / s);"),
    "quant_by_reciprocal": ("q = round_half_even_to_int(y[i] / s);",
                            "q = round_half_even_to_int(y[i] * (1.0f / s));"),
    "quant_amax_without_abs": ("amax = fmaxf(amax, fabsf(y[i]));", "amax = fmaxf(amax, y[i]);"),
    "plain_norm_adds_zero": ("acc[i] = oracle_bf16_to_f32(x[i]);",
                             "acc[i] = oracle_bf16_to_f32(x[i]) + 0.0f;"),
    "residual_add_subtracts": (
        "float acc = oracle_bf16_to_f32(x[i]) + oracle_bf16_to_f32(residual[i]);",
        "float acc = oracle_bf16_to_f32(x[i]) - oracle_bf16_to_f32(residual[i]);"),
    "residual_add_truncates": ("residual_out[i] = store_bf16(acc, store_mode);",
                               "residual_out[i] = store_bf16(acc, ORACLE_STORE_TRUNC);"),
    "e4m3_scale_480": ("float s = amax / E4M3_MAX;", "float s = amax / 480.0f;"),
    "e4m3_ties_to_odd": ("if (d_hi < d_lo || (d_hi == d_lo && (lo & 1u)))",
                         "if (d_hi < d_lo || (d_hi == d_lo && !(lo & 1u)))"),
    "e4m3_subnormal_exponent": ("return ldexp((double)m, -9);", "return ldexp((double)m, -10);"),
    "e4m3_exponent_bias_8": ("return ldexp(1.0 + m / 8.0, (int)e - 7);",
                             "return ldexp(1.0 + m / 8.0, (int)e - 8);"),
    "e2m1_scale_4": ("float s = amax / E2M1_MAX;", "float s = amax / 4.0f;"),
    "e2m1_ties_to_odd": ("if (d_hi < d_lo || (d_hi == d_lo && (lo & 1u)))\n        c = lo + 1;\n    return (uint8_t)(sign | c);\n}\n\n/* Per-row symmetric e2m1",
                         "if (d_hi < d_lo || (d_hi == d_lo && !(lo & 1u)))\n        c = lo + 1;\n    return (uint8_t)(sign | c);\n}\n\n/* Per-row symmetric e2m1"),
    "e2m1_nibbles_swapped": ("q_out[i / 2] = (uint8_t)(c0 | (c1 << 4));", "q_out[i / 2] = (uint8_t)(c1 | (c0 << 4));"),
    "e4m3_quotient_by_reciprocal": ("q_out[i] = s != 0.0f ? oracle_e4m3_rne(y[i] / s) : 0;",
                                    "q_out[i] = s != 0.0f ? oracle_e4m3_rne(y[i] * (1.0f / s)) : 0;"),
    "qk_group_scale_index_by_group_only": ("q_scale + r * groups + g,", "q_scale + g,"),
    "qk_group_codes_offset_by_group_index": ("(uint8_t*)q_out + base + g * group_size,",
                                             "(uint8_t*)q_out + base + g,"),
    "qk_group_values_not_offset": ("q_scale + r * groups + g, y + g * group_size, group_size);",
                                   "q_scale + r * groups + g, y, group_size);"),
    "qk_group_scale_over_whole_row": (
        "for (int64_t g = 0; g < groups; ++g)\n                quantize_row_e4m3(",
        "float am = 0.0f;\n"
        "            for (int64_t i = 0; i < hidden; ++i) am = fmaxf(am, fabsf(y[i]));\n"
        "            for (int64_t g = 0; g < groups; ++g)\n"
        "                for (int64_t i = 0; i < group_size; ++i) {\n"
        "                    float s = am / E4M3_MAX; q_scale[r * groups + g] = s;\n"
        "                    ((uint8_t*)q_out)[base + g * group_size + i] =\n"
        "                        s != 0.0f ? oracle_e4m3_rne(y[g * group_size + i] / s) : 0; }\n"
        "            if (0) for (int64_t g = 0; g < groups; ++g)\n                quantize_row_e4m3("),
    "qk_k_uses_q_eps": ("k_weight, k_eps, n_k_rows", "k_weight, q_eps, n_k_rows"),
    "qk_k_uses_q_weight": ("k_weight, k_eps, n_k_rows", "q_weight, k_eps, n_k_rows"),
    "qk_q_residual_ignored": ("residual ? residual + base : NULL, weight, eps, hidden, padded,\n                        ORACLE_STORE_RNE, NULL, NULL);\n        if (group_size == 0)",
                              "NULL, weight, eps, hidden, padded,\n                        ORACLE_STORE_RNE, NULL, NULL);\n        if (group_size == 0)"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    assert S.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"{name}.c"
    src.write_text(S.replace(old, new))
    lib = oracle.Oracle(oracle.compile_source(src, tmp_path / f"lib{name}.so"))
    caught = []
    for pin in pins.FAST_PINS:
        try:
            pin(lib)
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
