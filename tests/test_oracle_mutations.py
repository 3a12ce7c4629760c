"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies the oracle's C source, plants one mistake (a dropped term, a
wrong or transposed index, a wrong constant, a wrong rounding rule), builds the
copy with gcc into a temporary directory and runs the pin checks against it:
at least one pin must fail.  The committed oracle is never modified.
"""
import contextlib
import os
import subprocess

import pytest

import oracle
import test_oracle_dispatch_combine as tdc
import test_oracle_formats as tfm
import test_oracle_rms_norm as trn
import test_oracle_layout as tl
import test_oracle_nonfinite as tnf
import test_oracle_quant as tq
import test_oracle_quant_ext as tqx
import test_oracle_token_layout as ttl

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")

MUTANTS = {
    "layout_drop_running_position": ("pos[e] += 1;", ""),
    "layout_inclusive_source_prefix": (
        "src_prefix[(int64_t)s * E + e] = acc;\n            acc += cnt[(int64_t)s * E + e];",
        "acc += cnt[(int64_t)s * E + e];\n            src_prefix[(int64_t)s * E + e] = acc;"),
    "layout_alignment_off_by_one": ("aligned[e] = ((c + alpha - 1) / alpha) * alpha;",
                                    "aligned[e] = ((c + alpha) / alpha) * alpha;"),
    "layout_rank_of_expert_modulo": ("itr[n * R + e / L] = 1;", "itr[n * R + e % R] = 1;"),
    "layout_transposed_expert_map": ("int j = (int)(e / L), l = (int)(e % L);",
                                     "int j = (int)(e % R), l = (int)(e / R);"),
    "int8_wrong_type_max": ("float s = 127.0f / amax;", "float s = 128.0f / amax;"),
    "int8_inverse_as_amax_over_127": ("        q[h] = (int8_t)(int)r;\n    }\n    *inv = 1.0f / s;",
                                      "        q[h] = (int8_t)(int)r;\n    }\n    *inv = amax / 127.0f;"),
    "int8_round_half_up": ("return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;", "return f + 1.0f;"),
    "mx_exponent_off_by_one": ("se = (expfield - 127) - m.emax;", "se = (expfield - 127) - m.emax + 1;"),
    "mx_e2m1_nibble_swap": ("codes[h / 2] |= (uint8_t)(c << (4 * (h & 1)));",
                            "codes[h / 2] |= (uint8_t)(c << (4 * (1 - (h & 1))));"),
    "minifloat_ties_away": ("if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;",
                            "if (dhi <= dlo) c = c + 1;"),
    "minifloat_subnormal_scale": ("if (ef == 0) return ldexp((double)mf, 1 - m.bias - m.mbits);",
                                  "if (ef == 0) return ldexp((double)mf, -m.bias - m.mbits);"),
    "bf16_ties_up": ("else pick = (lo & 1u) ? hi : lo;", "else pick = hi;"),
    "combine_first_weight_only": ("float prod = w[n * K + k] * oracle_bf16_to_f32(y[yr * H + h]);",
                                  "float prod = w[n * K] * oracle_bf16_to_f32(y[yr * H + h]);"),
    "fp8_token_wrong_type_max": ("const float dmax = (fp8 == Q_E4M3) ? 448.0f : 57344.0f;",
                                 "const float dmax = (fp8 == Q_E4M3) ? 480.0f : 57344.0f;"),
    "fp8_group_drops_last_group": ("for (int g = 0; g < H / GROUP; ++g)\n        oracle_quant_fp8_token_row(",
                                   "for (int g = 0; g < H / GROUP - 1; ++g)\n        oracle_quant_fp8_token_row("),
    "int8_static_symmetric_saturation": ("if (r < -128.0f) r = -128.0f;", "if (r < -127.0f) r = -127.0f;"),
    "scaled_first_slot_expert": ("sm = scales + topk[n * K + k] * (int64_t)H;",
                                 "sm = scales + topk[n * K] * (int64_t)H;"),
    "mask_token_index": ("int active = (mask_dims == 1) ? mask[i / K] : mask[i];",
                         "int active = (mask_dims == 1) ? mask[i % (R * T)] : mask[i];"),
    "smooth_scales_ignored": ("return smooth ? v * smooth[h] : v;", "return v;"),
    "token_rank_of_expert_modulo": ("if (e >= 0 && e < E && e / L == j) hit = 1;",
                                    "if (e >= 0 && e < E && e % R == j) hit = 1;"),
    "token_global_expert_id": ("recv_topk_idx[row * K + k] = local ? (e - (int64_t)j * L) : -1;",
                               "recv_topk_idx[row * K + k] = local ? e : -1;"),
    "token_foreign_weights_kept": ("recv_topk_weights[row * K + k] = local ? w[n * K + k] : 0.0f;",
                                   "recv_topk_weights[row * K + k] = w[n * K + k];"),
    "token_reduce_skips_last_row": ("            for (int i = 0; i < K; ++i) {\n                int32_t r = tok_dst[n * K + i];",
                                    "            for (int i = 0; i < K - 1; ++i) {\n                int32_t r = tok_dst[n * K + i];"),
    "bytes_source_taken_at_destination": (
        "memcpy(out + (d - row_begin) * row_bytes, src + n * row_bytes, (size_t)row_bytes);",
        "memcpy(out + (d - row_begin) * row_bytes, src + d * row_bytes, (size_t)row_bytes);"),
    "bytes_first_slot_only": ("        for (int k = 0; k < K; ++k) {\n            int64_t d = dst_row[n * K + k];\n            if (d < row_begin || d >= row_end) continue;\n            memcpy(out + (d - row_begin) * row_bytes, src + n",
                              "        for (int k = 0; k < 1; ++k) {\n            int64_t d = dst_row[n * K + k];\n            if (d < row_begin || d >= row_end) continue;\n            memcpy(out + (d - row_begin) * row_bytes, src + n"),
    "expert_group_scale_index": ("memcpy(&inv, s + ((q == Q_FP8G_E4M3 || q == Q_FP8G_E5M2) ? 4 * (h / GROUP) : 0), 4);",
                                 "memcpy(&inv, s + ((q == Q_FP8G_E4M3 || q == Q_FP8G_E5M2) ? 4 * (h / 32) : 0), 4);"),
    "expert_static_codes_unsigned": ("                v = (float)(int8_t)d[h];\n            } else {",
                                     "                v = (float)d[h];\n            } else {"),
    "rms_residual_dropped": ("double v = c[n * H + h] + (double)oracle_bf16_to_f32(residual[n * H + h]);",
                             "double v = c[n * H + h];"),
    "rms_eps_outside_sqrt": ("double r = 1.0 / sqrt(ss / (double)H + eps);",
                             "double r = 1.0 / (sqrt(ss / (double)H) + eps);"),
    "rms_mean_over_h_minus_one": ("double r = 1.0 / sqrt(ss / (double)H + eps);",
                                  "double r = 1.0 / sqrt(ss / (double)(H - 1) + eps);"),
    "rms_gamma_shifted": ("x[n * H + h] * r * (double)oracle_bf16_to_f32(gamma[h]);",
                          "x[n * H + h] * r * (double)oracle_bf16_to_f32(gamma[(h + 1) % H]);"),
    "int8_nan_enters_the_maximum": ("        if (a > amax) amax = a;\n    }\n    float s = 127.0f / amax;",
                                    "        if (!(a <= amax)) amax = a;\n    }\n    float s = 127.0f / amax;"),
    "int8_nan_product_not_zero": ("            if (r != r) r = 0.0f;   /* NaN product",
                                  "            if (r != r) r = 127.0f;   /* NaN product"),
    "int8_upper_clamp_dropped": ("            if (r > 127.0f) r = 127.0f;\n            if (r < -127.0f) r = -127.0f;",
                                 "            if (r < -127.0f) r = -127.0f;"),
    "mx_exponent_cap_too_low": ("if (se > 127) se = 127;", "if (se > 100) se = 100;"),
    "mx_nan_enters_the_block_maximum": ("            if (a > amax) amax = a;\n        }\n        int expfield",
                                        "            if (!(a <= amax)) amax = a;\n        }\n        int expfield"),
    "rms32_residual_dropped": (
        "float v = oracle_bf16_to_f32(c[n * H + h]) + oracle_bf16_to_f32(residual[n * H + h]);",
        "float v = oracle_bf16_to_f32(c[n * H + h]);"),
    "rms32_eps_outside_sqrt": ("float r = 1.0f / sqrtf(mean + eps);", "float r = 1.0f / (sqrtf(mean) + eps);"),
    "rms32_mean_over_h_minus_one": ("float mean = ss / (float)H;", "float mean = ss / (float)(H - 1);"),
    "rms32_y_from_rounded_x": ("float t = x[h] * r;",
                               "float t = oracle_bf16_to_f32(oracle_bf16_from_f32(x[h])) * r;"),
    "combine_shared_axes_transposed": (
        "acc = acc + oracle_bf16_to_f32(shared[((s * S + qq) * T + t) * H + h]);",
        "acc = acc + oracle_bf16_to_f32(shared[((qq * (int64_t)R + s) * T + t) * H + h]);"),
}


def pins():
    """Cheap subset of the pin tests, each a zero-argument callable."""
    cases = [lambda: tl.test_exhaustive_tiny(),
             lambda: tl.test_workload1_matches_brute_force(),
             lambda: tl.test_edge_cases()]
    cases += [lambda s=s: tl.test_random_small(s) for s in range(8)]
    cases += [lambda c=c: tq.test_int8_golden(c) for c in tq.read_cases("int8_rows.txt")]
    cases += [lambda c=c: tq.test_mx_golden(c) for c in tq.read_cases("mx_blocks.txt")]
    cases += [tq.test_e2m1_nibble_order, tq.test_bf16_matches_torch_cast,
              tq.test_e2m1_encode_matches_rounding_route]
    import torch
    cases += [lambda: tq.test_fp8_decode_table_matches_torch("e4m3", torch.float8_e4m3fn, 0x7e),
              lambda: tq.test_fp8_encode_matches_torch_in_range("e4m3", torch.float8_e4m3fn, 0x7e)]
    cases += [lambda: tdc.test_combine_identity_and_marked_experts(1, 64, 4),
              lambda: tdc.test_combine_identity_and_marked_experts(5, 8, 0)]
    cases += [lambda c=c: tqx.test_golden(c) for c in tq.read_cases("fp8_static_rows.txt")]
    cases += [lambda: tqx.test_fp8_token_exact_route(oracle.Q_FP8T_E4M3),
              lambda: tqx.test_fp8_group_exact_route(oracle.Q_FP8G_E4M3),
              tqx.test_int8_static_exact_route, tqx.test_smooth_scales_exact_route_fp8,
              lambda: tqx.test_dispatch_per_expert_scales_pick_the_entrys_expert(oracle.Q_INT8),
              lambda: tqx.test_masked_layout_matches_brute_force(0),
              lambda: tqx.test_masked_layout_matches_brute_force(1)]
    cases += [lambda s=s: ttl.test_random_small_against_brute_force(s) for s in range(6)]
    cases += [lambda: ttl.test_combine_through_rank_expert_stage_closed_form(2, 24, 4),
              ttl.test_reduced_weights_equal_original_for_valid_entries]
    cases += [lambda s=s: tfm.test_dispatch_bytes_brute_force(s) for s in range(4)]
    cases += [lambda: tdc.test_expert_dequant_rows_more_modes(oracle.Q_FP8G_E4M3),
              lambda: tdc.test_expert_dequant_rows_more_modes(oracle.Q_INT8_STATIC)]
    cases += [tnf.test_int8_infinite_element_zeroes_the_row, tnf.test_int8_subnormal_row_overflows_the_scale,
              tnf.test_int8_nan_elements_are_skipped_and_coded_zero, tnf.test_int8_all_nan_row_is_the_zero_row,
              tnf.test_int8_static_saturates_infinities_and_zeroes_nan, tnf.test_mx_block_with_infinity,
              tnf.test_mx_all_subnormal_block, tnf.test_mx_block_maximum_skips_nan,
              tnf.test_mx_block_of_nan_only_takes_the_smallest_exponent]
    cases += [trn.test_hand_worked_row, lambda: trn.test_constant_row(1e-3, 1e-6),
              lambda: trn.test_constant_row(0.75, 1e-6), lambda: trn.test_matches_torch_rms_norm_float64(1e-6),
              trn.test_f32_steps_hand_worked_exact,
              lambda: trn.test_f32_steps_match_an_independent_float32_route(256, 1e-6),
              lambda: trn.test_f32_steps_match_an_independent_float32_route(520, 0.5)]
    return cases


@contextlib.contextmanager
def use_library(path):
    saved = oracle._lib
    oracle._lib = oracle.load(path)
    try:
        yield
    finally:
        oracle._lib = saved


def test_unmutated_oracle_passes_the_pin_subset():
    for check in pins():
        check()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {name}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so, str(mutant_c), "-lm"], check=True)
    caught = 0
    with use_library(so):
        for check in pins():
            try:
                check()
            except AssertionError:
                caught += 1
                break
    assert caught, f"no pin caught the planted mistake {name}"
