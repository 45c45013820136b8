"""The pins are strong enough: each plausible mistake, planted in a private
copy of the oracle's C source, makes at least one pin fail.

Everything here runs on the CPU; the real oracle is never modified.
"""
import importlib.util
import os
import shutil

import numpy as np
import pytest

import test_oracle as pins

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("eps_outside_root", "sqrt(ms + (double)eps)", "(sqrt(ms) + (double)eps)"),
    ("mean_over_h_minus_1", "ss / (double)H", "ss / (double)(H - 1)"),
    ("sum_not_mean", "ss / (double)H", "ss"),
    ("weight_ignored", "w ? load_elem(fmt, w, j) : 1.0", "1.0"),
    ("weight_divides", "load_elem(fmt, x, r * H + j) * wj / denom",
     "load_elem(fmt, x, r * H + j) / wj / denom"),
    ("rope_sign_a", "o[ia] = a * c - b * s;", "o[ia] = a * c + b * s;"),
    ("rope_sign_b", "o[ib] = a * s + b * c;", "o[ib] = b * c - a * s;"),
    ("rope_cos_sin_swapped", "o[ib] = a * s + b * c;", "o[ib] = a * c + b * s;"),
    ("split_pairs_adjacent", "ia = h * head_dim + p;     ib = ia + P;",
     "ia = h * head_dim + 2 * p; ib = ia + 1;"),
    ("interleaved_pairs_split", "ia = h * head_dim + 2 * p; ib = ia + 1;",
     "ia = h * head_dim + p;     ib = ia + P;"),
    ("table_column_off_by_one", "cos_t[pos * P + p]", "cos_t[pos * P + (p + 1) % P]"),
    ("position_ignores_first_row", "(first_row + r) % table_rows", "r % table_rows"),
    ("position_fixed", "(first_row + r) % table_rows", "0"),
    ("round_ties_away", "frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) != 0.0)",
     "frac >= 0.5"),
    ("round_truncates", "if (frac > 0.5 || (frac == 0.5 && fmod(k, 2.0) != 0.0)) k += 1.0;",
     ""),
    ("subnormal_spacing", "if (e - 1 < emin) e = emin + 1;", "if (e < emin) e = emin;"),
    ("precision_plus_one_bit", "ldexp(1.0, e - prec)", "ldexp(1.0, e - prec - 1)"),
    ("adaln_scale_not_plus_one", "n[j] * (1.0 + sc) + sh", "n[j] * sc + sh"),
    ("adaln_shift_subtracted", "n[j] * (1.0 + sc) + sh", "n[j] * (1.0 + sc) - sh"),
    ("adaln_scale_shift_swapped", "n[j] * (1.0 + sc) + sh", "n[j] * (1.0 + sh) + sc"),
    ("adaln_cond_ignores_first_row", "(first_row + r) / rows_per_cond", "r / rows_per_cond"),
    ("adaln_cond_modulo", "(first_row + r) / rows_per_cond", "(first_row + r) % rows_per_cond"),
    ("add_norm_of_x", "normalise_row(fmt, h, r, w, H, eps, n);",
     "normalise_row(fmt, x, r, w, H, eps, n);"),
    ("add_subtracts", "load_elem(fmt, x, r * H + j) + load_elem(fmt, res, r * H + j)",
     "load_elem(fmt, x, r * H + j) - load_elem(fmt, res, r * H + j)"),
    ("gelu_cubic_coefficient", "0.044715 * x * x * x", "0.0447 * x * x * x"),
    ("gelu_exp_sign", "x / (1.0 + exp(-2.0 * z))", "x / (1.0 + exp(2.0 * z))"),
    ("gelu_half_scale", "sqrt(2.0 / M_PI)", "sqrt(1.0 / M_PI)"),
    ("geglu_halves_swapped",
     "const double v = value * gelu_tanh(gate);",
     "const double v = gate * gelu_tanh(value);"),
    ("gelu_stored_as_bf16", "        store_elem(fmt, y, i, v);\n", "        store_elem(FMT_BF16, y, i, v);\n"),
    ("geglu_gate_shifted", "load_elem(fmt, x, r * 2 * h + h + j)",
     "load_elem(fmt, x, r * 2 * h + h + (j + 1) % h)"),
    ("rope_tables_no_wrap", "rope_angles(s % (T * H * W), T, H, W, nt, nh, nw, theta, cos_out",
     "rope_angles(s, T, H, W, nt, nh, nw, theta, cos_out"),
    ("overflow_kept_finite", "if (r > ldexp(2.0 - ldexp(1.0, 1 - prec), emax)) r = INFINITY;", ""),
    ("f16_exponent_bias", "ldexp((double)(1024 + M), E - 25)", "ldexp((double)(1024 + M), E - 24)"),
    ("f16_subnormal_scale", "v = ldexp((double)M, -24)", "v = ldexp((double)M, -25)"),
    ("f16_round_10_bits", "round_binary(v, 11, -14, 15)", "round_binary(v, 10, -14, 15)"),
    ("f16_round_emin", "round_binary(v, 11, -14, 15)", "round_binary(v, 11, -15, 15)"),
    ("f16_round_emax", "round_binary(v, 11, -14, 15)", "round_binary(v, 11, -14, 16)"),
    ("f16_encode_mantissa", "(int)(m * 2048.0) - 1024", "(int)(m * 2048.0) - 1023"),
    ("f32_round_23_bits", "round_binary(v, 24, -126, 127)", "round_binary(v, 23, -126, 127)"),
    ("f32_round_emin", "round_binary(v, 24, -126, 127)", "round_binary(v, 24, -125, 127)"),
    ("f16_read_as_bf16", "return fmt == FMT_F16 ? widen_f16(b) : widen_bf16(b);",
     "return widen_bf16(b);"),
    ("rpos_exponent_doubled", "pow(theta, -(double)k / (double)n[axis])",
     "pow(theta, -2.0 * (double)k / (double)n[axis])"),
    ("rpos_axes_reversed", "{s / (H * W), (s / W) % H, s % W}", "{s % W, (s / W) % H, s / (H * W)}"),
    ("rpos_w_h_swapped", "{s / (H * W), (s / W) % H, s % W}", "{s / (H * W), s % W, (s / W) % H}"),
    ("rpos_ignores_first_row", "rope_angles((first_row + r) % (T * H * W)",
     "rope_angles((r) % (T * H * W)"),
    ("rpos_sign_a", "const double ya = a * c[p] - b * sn[p];", "const double ya = a * c[p] + b * sn[p];"),
    ("rpos_sign_b", "const double yb = a * sn[p] + b * c[p];", "const double yb = b * c[p] - a * sn[p];"),
    ("rpos_position_plus_one", "const double ang = (double)coord[axis] *",
     "const double ang = (double)(coord[axis] + 1) *"),
    ("f32_stored_as_f16", "if (fmt == FMT_F32) ((float*)p)[i] = round_to_f32(v);",
     "if (fmt == FMT_F32) ((float*)p)[i] = (float)widen_f16(round_to_f16(v));"),
]


def _pin_calls():
    hand = {c["name"]: c for c in pins._parse_golden()}
    calls = [
        ("widen", pins.test_widen_all_patterns, ()),
        ("identity", pins.test_round_identity_all_patterns, ()),
        ("midpoints", pins.test_round_midpoints_ties_to_even, ()),
        ("specials", pins.test_round_special_values, ()),
        ("direct", pins.test_round_direct_not_through_binary32, ()),
        ("eps_order", pins.test_eps_first_order, ()),
        ("unit_rms", pins.test_unit_rms_closed_form, (24,)),
        ("scale", pins.test_scale_invariance_exact, (1,)),
        ("torch", pins.test_matches_torch_rms_norm_fp64, ()),
        ("threaded", pins.test_threaded_rows_identical, ()),
        ("identity0", pins.test_rope_identity_at_angle_zero, (0,)),
        ("quarter0", pins.test_rope_quarter_and_half_turn, (0,)),
        ("quarter1", pins.test_rope_quarter_and_half_turn, (1,)),
        ("pairnorm0", pins.test_rope_preserves_pair_norm, (0,)),
        ("pairnorm1", pins.test_rope_preserves_pair_norm, (1,)),
        ("perm", pins.test_split_half_is_permuted_interleaved, ()),
        ("position", pins.test_rope_position_is_row_mod_table_rows, ()),
    ]
    for name, case in hand.items():
        calls.append(("hand_" + name, pins.test_hand_cases, (case,)))
    for case in pins._parse_adaln():
        calls.append(("adaln_hand_" + case["name"], pins.test_adaln_hand_cases, (case,)))
    calls += [
        ("adaln_zero", pins.test_adaln_zero_modulation_is_rms_norm, ()),
        ("adaln_minus1", pins.test_adaln_scale_minus_one_gives_shift, ()),
        ("adaln_affine", pins.test_adaln_is_affine_in_scale_and_shift, ()),
        ("adaln_cond", pins.test_adaln_conditioning_rows, ()),
        ("add_hand", pins.test_add_norm_hand_cases, ()),
        ("add_zero", pins.test_add_norm_zero_residual_is_rms_norm, ()),
        ("add_commute", pins.test_add_norm_commutes_and_cancels, ()),
        ("add_rounded", pins.test_add_norm_h_is_the_rounded_sum, ()),
        ("gelu_odd", pins.test_gelu_is_x_sigma_identity, ()),
        ("gelu_torch", pins.test_gelu_matches_tanh_form_and_torch, ()),
        ("gelu_tails", pins.test_gelu_tails, ()),
        ("geglu", pins.test_geglu_value_times_gelu_of_gate, ()),
        ("gelu_fmt_f16", pins.test_gelu_formats_match_torch_and_numpy_rounding, (np.float16,)),
        ("gelu_fmt_f32", pins.test_gelu_formats_match_torch_and_numpy_rounding, (np.float32,)),
        ("gelu_tails_f32", pins.test_gelu_formats_tails_and_specials, (np.float32,)),
        ("geglu_fmt_f16", pins.test_geglu_formats_value_times_gelu_of_gate, (np.float16,)),
        ("geglu_fmt_f32", pins.test_geglu_formats_value_times_gelu_of_gate, (np.float32,)),
        ("f16_widen", pins.test_f16_widen_all_patterns, ()),
        ("f16_midpoints", pins.test_f16_round_identity_and_midpoints, ()),
        ("f16_specials", pins.test_f16_round_specials, ()),
        ("f16_numpy", pins.test_f16_round_matches_numpy_conversion, ()),
        ("f32_hw", pins.test_f32_round_matches_hardware_conversion, ()),
        ("fmt_shared_f16", pins.test_formats_share_the_arithmetic, (np.float16,)),
        ("fmt_shared_f32", pins.test_formats_share_the_arithmetic, (np.float32,)),
        ("fmt_torch_f16", pins.test_formats_match_torch_rms_norm_fp64, (np.float16,)),
        ("fmt_torch_f32", pins.test_formats_match_torch_rms_norm_fp64, (np.float32,)),
        ("rpos_identity", pins.test_rope_positions_identity_at_token_zero, ()),
        ("rpos_closed0", pins.test_rope_positions_closed_form_frequencies, (0,)),
        ("rpos_closed1", pins.test_rope_positions_closed_form_frequencies, (1,)),
        ("rpos_3axis", pins.test_rope_positions_three_axis_coordinates, ()),
        ("rpos_additive", pins.test_rope_positions_angle_is_additive_in_position, ()),
        ("rpos_norms", pins.test_rope_positions_norms_wrap_and_permutation, ()),
        ("rtab_recipe", pins.test_rope_tables_are_the_fused_forms_table_recipe, ()),
        ("rtab_wrap", pins.test_rope_tables_identity_wrap_and_norms, ()),
    ]
    return calls


def _load_mutant(tmp_path, name, old, new):
    d = tmp_path / f"oracle_{name}"
    d.mkdir()
    shutil.copy(os.path.join(ORACLE_DIR, "__init__.py"), d / "__init__.py")
    src = open(os.path.join(ORACLE_DIR, "oracle.c")).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    (d / "oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(
        f"oracle_{name}", d / "__init__.py", submodule_search_locations=[str(d)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def test_unmutated_copy_passes_every_pin(tmp_path):
    mod = _load_mutant(tmp_path, "none", "oracle", "oracle")
    for _, fn, args in _pin_calls():
        fn(mod, *args)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    mod = _load_mutant(tmp_path, name, old, new)
    caught = []
    for pin, fn, args in _pin_calls():
        try:
            fn(mod, *args)
        except (AssertionError, RuntimeError, ValueError, MemoryError):
            caught.append(pin)
    assert caught, f"no pin caught mutant {name}"
