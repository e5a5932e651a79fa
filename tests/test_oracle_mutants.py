"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that at least one pin in test_oracle.py catches each of them. This is what
makes the pins trustworthy: a dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the oracle must fail something. Every planted
mistake keeps its reads and writes inside the arrays (one that wrote outside
would corrupt this process instead of failing a pin)."""
import os
import subprocess

import pytest

import oracle
import test_oracle as pins
import test_oracle_fp8 as fp8_pins
import test_oracle_multi as multi_pins
import test_oracle_multi_rope as multi_rope_pins
import test_oracle_multi_fp8 as multi_fp8_pins
import test_oracle_rope as rope_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("drop_sink", "double den = isinf(sigma) && sigma < 0 ? 0.0 : exp(sigma - M);",
     "double den = 0.0;"),
    ("sink_scaled", "const double sigma = pr->sinks ? (double)pr->sinks[h] : -INFINITY;",
     "const double sigma = pr->sinks ? pr->scale * (double)pr->sinks[h] : -INFINITY;"),
    ("gqa_modulo", "const int g = h / G;", "const int g = h % pr->Hkv;"),
    ("window_one_short", "const int lo = (W > 0 && L - W > 0) ? L - W : 0;",
     "const int lo = (W > 0 && L - W + 1 > 0) ? L - W + 1 : 0;"),
    ("window_one_long", "const int lo = (W > 0 && L - W > 0) ? L - W : 0;",
     "const int lo = (W > 0 && L - W - 1 > 0) ? L - W - 1 : 0;"),
    ("ignore_new_token", "if (j == L - 1 && pr->k_new != NULL && pr->kind != LAYOUT_CONTIG) {",
     "if (0) {"),
    ("page_slot_swapped",
     "return base + (((size_t)page * Hkv + g) * pr->P + (size_t)(j % pr->P)) * D;",
     "return base + (((size_t)page * Hkv + g) * pr->P + (size_t)((j / pr->P) % pr->P)) * D;"),
    ("page_head_token_swapped",
     "return base + (((size_t)page * Hkv + g) * pr->P + (size_t)(j % pr->P)) * D;",
     "return base + (((size_t)page * pr->P + (size_t)(j % pr->P)) * Hkv + g) * D;"),
    ("ring_cell_shift", "int cell = j % pr->window;", "int cell = (j + 1) % pr->window;"),
    ("no_scale", "s[i] = pr->scale * dot;", "s[i] = dot;"),
    ("exp_sign", "double w = exp(s[i] - M);", "double w = exp(M - s[i]);"),
    ("value_is_key", "const uint16_t *vrow = token_row(pr, b, g, lo + i, 1);",
     "const uint16_t *vrow = token_row(pr, b, g, lo + i, 0);"),
    ("q_transposed", "const uint16_t *qrow = pr->q + ((size_t)b * pr->Hq + h) * D;",
     "const uint16_t *qrow = pr->q + ((size_t)h * pr->B + b) * D;"),
    ("rope_sign", "out[i] = x1 * (double)c[i] - x2 * (double)sn[i];",
     "out[i] = x1 * (double)c[i] + x2 * (double)sn[i];"),
    ("rope_mirror_pairs", "const double x1 = bf16_to_f64(x[i]), x2 = bf16_to_f64(x[i + h]);",
     "const double x1 = bf16_to_f64(x[i]), x2 = bf16_to_f64(x[D - 1 - i]);"),
    ("rope_q_position", "            const size_t row = (size_t)(L - 1) * h;\n            rope_row_f64",
     "            const size_t row = (size_t)(L % max_position) * h;\n            rope_row_f64"),
    ("rope_q_unrotated", "pr.q = q; pr.q64 = q64; pr.k_new = krot; pr.v_new = v_new; pr.k_src = k_cache; "
     "pr.v_src = v_cache;\n        pr.block_table",
     "pr.q = q; pr.q64 = NULL; pr.k_new = krot; pr.v_new = v_new; pr.k_src = k_cache; "
     "pr.v_src = v_cache;\n        pr.block_table"),
    ("rope_key_truncated", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0u;"),
    ("e4m3_bias", "ldexp(1.0 + m / 8.0, e - 7);", "ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3_ties_away", "if (rem > step / 2 || (rem == step / 2 && fmod(k, 2.0) == 1.0)) k += 1.0;",
     "if (rem >= step / 2) k += 1.0;"),
    ("fp8_vt_stride", "v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d * P + slot]) * sv;",
     "v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d + slot]) * sv;"),
    ("fp8_no_vscale", "v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d * P + slot]) * sv;",
     "v[d] = e4m3_decode(blk[(size_t)P * D + (size_t)d * P + slot]);"),
    ("fp8_scales_swapped", "const double sk = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)slot);",
     "const double sk = f32_at(blk + 2 * (size_t)P * D + 4 * (size_t)(P + slot));"),
    ("fp8_ring_slot", "*slot = cell % P;\n    return ((long long)b * Hkv + g) * (W / P) + cell / P;",
     "*slot = (cell + 1) % P;\n    return ((long long)b * Hkv + g) * (W / P) + cell / P;"),
    ("fp8_scale_rule", "amax / 448.0f", "amax / 447.0f"),
    ("multi_not_causal_self", "const int cnt = p - lo + 1;", "const int cnt = p - lo;"),
    ("multi_position_shift", "const int p = L - n + t;", "const int p = L - n + t - 1;"),
    ("multi_new_token_index", "const int t = j - base;", "const int t = (j - base + 1) % pr->T;"),
    ("multi_window_one_long", "const int lo = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;",
     "const int lo = (W > 0 && p - W > 0) ? p - W : 0;"),
    ("multi_q_lens_ignored", "static int q_count(const int32_t *q_lens, int T, int b) { return q_lens ? q_lens[b] : T; }",
     "static int q_count(const int32_t *q_lens, int T, int b) { (void)q_lens; (void)b; return T; }"),
    ("multi_append_shift", "const int pos = L - n + t;", "const int pos = L - n + t + 1;"),
    ("multi_q_token_stride", "const size_t qoff = (((size_t)b * pr->T + t) * pr->Hq + h) * D;",
     "const size_t qoff = (((size_t)t * pr->B + b) * pr->Hq + h) * D;"),
    ("multi_rope_position", "const int p = L - n + t;\n            if (active && p >= max_position)",
     "const int p = L - 1;\n            if (active && p >= max_position)"),
    ("multi_fp8_new_token_from_cache",
     "const int L = pr->seq_lens[b], n = q_count(pr->q_lens, pr->T, b), base = L - n, D = pr->D, P = pr->P;\n    if (j >= base) {",
     "const int L = pr->seq_lens[b], n = q_count(pr->q_lens, pr->T, b), base = L - n, D = pr->D, P = pr->P;\n    if (j > base) {"),
    ("multi_fp8_append_order",
     "const int st = put8(ring, blocks, b, g, L - n + t, k_new + src",
     "const int st = put8(ring, blocks, b, g, L - 1 - t, k_new + src"),
    ("append_wrong_cell",
     "size_t dst = (((size_t)page * Hkv + g) * page_size + (size_t)(p % page_size)) * D;",
     "size_t dst = (((size_t)page * Hkv + g) * page_size + (size_t)(L % page_size)) * D;"),
]

PIN_CALLS = [
    lambda: pins.test_brute_force_matches_all_layouts(11, 2, 4, 2, 8, [5, 17], 0),
    lambda: pins.test_brute_force_matches_all_layouts(12, 3, 6, 3, 4, [1, 16, 33], 7),
    lambda: pins.test_no_sink_equals_torch_sdpa_fp64(9),
    pins.test_single_token_is_sigmoid_weighted_value,
    pins.test_zero_query_is_windowed_mean_with_sink,
    pins.test_equal_keys_equal_values_closed_form,
    pins.test_window_at_or_beyond_length_equals_full,
    lambda: pins.test_ring_paged_contig_agree(13),
    pins.test_gqa_equals_mha_on_repeated_kv,
    pins.test_append_is_bit_exact_and_touches_only_target_cells,
    pins.test_hand_worked_example,
    rope_pins.test_identity_tables_change_nothing,
    rope_pins.test_quarter_turn_is_a_signed_half_swap,
    rope_pins.test_position_zero_is_the_identity,
    rope_pins.test_rotation_keeps_norms,
    rope_pins.test_stored_key_rounding_is_fp32_then_bf16_nearest_even,
    lambda: rope_pins.test_attention_depends_only_on_relative_positions(37),
    fp8_pins.test_decode_every_code_like_torch,
    fp8_pins.test_encode_rounds_to_nearest_even_like_torch,
    fp8_pins.test_quantisation_rule_closed_form,
    lambda: fp8_pins.test_fp8_equals_bf16_on_values_exact_in_both(0),
    fp8_pins.test_paged_and_ring_agree_and_append_is_fused,
    fp8_pins.test_block_layout_byte_by_byte,
    lambda: multi_pins.test_multi_brute_force_paged(0, 3),
    lambda: multi_pins.test_multi_brute_force_ring(1, 16),
    multi_pins.test_multi_equals_torch_sdpa_with_causal_mask,
    multi_pins.test_one_token_equals_the_single_token_step,
    multi_pins.test_rows_beyond_q_lens_and_inactive_slots_are_zero,
    lambda: multi_pins.test_append_is_bit_exact_and_touches_only_the_new_cells(True),
    lambda: multi_pins.test_append_is_bit_exact_and_touches_only_the_new_cells(False),
    multi_rope_pins.test_identity_tables_give_the_plain_step,
    lambda: multi_rope_pins.test_one_new_token_is_the_one_token_step(0),
    multi_rope_pins.test_each_token_is_rotated_at_its_own_position,
    multi_rope_pins.test_rotated_rows_round_as_fp32_then_bf16,
    lambda: multi_fp8_pins.test_one_new_token_is_the_one_token_fp8_step(0),
    lambda: multi_fp8_pins.test_exact_values_give_the_bf16_step(0),
    lambda: multi_fp8_pins.test_append_equals_quantising_the_whole_history(False),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutant {name}: anchor text not found in oracle.c"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"lib{name}.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", str(c_path),
                    "-o", str(so_path), "-lm"], check=True)
    return str(so_path)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    so = _build_mutant(tmp_path, name, old, new)
    prev = oracle.load_library(so)
    caught = []
    try:
        for call in PIN_CALLS:
            try:
                call()
            except (AssertionError, ValueError):
                caught.append(call)
    finally:
        oracle.restore_library(prev)
    assert caught, f"no pin caught the planted mistake {name!r}"
