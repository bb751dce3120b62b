"""The oracle's pins are sensitive, not only present.

Each case plants one plausible mistake in a copy of the oracle's C source: a
dropped term, a wrong sign, index or bound, a swapped operand, a reversed
order. The copy is built with gcc in a temporary directory and loaded in place
of the oracle, and at least one of the pins written for that step of the
method must fail against it. The oracle itself is never modified; the copies
exist only inside this test, on the CPU.

Every planted mistake keeps each memory access inside its buffer (indices stay
within the block, the table row or the allocated token list), so a mutant can
compute wrong values but cannot crash the test process.
"""

import os

import pytest

import oracle
import test_oracle_fp8_block_pins as FB
import test_oracle_fp8_pins as F
import test_oracle_multi_pins as M
import test_oracle_pins as P


def _pin(mod, test_name, **kw):
    return (mod, test_name, kw)


SDPA_G3 = _pin(P, "test_dense_matches_library_sdpa", B=2, Hq=6, Hkv=2, D=8, BS=4, ctx=[3, 13],
               permute=True)
SDPA_G7 = _pin(P, "test_dense_matches_library_sdpa", B=2, Hq=28, Hkv=4, D=16, BS=16, ctx=[16, 17],
               permute=False)

# (id, text in oracle.c, replacement, which occurrence (1-based), pins expected to catch it)
MUTANTS = [
    # ReshapeAndCache: the slot -> (block, offset) decomposition and the operands
    ("reshape_offset", "const int64_t block_offset = slot % BS;",
     "const int64_t block_offset = (slot + 1) % BS;", 1,
     [_pin(P, "test_reshape_slot_math_golden")]),
    ("reshape_value_from_key", "value_cache[dst + e] = value[t * row + e];",
     "value_cache[dst + e] = key[t * row + e];", 1,
     [_pin(P, "test_reshape_slot_math_golden")]),
    ("reshape_fp8_offset", "const int64_t block_offset = slot % BS;",
     "const int64_t block_offset = (slot + 1) % BS;", 2,
     [_pin(F, "test_fp8_write_quantises_each_element")]),
    # dense attention: scale, GQA head mapping, context bound, normalisation
    ("score_scale_dropped", "s[i] = scale * dot;", "s[i] = dot;", 1,
     [SDPA_G3, SDPA_G7, _pin(P, "test_dense_closed_forms")]),
    ("gqa_head_interleaved", "const int kvh = (int)(h / G);", "const int kvh = (int)(h % Hkv);", 1,
     [SDPA_G3, SDPA_G7]),
    ("context_off_by_one", "for (int64_t t = 0; t < ctx; ++t)", "for (int64_t t = 0; t + 1 < ctx; ++t)", 1,
     [SDPA_G3, SDPA_G7]),
    ("softmax_not_normalised", "out[d] /= l;", "out[d] /= 1.0;", 1,
     [SDPA_G3, SDPA_G7, _pin(P, "test_dense_closed_forms")]),
    # online softmax and the split-KV combine
    ("online_no_rescale", "const double alpha = exp(m - m_new);", "const double alpha = 1.0;", 1,
     [_pin(P, "test_online_softmax_equals_two_pass", chunk=1),
      _pin(P, "test_online_softmax_equals_two_pass", chunk=3)]),
    ("split_equal_weights", "const double w = exp(lse[sp] - mstar);", "const double w = 1.0;", 1,
     [_pin(P, "test_split_combine_equals_two_pass", splits=3),
      _pin(P, "test_split_combine_equals_two_pass", splits=7)]),
    ("split_lse_without_sum", "lse[sp] = m + log(l);", "lse[sp] = m;", 1,
     [_pin(P, "test_split_combine_equals_two_pass", splits=3),
      _pin(P, "test_split_combine_equals_two_pass", splits=7)]),
    # sparse attention: tokens of a selected block past the context
    ("sparse_tail_unmasked", "t < (j + 1) * BS && t < ctx; ++t)", "t < (j + 1) * BS; ++t)", 1,
     [_pin(P, "test_sparse_matches_sdpa_on_selected_tokens"),
      _pin(P, "test_sparse_all_blocks_equals_dense")]),
    # Quest metadata
    ("rebuild_tail_included", "const int64_t t_end = (j + 1) * BS < ctx ? (j + 1) * BS : ctx;",
     "const int64_t t_end = (j + 1) * BS;", 1,
     [_pin(P, "test_rebuild_meta_is_elementwise_min_max")]),
    ("update_never_resets", "reset = 1;", "reset = 0;", 1,
     [_pin(P, "test_update_meta_brute_force_and_order_independent"),
      _pin(P, "test_incremental_decode_meta_equals_rebuild")]),
    ("update_min_compare_flipped", "if (bf16_order_key(k[e]) < bf16_order_key(lo[e]))",
     "if (bf16_order_key(k[e]) > bf16_order_key(lo[e]))", 1,
     [_pin(P, "test_update_meta_brute_force_and_order_independent"),
      _pin(P, "test_incremental_decode_meta_equals_rebuild")]),
    ("rebuild_fp8_tail_included", "const int64_t t_end = (j + 1) * BS < ctx ? (j + 1) * BS : ctx;",
     "const int64_t t_end = (j + 1) * BS;", 2,
     [_pin(F, "test_fp8_rebuild_meta_is_numeric_min_max")]),
    ("update_fp8_never_resets", "reset = 1;", "reset = 0;", 2,
     [_pin(F, "test_fp8_incremental_meta_equals_rebuild")]),
    ("fp8_order_negatives_reversed", "(uint8_t)(~c & 0x7Fu)", "(uint8_t)(c & 0x7Fu)", 1,
     [_pin(F, "test_fp8_rebuild_meta_is_numeric_min_max"),
      _pin(F, "test_fp8_incremental_meta_equals_rebuild")]),
    # Quest block score
    ("score_max_uses_min", "P[d] * meta_f32(kmax, kmax8, base + d)", "P[d] * meta_f32(kmin, kmin8, base + d)", 1,
     [_pin(P, "test_quest_score_exact_on_integers"), _pin(P, "test_quest_bound_dominates_true_max")]),
    ("score_negative_part_sign", "nn = nn + (v < 0.0f ? v : 0.0f);", "nn = nn + (v < 0.0f ? -v : 0.0f);", 1,
     [_pin(P, "test_quest_score_exact_on_integers"), _pin(P, "test_quest_bound_dominates_true_max")]),
    ("score_last_reduction_step_dropped", "for (int off = 16; off >= 1; off >>= 1)",
     "for (int off = 16; off > 1; off >>= 1)", 1,
     [_pin(P, "test_quest_score_exact_on_integers"),
      _pin(P, "test_quest_score_kernel_order_within_fp32_bound", name="tiny")]),
    ("score_block_past_context_kept", "if (j >= nblk) {", "if (j > nblk) {", 1,
     [_pin(P, "test_quest_score_exact_on_integers")]),
    # Quest block score, plain fp64 form
    ("plain_score_max_uses_min", "const double x = qv * lo, y = qv * hi;",
     "const double x = qv * lo, y = qv * lo;", 1,
     [_pin(P, "test_quest_score_exact_on_integers"), _pin(P, "test_quest_score_sign_closed_forms")]),
    ("plain_score_min_of_products", "s += x > y ? x : y;", "s += x < y ? x : y;", 1,
     [_pin(P, "test_quest_score_exact_on_integers"), _pin(P, "test_quest_bound_dominates_true_max")]),
    ("plain_score_group_interleaved", "const int64_t h = (int64_t)kvh * G + g;",
     "const int64_t h = (int64_t)g * Hkv + kvh;", 1,
     [_pin(P, "test_quest_score_group_mapping"), _pin(P, "test_quest_score_identical_tokens_is_group_dot_product")]),
    ("plain_score_block_past_context_kept",
     "const int64_t p = j < nblk ? block_tables[(int64_t)b * MBS + j] : -1;",
     "const int64_t p = j <= nblk ? block_tables[(int64_t)b * MBS + j] : -1;", 1,
     [_pin(P, "test_quest_score_exact_on_integers")]),
    ("plain_abs_sum_min_side_only", "const double m = fabs(lo) > fabs(hi) ? fabs(lo) : fabs(hi);",
     "const double m = fabs(lo);", 1,
     [_pin(P, "test_quest_score_abs_sum")]),
    # Quest top-K
    ("topk_f64_raw_bits_order", "return (u >> 63) ? ~u : (u | (1ull << 63));", "return u;", 1,
     [_pin(P, "test_topk_f64_brute_force_with_ties_and_signs")]),
    ("topk_lowest_first", "return x->key > y->key ? -1 : 1;", "return x->key < y->key ? -1 : 1;", 1,
     [_pin(P, "test_topk_brute_force_with_ties"), _pin(P, "test_topk_tie_goes_to_lower_index")]),
    ("topk_tie_to_higher_index", "return x->j < y->j ? -1 : (x->j > y->j);",
     "return x->j > y->j ? -1 : (x->j < y->j);", 1,
     [_pin(P, "test_topk_brute_force_with_ties"), _pin(P, "test_topk_tie_goes_to_lower_index")]),
    ("topk_output_descending", "return x < y ? -1 : (x > y);", "return x > y ? -1 : (x < y);", 1,
     [_pin(P, "test_topk_brute_force_with_ties"), _pin(P, "test_topk_fewer_blocks_than_k_selects_all")]),
    # E4M3 codec and the 8-bit cache
    ("e4m3_subnormal_exponent", "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", 1,
     [_pin(F, "test_e4m3_format_constants"), _pin(F, "test_e4m3_decode_matches_library_on_every_code")]),
    ("e4m3_ties_to_odd", "fmod(r, 2.0) == 1.0", "fmod(r, 2.0) == 0.0", 1,
     [_pin(F, "test_e4m3_encode_is_brute_force_nearest_even"),
      _pin(F, "test_e4m3_encode_matches_library_in_range")]),
    ("e4m3_saturation_loses_sign", "return sgn | 0x7E;", "return 0x7E;", 1,
     [_pin(F, "test_e4m3_encode_saturates_and_keeps_nan")]),
    ("fp8_quantise_multiplies", "const float y = bf16_f32(x) / scale;", "const float y = bf16_f32(x) * scale;", 1,
     [_pin(F, "test_fp8_write_quantises_each_element")]),
    ("fp8_dequantise_without_scale", "return oracle_e4m3_decode(c->e4m3[idx]) * sc;",
     "return oracle_e4m3_decode(c->e4m3[idx]);", 1,
     [_pin(F, "test_fp8_attention_brute_force_any_scale")]),
    ("fp8_v_layout_natural_order", "return 4 * ((o & 7) >> 1) + 2 * (o >> 3) + (o & 1);", "return o;", 1,
     [_pin(F, "test_fp8_write_quantises_each_element")]),
    # the 8-bit cache with per-block power-of-two scales
    ("block_fit_pow2_max", "while (a > ldexp(448.0, e))", "while (a > ldexp(256.0, e))", 1,
     [_pin(FB, "test_hand_worked_example"), _pin(FB, "test_first_write_scale_and_codes")]),
    ("block_old_rows_not_rescaled", "*kc = rescale_code(*kc, eko - ekn);", "*kc = rescale_code(*kc, 0);", 1,
     [_pin(FB, "test_hand_worked_example"), _pin(FB, "test_incremental_equals_from_scratch")]),
    ("block_v_rows_use_k_shift", "*vc = rescale_code(*vc, evo - evn);", "*vc = rescale_code(*vc, eko - ekn);",
     1, [_pin(FB, "test_incremental_equals_from_scratch")]),
    ("block_meta_not_rescaled", "kmin[m] = rescale_code(kmin[m], eko - ekn);", "kmin[m] = kmin[m];", 1,
     [_pin(FB, "test_incremental_equals_from_scratch")]),
    ("block_restart_keeps_scale", "if (!reset && s > 0.0f) {", "if (s > 0.0f) {", 1,
     [_pin(FB, "test_restart_resets_scale_and_keeps_other_rows")]),
    ("block_kernel_order_score_unscaled", "srow[j] = k_bscale ? c[0] * k_bscale[p * Hkv + kvh] : c[0];",
     "srow[j] = c[0];", 1, [_pin(FB, "test_block_scores_equal_bf16_scores_on_scaled_meta")]),
    ("block_plain_score_unscaled", "s *= (double)k_bscale[p * Hkv + kvh];", "s *= 1.0;", 1,
     [_pin(FB, "test_block_scores_equal_bf16_scores_on_scaled_meta"),
      _pin(FB, "test_block_score_bounds_every_token")]),
    ("block_attention_head_scale", "c->scale[c->per_block ? p * c->Hkv + kvh : kvh]", "c->scale[kvh]", 1,
     [_pin(FB, "test_block_attention_equals_bf16_attention_on_exact_values")]),
    # multi-row queries: right-aligned causal mask and head mapping
    ("multi_mask_excludes_self", "int64_t lim = ctx - q_len + (row - cu_seqlens_q[b]) + 1;",
     "int64_t lim = ctx - q_len + (row - cu_seqlens_q[b]);", 1,
     [_pin(M, "test_multi_rows_match_sdpa_with_tril_mask")]),
    ("multi_gqa_head_interleaved", "n, (int)(h / G), Hkv", "n, (int)(h % Hkv), Hkv", 1,
     [_pin(M, "test_multi_rows_match_sdpa_with_tril_mask")]),
]


def _replace_nth(text: str, old: str, new: str, nth: int) -> str:
    at = -1
    for _ in range(nth):
        at = text.find(old, at + 1)
        assert at >= 0, f"mutation site not found: {old!r} (occurrence {nth})"
    return text[:at] + new + text[at + len(old):]


def _failing_pins(tmp_path, monkeypatch, mid, old, new, nth, pins):
    """Build oracle.c with one edit, load it in place of the oracle and return
    the names of the pins that fail against it."""
    with open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")) as f:
        src = f.read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    path = tmp_path / f"oracle_{mid}.c"
    path.write_text(mutated)
    lib = oracle.load(oracle.compile_source(str(path), str(tmp_path / f"liboracle_{mid}.so")))
    monkeypatch.setattr(oracle, "_lib", lib)
    failing = []
    for mod, name, kw in pins:
        try:
            getattr(mod, name)(oracle_lib=oracle, **kw)
        except AssertionError:
            failing.append(name)
    return failing


@pytest.mark.parametrize("mid,old,new,nth,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, mid, old, new, nth, pins):
    failing = _failing_pins(tmp_path, monkeypatch, mid, old, new, nth, pins)
    assert failing, f"no pin fails with the planted mistake {mid!r}: {old!r} -> {new!r}"


def test_equivalent_rewrite_passes_every_pin(tmp_path, monkeypatch):
    """Control: an edit that changes no result (IEEE multiplication commutes
    exactly) must fail no pin, so a caught mutant is caught by its mistake."""
    pins = [SDPA_G3, SDPA_G7, _pin(P, "test_dense_closed_forms"),
            _pin(P, "test_split_combine_equals_two_pass", splits=3),
            _pin(P, "test_sparse_matches_sdpa_on_selected_tokens")]
    failing = _failing_pins(tmp_path, monkeypatch, "control", "s[i] = scale * dot;",
                            "s[i] = dot * scale;", 1, pins)
    assert failing == []
