"""Negative controls: plant plausible mistakes in a copy of the oracle and
check that the pins catch every one of them.

Each mutation is a textual edit of kvq_oracle.c, compiled with the oracle's
own flags into a temporary library; the pins (the same test functions that
run against the real oracle) must fail on it.  This is the check that the
pins are strong enough to catch a dropped term, a wrong sign or index, or a
transposed operand, in the spirit of the negative control described in
#711 kv: --kv k8v4 streams with --kv-resident, "Tests".
"""
import numpy as np
import pytest

import oracle
from tests import test_oracle_attention as att
from tests import test_oracle_chunk as chk
from tests import test_oracle_k8v4 as k84
from tests import test_oracle_persist as per
from tests import test_oracle_fp16 as f16
from tests import test_oracle_quant as qt

F16, Q8 = oracle.FMT_F16, oracle.FMT_Q8

MUTATIONS = {
    "round_half_away": ("float rr = rintf(ratio);", "float rr = roundf(ratio);"),
    "times_reciprocal": ("const float ratio = xg[i] / sf;",
                         "const float ratio = xg[i] * (1.0f / sf);"),
    "unrounded_scale": ("const float ratio = xg[i] / sf;", "const float ratio = xg[i] / t;"),
    "max_not_abs": ("const float ax = fabsf(xg[i]);", "const float ax = xg[i];"),
    "clamp_128": ("if (rr < -127.0f)\n                        rr = -127.0f;",
                  "if (rr < -128.0f)\n                        rr = -128.0f;"),
    "fp16_ties_away": ("const double r = nearbyint(n);", "const double r = floor(n + 0.5);"),
    "fp16_subnormal_edge": ("if (a < ldexp(1.0, -14)) {", "if (a < ldexp(1.0, -15)) {"),
    "gqa_modulo": ("const int kvh = h / G;", "const int kvh = h % n_kv;"),
    "causal_drop_diagonal": ("const int last = L - W + w; /* last visible cell */",
                             "const int last = L - W + w - 1;"),
    "no_softmax_scale": ("z[c] = (double)sm_scale * dot;", "z[c] = dot;"),
    "scale_group_index": ("+ d / KVO_GROUP];", "+ 0];"),
    "slot_off_by_one": ("const int slot = pos % block_size;",
                        "const int slot = (pos + 1) % block_size;"),
    "k_reads_v": ("dot += (double)qv[d] * dequant(fmt, hd, k_data, k_scales, row, d);",
                  "dot += (double)qv[d] * dequant(fmt, hd, v_data, v_scales, row, d);"),
    "no_normalisation": ("o[d] /= den;", "o[d] /= (den + 1.0);"),
    "compact_k_from_v": ("(float)dequant(fmt, hd, k_data, k_scales, row, d));",
                         "(float)dequant(fmt, hd, v_data, v_scales, row, d));"),
    "chunk_causal_drop_diagonal": ("const int last = P - T + t; /* last visible cell */",
                                   "const int last = P - T + t - 1;"),
    "chunk_causal_from_start": ("const int last = P - T + t; /* last visible cell */",
                                "const int last = t;"),
    "chunk_gqa_modulo": ("const int src_head = h / G;", "const int src_head = h % n_kv;"),
    "chunk_no_softmax_scale": ("z[c] = dot * (double)sm_scale;", "z[c] = dot;"),
    "chunk_k_reads_v": ("const uint16_t *kr = k16 +", "const uint16_t *kr = v16 +"),
    "chunk_no_normalisation": ("o[d] = o[d] / den;", "o[d] = o[d] / (den + 1.0);"),
    "gather_v_from_k": ("memcpy((char *)codes_v + dst * vb, (const char *)v_data +",
                        "memcpy((char *)codes_v + dst * vb, (const char *)k_data +"),
    "gather_k_scales_from_v": ("scales_k[dst * kng + gi] = k_scales[(size_t)row * kng + gi];",
                               "scales_k[dst * kng + gi] = v_scales[(size_t)row * kng + gi];"),
    "persist_slot_off_by_one": ("return ((int64_t)blk * n_kv + kvh) * block_size + pos % block_size;",
                                "return ((int64_t)blk * n_kv + kvh) * block_size + (pos + 1) % block_size;"),
    "scatter_drops_v_scales": ("v_scales[(size_t)row * vng + gi] = scales_v[src * vng + gi];",
                               "v_scales[(size_t)row * vng + gi] = scales_k[src * vng + gi];"),
    # K8V4
    "q4_max_last_on_ties": ("if (fabsf(y[i]) > fabsf(m))", "if (fabsf(y[i]) >= fabsf(m))"),
    "q4_positive_scale": ("kvo_fp16_from_float(m / -8.0f)", "kvo_fp16_from_float(m / 8.0f)"),
    "q4_scale_over_7": ("kvo_fp16_from_float(m / -8.0f)", "kvo_fp16_from_float(m / -7.0f)"),
    "q4_round_half_away": ("float r = rintf(y[i + e] / d);", "float r = roundf(y[i + e] / d);"),
    "q4_clamp_8": ("if (r > 7.0f)\n                        r = 7.0f;",
                   "if (r > 8.0f)\n                        r = 8.0f;"),
    "q4_nibble_swap": ("codes[i / 2] = (uint8_t)(c[0] | (c[1] << 4));",
                       "codes[i / 2] = (uint8_t)(c[1] | (c[0] << 4));"),
    "q4_offset_7": ("return (double)(c - 8) * (double)g_fp16_table[s];",
                    "return (double)(c - 7) * (double)g_fp16_table[s];"),
    "q4_scale_per_64_dims": ("+ d / KVO_Q4_BLOCK];", "+ d / KVO_GROUP];"),
    "hadamard_difference_reversed": ("x[j + h] = a - b;", "x[j + h] = b - a;"),
    "hadamard_skips_last_stage": ("for (int h = 1; h < n; h *= 2)", "for (int h = 1; h < n / 2; h *= 2)"),
    "attention_no_unrotate": ("if (fmt == KVO_FMT_K8V4)\n        unrotate_f64(o, hd);\n    return 0;", "return 0;"),
    "unrotate_not_divided": ("o[d] /= (double)hd;", "o[d] /= 1.0;"),
    "unrotate_difference_reversed": ("o[j + h] = a - b;", "o[j + h] = b - a;"),
    "compact_v_not_rotated_back": ("kvo_hadamard_f32(w, hd);", ""),
    "compact_v_not_divided": ("dv[d] = kvo_fp16_from_float(w[d] / (float)hd);",
                              "dv[d] = kvo_fp16_from_float(w[d]);"),
}


def _all_pins():
    """Every pin, as zero-argument callables."""
    pins = [f16.test_decode_every_bit_pattern,
            f16.test_encode_grid_points_midpoints_and_neighbours,
            qt.test_scale_one_ties_round_half_even, qt.test_scale_two_and_half,
            qt.test_negative_maximum_uses_absolute_value,
            qt.test_zero_group_and_underflowing_scale,
            qt.test_scale_is_rounded_to_fp16_before_dividing,
            qt.test_subnormal_scale_and_clamp, qt.test_overflowing_scale_gives_zero_codes,
            qt.test_division_is_by_the_scale_not_times_its_reciprocal,
            lambda: qt.test_invariants_on_random_rows(256),
            att.test_shuffled_block_table_moves_whole_blocks,
            att.test_two_cells_closed_form,
            att.test_queries_without_visible_cells_are_zero]
    for fmt in (F16, Q8):
        pins += [lambda fmt=fmt: att.test_fp16_store_and_q8_roundtrip(fmt),
                 lambda fmt=fmt: att.test_one_visible_cell_returns_its_value(fmt),
                 lambda fmt=fmt: att.test_equal_keys_give_mean_of_values(fmt),
                 lambda fmt=fmt: att.test_compaction(fmt)]
    for args in [(F16, 4, 2, 64, 3), (Q8, 3, 4, 128, 4), (Q8, 2, 8, 256, 1)]:
        pins.append(lambda args=args: att.test_matches_torch_sdpa(*args))
    pins += [lambda: chk.test_matches_torch_sdpa(1, 4, 128, 200, 37),
             lambda: chk.test_matches_torch_sdpa(2, 2, 64, 96, 96),
             chk.test_matches_paged_attention_over_an_fp16_pool,
             chk.test_first_token_of_a_whole_prompt_sees_one_cell,
             chk.test_equal_keys_give_the_running_mean_of_v,
             per.test_int8_codes_without_scales_are_refused]
    pins += [lambda: k84.test_transform_is_sylvester_hadamard(64),
             k84.test_designed_block_scale_codes_and_nibble_order,
             k84.test_zero_block_gives_zero_scale_and_offset_codes,
             k84.test_random_rows_within_half_a_step,
             k84.test_stored_codes_are_the_row_quantizers,
             k84.test_one_visible_cell_returns_its_derotated_value,
             lambda: k84.test_matches_torch_sdpa(2, 4, 256, 3),
             k84.test_compaction_derotates_v,
             k84.test_compaction_exact_when_every_block_shares_its_scale]
    for fmt in (F16, Q8, oracle.FMT_K8V4):
        pins += [lambda fmt=fmt: per.test_gather_returns_the_stored_rows_in_order(fmt),
                 lambda fmt=fmt: per.test_scatter_into_another_layout_then_gather_is_the_identity(fmt)]
    return pins


def _failures(so_path):
    failed = 0
    with oracle.use_library(so_path):
        for pin in _all_pins():
            try:
                pin()
            except (AssertionError, RuntimeError, ValueError, FloatingPointError):
                failed += 1
    return failed


def test_unmodified_copy_passes_every_pin(tmp_path):
    so = oracle.build_variant(oracle.source_text(), str(tmp_path), "kvq_oracle_copy")
    assert _failures(so) == 0


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {name}"
    so = oracle.build_variant(src.replace(old, new), str(tmp_path), "kvq_oracle_" + name)
    assert _failures(so) > 0, f"no pin caught the planted mistake '{name}'"
