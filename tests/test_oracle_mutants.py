"""Negative controls: plant plausible mistakes in a copy of the oracle source,
rebuild it, and check that at least one pin catches each mistake (the Kestrel
article's section 3.2.1 makes the same point: a check that still passes with
the mechanism removed proves nothing)."""
import os
import shutil

import pytest

import _pins
import oracle

MUTANTS = {
    "ratio_inverted": ("ratio[i] = qi > 0.0 ? pi / qi : INFINITY;",
                       "ratio[i] = qi > 0.0 ? qi / pi : INFINITY;"),
    "accept_wrong_row": ("oracle_softmax(tb + (size_t)i * V * es, dtype, T, V, p);",
                         "oracle_softmax(tb + (size_t)(i + 1) * V * es, dtype, T, V, p);"),
    "residual_without_clamp_resamples_p": ("w[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;",
                                           "w[t] = p[t];"),
    "residual_sign_flipped": ("w[t] = p[t] - q[t] > 0.0 ? p[t] - q[t] : 0.0;",
                              "w[t] = q[t] - p[t] > 0.0 ? q[t] - p[t] : 0.0;"),
    "bonus_from_draft_row": ("memcpy(w, p, sizeof(double) * (size_t)V);",
                             "oracle_softmax(db + (size_t)(j - 1) * V * es, dtype, T, V, w);"),
    "inverse_cdf_non_strict": ("if (c > target) {", "if (c >= target) {"),
    "argmax_last_tie": ("if (v > bv) {", "if (v >= bv) {"),
    "tree_compares_own_row": ("if (node < 0 || tok[node] != g[path[j - 1]])",
                              "if (node < 0 || tok[node] != g[node])"),
    "temperature_multiplies": ("p[t] = logit_at(x, dtype, (size_t)t) / temperature;",
                               "p[t] = logit_at(x, dtype, (size_t)t) * temperature;"),
    "softmax_unnormalised": ("p[t] /= sum;", "p[t] /= 1.0;"),
    "softmax_without_max_shift": ("p[t] = exp(p[t] - zmax);", "p[t] = exp(p[t]);"),
    "bf16_widened_with_wrong_shift": ("uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;",
                                      "uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 15;"),
    "rollback_drops_committed_token": ("new_lens[b] = old_lens[b] + n + 1;",
                                       "new_lens[b] = old_lens[b] + n;"),
    "scan_does_not_stop": ("j = i;\n                break;", "j = i;"),
    # symmetric filtering (TensorRT-LLM walkthrough, rejection-sampling section)
    "filtered_tie_keeps_higher_index": ("return u->t < v->t ? -1 : (u->t > v->t);",
                                        "return u->t > v->t ? -1 : (u->t < v->t);"),
    "top_p_cut_strict": ("if (cum >= top_p) {", "if (cum > top_p) {"),
    "top_p_mass_over_vocabulary": ("for (int i = 0; i < kk; ++i)\n        sk += exp(",
                                   "for (int i = 0; i < V; ++i)\n        sk += exp("),
    "kept_set_not_renormalised": ("p[it[i].t] = exp(it[i].x / temperature - zmax) / sm;",
                                  "p[it[i].t] = exp(it[i].x / temperature - zmax) / sk;"),
    "draft_side_not_filtered": ("oracle_filter_row(db + (size_t)i * V * es, dtype, T, V, top_k, top_p, min_p, q, &tq);",
                                "oracle_softmax(db + (size_t)i * V * es, dtype, T, V, q);"),
    "residual_draft_not_filtered": ("oracle_filter_row(db + (size_t)j * V * es, dtype, T, V, top_k, top_p, min_p, q, &tq);",
                                    "oracle_softmax(db + (size_t)j * V * es, dtype, T, V, q);"),
    # per-request Philox uniforms (TensorRT-LLM walkthrough, rejection-sampling section)
    "philox_nine_rounds": ("for (int round = 0; round < 10; ++round) {",
                           "for (int round = 0; round < 9; ++round) {"),
    "philox_key_words_swapped": ("const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;",
                                 "const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k1;"),
    "uniform_from_low_bits": ("(float)((double)(r[i % 4] >> 8) * (1.0 / 16777216.0))",
                              "(float)((double)(r[i % 4] & 0xFFFFFFu) * (1.0 / 16777216.0))"),
    "uniform_counter_words_swapped": ("(uint32_t)(i / 4), 0u};", "0u, (uint32_t)(i / 4)};"),
    # ragged lengths and paged rollback (TensorRT-LLM walkthrough, update_requests, rewind_cache)
    "paged_blocks_rounded_down": ("const long long need = (len + tokens_per_block - 1) / tokens_per_block;",
                                  "const long long need = len / tokens_per_block;"),
    "paged_rewind_from_padded_k": ("rewind_lens[b] = kb - n;", "rewind_lens[b] = k - n;"),
    "ragged_draw_uniform_at_padded_k": ("int tok = oracle_inverse_cdf(w, V, (double)r[kb], SAMPLE_TIE, &tie);",
                                        "int tok = oracle_inverse_cdf(w, V, (double)r[k], SAMPLE_TIE, &tie);"),
    "greedy_scans_padding": ("while (j < kb && oracle_argmax", "while (j < k && oracle_argmax"),
    "tree_tie_keeps_later_path": ("if (acc > best_acc) {", "if (acc >= best_acc) {"),
    "rollback_bad_entry_rewind_zero": ("if (n < 0 || n > k) {\n            new_lens[b] = old_lens[b];\n            if (rewind_lens)\n                rewind_lens[b] = -1;",
                                       "if (n < 0 || n > k) {\n            new_lens[b] = old_lens[b];\n            if (rewind_lens)\n                rewind_lens[b] = 0;"),
    "paged_bad_entry_rewind_zero": ("if (kb < 0 || kb > k || n < 0 || n > kb) {\n            new_lens[b] = old_lens[b];\n            if (rewind_lens)\n                rewind_lens[b] = -1;",
                                    "if (kb < 0 || kb > k || n < 0 || n > kb) {\n            new_lens[b] = old_lens[b];\n            if (rewind_lens)\n                rewind_lens[b] = 0;"),
    # stochastic tree verify (children as point-mass proposals)
    "tree_sampled_not_renormalised": ("const double ratio = (1.0 - removed) > 0.0 ? pc / (1.0 - removed) : 0.0;",
                                      "const double ratio = pc;"),
    "tree_sampled_rejected_kept": ("p[tok[c]] = 0.0; /* the residual no longer holds tok c */", ";"),
    "tree_sampled_children_descending": ("for (int j2 = i; j2 > 0 && cand[j2 - 1] > cand[j2]; --j2) {",
                                         "for (int j2 = i; j2 > 0 && cand[j2 - 1] < cand[j2]; --j2) {"),
    "tree_sampled_final_uniform_of_node": ("final_tok = oracle_inverse_cdf(w, V, (double)u[0], SAMPLE_TIE, &tie);",
                                           "final_tok = oracle_inverse_cdf(w, V, (double)u[node], SAMPLE_TIE, &tie);"),
    "tree_sampled_tests_root_row": ("oracle_softmax(tb + (size_t)node * V * es, dtype, T, V, p);\n            /* candidates",
                                    "oracle_softmax(tb, dtype, T, V, p);\n            /* candidates"),
    "tree_sampled_window_unscaled": ("fabs((double)u[c] - ratio) < ACCEPT_TIE / (1.0 - removed))",
                                     "fabs((double)u[c] - ratio) < ACCEPT_TIE)"),
    # min_p and top-p over the whole vocabulary (reading F6)
    "min_p_against_mass": ("const double ratio = exp(it[i].x / temperature - zmax);",
                           "const double ratio = exp(it[i].x / temperature - zmax) / sk;"),
    "min_p_strict": ("if (ratio >= min_p)", "if (ratio > min_p)"),
    "no_top_k_means_no_filter": ("    qsort(it, (size_t)V, sizeof(orc_item), orc_item_order);",
                                 "    if (top_k <= 0) {\n        free(it);\n        return oracle_softmax(x, dtype, temperature, V, p);\n    }\n    qsort(it, (size_t)V, sizeof(orc_item), orc_item_order);"),
    "min_p_skipped_on_target_rows": ("oracle_filter_row(tb + (size_t)i * V * es, dtype, T, V, top_k, top_p, min_p, p, &tp);",
                                     "oracle_filter_row(tb + (size_t)i * V * es, dtype, T, V, top_k, top_p, 0.0, p, &tp);"),
    # near-tie windows (|r - p/q| < 1e-5; u*Z within 1e-6*Z of a CDF boundary)
    "accept_window_wide": ("static const double ACCEPT_TIE = 1e-5;",
                           "static const double ACCEPT_TIE = 1.0;"),
    "sample_window_wide": ("static const double SAMPLE_TIE = 1e-6;",
                           "static const double SAMPLE_TIE = 1.0;"),
    "draw_always_flagged": ("*near_tie = (fabs(c - target) <= tol * Z) || (fabs(c_prev - target) <= tol * Z);",
                            "*near_tie = 1;"),
    "draw_never_flagged": ("*near_tie = (fabs(c - target) <= tol * Z) || (fabs(c_prev - target) <= tol * Z);",
                           "*near_tie = 0;"),
    "accept_never_flagged": ("if (flags && fabs((double)r[i] - ratio[i]) < ACCEPT_TIE)",
                             "if (flags && fabs((double)r[i] - ratio[i]) < 0.0)"),
    "draw_flag_one_side_only": ("*near_tie = (fabs(c - target) <= tol * Z) || (fabs(c_prev - target) <= tol * Z);",
                                "*near_tie = (fabs(c - target) <= tol * Z);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    mutated = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    so = str(tmp_path / "libmutant.so")
    oracle.build(src=str(path), out=so, force=True)
    lib = oracle.load(so)
    caught = [n for n, pin in _pins.ALL_PINS.items() if pin(lib=lib)]
    assert caught, f"no pin catches mutant {name}"
