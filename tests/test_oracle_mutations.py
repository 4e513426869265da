"""The oracle pins must catch plausible mistakes.

Each case edits one line of a copy of the oracle source (a dropped term, a
wrong sign or index, a swapped operand), compiles it to a temporary library on
the CPU, and runs the pin checks against it: at least one must fail.  The
unmodified source must pass the same checks.
"""
import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

MUTATIONS = {
    "causal_diagonal_dropped": ("const int pos = nb - w + t;", "const int pos = nb - w + t - 1;"),
    "ratio_without_one_minus_p": ("const double ratio = p / one_minus_p;", "const double ratio = p;"),
    "residual_sign": ("const double diff = a[c] - load_elem", "const double diff = a[c] + load_elem"),
    "gqa_sum_not_mean": ("raw[j] = sum / (double)g;", "raw[j] = sum;"),
    "gqa_last_head_dropped": ("for (int hl = 0; hl < g; ++hl) sum += heads", "for (int hl = 0; hl + 1 < g; ++hl) sum += heads"),
    "gqa_interleaved_heads": ("const int hq = h * g + hl;", "const int hq = hl * s->Hkv + h;"),
    "scale_1_over_d": ("const double inv_sqrt_d = 1.0 / sqrt((double)d);\n    const size_t kv_base",
                       "const double inv_sqrt_d = 1.0 / (double)d;\n    const size_t kv_base"),
    "prefill_scale_1_over_d": ("const double inv_sqrt_d = 1.0 / sqrt((double)d);\n    for (;;) {",
                               "const double inv_sqrt_d = 1.0 / (double)d;\n    for (;;) {"),
    "unnormalised_output": ("a[c] += p * load_elem", "a[c] += e[j] * load_elem"),
    "pool_window_short": ("int lo = j - half, hi = j + half;", "int lo = j - half, hi = j + half - 1;"),
    "protect_one_short": ("for (int j = nb - job->protect; j < nb; ++j)",
                          "for (int j = nb - job->protect + 1; j < nb; ++j)"),
    "tie_break_reversed": ("return (a->idx > b->idx) - (a->idx < b->idx);",
                           "return (a->idx < b->idx) - (a->idx > b->idx);"),
    "square_not_taken": ("s_head[j] += ratio * ratio * dist;", "s_head[j] += ratio * dist;"),
    "dominant_key_in_its_own_rest": ("if (i == j) continue;", "if (i == j && i < 0) continue;"),
    "dominant_square_not_taken": ("s_head[j] += p_dom * p_dom * dist_rest;", "s_head[j] += p_dom * dist_rest;"),
    "dominant_rest_unnormalised": ("const double diff = ar[c] / l_rest - load_elem",
                                   "const double diff = ar[c] - load_elem"),
    "snapkv_unnormalised": ("for (int j = 0; j <= pos; ++j) s_head[j] += e[j] / l;",
                            "for (int j = 0; j <= pos; ++j) s_head[j] += e[j];"),
    "snapkv_singular_rule": ("if (p == 1.0 && job->kind == ORACLE_KIND_DROPKV) return ORACLE_SINGULAR;",
                             "if (p == 1.0) return ORACLE_SINGULAR;"),
    "layer_evicts_one_more": ("for (size_t i = (size_t)evict_total[b]; i < m; ++i) keep[tmp[i].idx] = 1;",
                              "for (size_t i = (size_t)evict_total[b] + 1; i < m; ++i) keep[tmp[i].idx] = 1;"),
    "prefill_diagonal_dropped": ("for (int j = 0; j <= i; ++j) {\n                double dot = 0.0;",
                                 "for (int j = 0; j < i; ++j) {\n                double dot = 0.0;"),
    "prefill_unnormalised": ("const double p = x[j] / l;\n                for (int c = 0; c < d; ++c) acc[c]",
                             "const double p = x[j];\n                for (int c = 0; c < d; ++c) acc[c]"),
    "layer_ties_by_position_first": ("tmp[m].idx = (int32_t)((size_t)h * n_max + (size_t)j);",
                                     "tmp[m].idx = (int32_t)((size_t)j * s->Hkv + (size_t)h);"),
}


def _run_pins():
    pins.test_raw_score_equals_actual_deletion_tiny(42)
    pins.test_raw_score_gqa_group7()
    pins.test_raw_score_equals_actual_deletion_ragged_mha()
    pins.test_window_attention_vs_sdpa(42)
    pins.test_pool_vs_max_pool1d_and_protection(3)
    pins.test_select_vs_stable_sort_with_ties(0)
    pins.test_snapkv_raw_vs_torch_softmax(42)
    pins.test_snapkv_has_no_singular_rule()
    pins.test_select_layer_vs_stable_sort(0)
    pins.test_sink_score_equals_deletion_near_one(13.8)
    pins.test_prefill_attention_vs_sdpa(0)


def test_unmodified_source_passes(tmp_path):
    lib = oracle.compile_variant(oracle.source(), str(tmp_path / "lib_ok.so"))
    with oracle.use_library(lib):
        _run_pins()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source()
    assert src.count(old) == 1, name
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / ("lib_%s.so" % name)))
    with oracle.use_library(lib):
        with pytest.raises((AssertionError, oracle.OracleError)):
            _run_pins()
