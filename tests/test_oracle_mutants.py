"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins in test_oracle_pins reject every one. This shows the pins constrain
each part of the oracle (sign, index, rounding rule, tie rule, parameter
formulas), not just that the oracle agrees with itself."""
import os
import subprocess

import pytest

import oracle
import test_oracle_backward as bpins
import test_oracle_pins as pins

MUTANTS = [
    ("no_relu", "float relu = dot[h] > 0.0f ? dot[h] : 0.0f;", "float relu = dot[h];"),
    ("no_weight", "acc += wt[h] * relu;", "acc += relu;"),
    ("dropped_head", "    acc += wt[h] * relu;\n", "    acc += h + 1 < H ? wt[h] * relu : 0.0f;\n"),
    ("ties_high_pos", "return (x->pos > y->pos) - (x->pos < y->pos);",
     "return (x->pos < y->pos) - (x->pos > y->pos);"),
    ("no_k_scale", "p->kf[(size_t)s * d + i] = kd == ORACLE_E4M3 ? v * scale : v;",
     "p->kf[(size_t)s * d + i] = v;"),
    ("no_q_scale", "qT[(size_t)i * p->H + h] = qd == ORACLE_E4M3 ? v * scale : v;",
     "qT[(size_t)i * p->H + h] = v;"),
    ("transposed_q", "size_t at = ((size_t)t * p->H + h) * p->d + i;",
     "size_t at = (size_t)t * p->H * p->d + ((size_t)i * p->H + h) % ((size_t)p->H * p->d);"),
    ("exclusive_causal",
     "int64_t ctx = (int64_t)positions[t] + 1;\n      query_operand(&p, t, qT);\n"
     "      for (int64_t s = 0; s < ctx; ++s) {",
     "int64_t ctx = (int64_t)positions[t];\n      query_operand(&p, t, qT);\n"
     "      for (int64_t s = 0; s < ctx; ++s) {"),
    ("M_ceil", "int64_t m = ctx / 128;", "int64_t m = (ctx + 127) / 128;"),
    ("r_floor", "(3 * k_top * m + ctx - 1) / ctx", "(3 * k_top * m) / ctx"),
    ("r_off_by_one", "float T = samp[rank - 1];", "float T = samp[rank];"),
    ("strict_filter", "cnt += row[s] >= T;", "cnt += row[s] > T;"),
    ("sample_midpoint", "return (j * ctx) / m;", "return (j * ctx + ctx / 2) / m;"),
    ("subnormal_exp", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("e4m3_bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("mixed_q_as_bf16", "static int q_dtype(int dtype) { return dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_E4M3; }",
     "static int q_dtype(int dtype) { return dtype == ORACLE_E4M3 ? ORACLE_E4M3 : ORACLE_BF16; }"),
    # the backward at selected entries
    ("bwd_dq_no_weight", "dqt[e] += coef * ks[i];", "dqt[e] += g * ks[i];"),
    ("bwd_dk_uses_key", "dk[e] += coef * qd[(size_t)h * d + i];", "dk[e] += coef * ks[i];"),
    ("bwd_dw_no_relu", "dw[t * H + h] += g * relu;", "dw[t * H + h] += g * x;"),
    ("bwd_mask_at_zero", "if (x > 0.0) {\n              dqt[e]", "if (x >= 0.0) {\n              dqt[e]"),
    ("bwd_wrong_key_row", "size_t e = (size_t)s * d + i;", "size_t e = (size_t)((s + 1) % L) * d + i;"),
    ("bwd_no_k_scale", "double v = (double)element(k, k_dtype(dtype), (size_t)s * d + i) * scale;",
     "double v = (double)element(k, k_dtype(dtype), (size_t)s * d + i);"),
    ("bwd_grad_row", "double g = (double)grad[t * k_top + j];\n        const double* ks = kd + (size_t)s * d;\n        for (int h = 0; h < H; ++h) {\n          double x = 0.0;\n          for (int i = 0; i < d; ++i) x += qd[(size_t)h * d + i] * ks[i];\n          int amb = fabs(x) <= eps * qnorm[h] * knorm[s];\n          double relu",
     "double g = (double)grad[((t + 1) % n) * k_top + j];\n        const double* ks = kd + (size_t)s * d;\n        for (int h = 0; h < H; ++h) {\n          double x = 0.0;\n          for (int i = 0; i < d; ++i) x += qd[(size_t)h * d + i] * ks[i];\n          int amb = fabs(x) <= eps * qnorm[h] * knorm[s];\n          double relu"),
]


def battery():
    """Fast pins; returns how many of them reject the current oracle build."""
    checks = [
        pins.test_worked_example_closed_forms,
        lambda: pins.test_sample_count_within_printed_bounds(65536),
        lambda: pins.test_sample_count_within_printed_bounds(600000),
        pins.test_sample_count_small_contexts,
        pins.test_e4m3_decode_every_code,
        lambda: pins.test_select_matches_exact_bruteforce(40, 8, 2, 3, 7, 1),
        lambda: pins.test_select_matches_exact_bruteforce(64, 10, 4, 8, 16, 2),
        pins.test_select_e4m3_scales_exact,
        pins.test_negative_weights_and_relu,
        pins.test_scalar_textbook_case,
        pins.test_all_equal_scores_and_short_context,
        pins.test_filter_full_sampling_threshold_is_exact_rank,
        pins.test_filter_certificate_holds,
        pins.test_filter_threshold_rank_on_distinct_scores,
        pins.test_mixed_e4m3_q_bf16_k_reduces_to_bf16,
        bpins.test_dw_is_the_difference_in_w,
        bpins.test_dq_is_the_difference_in_q,
        bpins.test_dk_is_the_difference_in_k,
        bpins.test_relu_kink_derivative_is_zero,
        bpins.test_empty_and_bad_indices,
        bpins.test_e4m3_scales_enter_the_gradient,
    ]
    failed = 0
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    return failed


def test_unmutated_oracle_passes_battery():
    assert battery() == 0


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    c = tmp_path / f"{name}.c"
    c.write_text(src.replace(old, new))
    so = str(tmp_path / f"lib_{name}.so")
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(c), "-o", so, "-lm"])
    with oracle._use_library(so):
        rejected = battery()
    assert rejected > 0, f"no pin rejects the planted mistake {name}"
