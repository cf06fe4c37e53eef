"""Plausible mistakes planted in copies of the oracle must each fail a pin.

Every mutant is the oracle's C source with one textual change, compiled on
the CPU into a temporary directory.  The pins of test_oracle_pins.py run on
each mutant; the test passes only if at least one pin rejects it.  This shows
the pins would notice a dropped term, a wrong sign or index, a swapped
operand, a wrong initial state, the wrong-order update that the Lesson 7 page
warns about (section 3), or a reversed tie rule.
"""
import os

import pytest

import oracle
from tests.test_oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "sum_without_max_shift": ("d += exp(x[j] - m);", "d += exp(x[j]);"),
    "combine_wrong_sign": ("d1 * exp(m1 - m)", "d1 * exp(m - m1)"),
    "combine_drops_second_term": ("d1 * exp(m1 - m) + d2 * exp(m2 - m)", "d1 * exp(m1 - m)"),
    "combine_swapped_operands": ("d2 * exp(m2 - m)", "d2 * exp(m1 - m)"),
    "recurrence_overwrites_max_first": (
        "d = d * exp(m - m_new) + exp(x[j] - m_new);\n        m = m_new;",
        "m = m_new;\n        d = d * exp(m - m_new) + exp(x[j] - m_new);"),
    "max_starts_at_zero": ("double m = -INFINITY;\n    for", "double m = 0.0;\n    for"),
    "output_divides_by_max": ("yr[j] = exp(xr[j] - m) / d;", "yr[j] = exp(xr[j] - m) / (d + m * 0.0 + 1e-3);"),
    "topk_ties_to_higher_index": ("return (a->j > b->j) - (a->j < b->j);",
                                  "return (a->j < b->j) - (a->j > b->j);"),
    "topk_value_transposed": ("vals[r * K + k] = exp(order[k].x - m) / d;",
                              "vals[r * K + k] = exp(m - order[k].x) / d;"),
    "topk_ascending": ("if (a->x > b->x) return -1;\n    if (a->x < b->x) return 1;",
                       "if (a->x < b->x) return -1;\n    if (a->x > b->x) return 1;"),
    "lse_drops_max": ("lse[r] = m == -INFINITY ? -INFINITY : m + log(d);",
                      "lse[r] = m == -INFINITY ? -INFINITY : log(d);"),
    "lse_log10": ("lse[r] = m == -INFINITY ? -INFINITY : m + log(d);",
                  "lse[r] = m == -INFINITY ? -INFINITY : m + log10(d);"),
    "causal_mask_off_by_one": ("c > (r % period) + offset ? -INFINITY",
                               "c >= (r % period) + offset ? -INFINITY"),
    "causal_mask_ignores_period": ("c > (r % period) + offset ? -INFINITY",
                                   "c > r + offset ? -INFINITY"),
    "sample_ge_instead_of_gt": ("if (run > target) {", "if (run >= target) {"),
    "sample_compares_single_value": ("run += p[k];", "run = p[k];"),
    "sample_unnormalised_target": ("const double target = u[r] * total;",
                                   "const double target = u[r];"),
    "sample_total_skips_last": ("for (int32_t k = 0; k < K; ++k) total += p[k];",
                                "for (int32_t k = 0; k + 1 < K; ++k) total += p[k];"),
    "attention_drops_scale": ("s[j] = scale * acc;", "s[j] = acc;"),
    "attention_mask_excludes_diagonal": ("const int64_t seen = causal ? i + 1 : n;",
                                         "const int64_t seen = causal ? i : n;"),
    "attention_mask_from_the_end": ("const int64_t seen = causal ? i + 1 : n;",
                                    "const int64_t seen = causal ? n - i : n;"),
    "attention_value_row_of_query": ("oi[c] += p * vb[j * dh + c];", "oi[c] += p * vb[i * dh + c];"),
    "attention_key_row_of_query": ("acc += qi[c] * kb[j * dh + c];", "acc += qi[c] * kb[i * dh + c];"),
    "attention_unnormalised": ("const double p = exp(s[j] - m) / d;",
                               "const double p = exp(s[j] - m);"),
    "attention_lse_drops_max": ("*lse_out = m + log(d);", "*lse_out = log(d);"),
    "attention_max_not_subtracted_in_weights": ("d += exp(s[j] - m);\n    for (int64_t c",
                                                "d += exp(s[j]);\n    for (int64_t c"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(before) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text.replace(before, after))
    lib = oracle.load(oracle.compile_oracle(str(src), str(tmp_path / "liboracle_mutant.so")))
    failures = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"no pin rejects the mutant {name}"
