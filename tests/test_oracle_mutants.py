"""Plant mistakes in copies of the oracle and check that the pins catch each one.

Every mutant is a one-line textual change to the oracle's C++ source, compiled
into a temporary library (on the CPU; nothing here touches the CUDA selector).
The pin tests in test_oracle_pins.py are then run against the mutant, and at
least one of them must fail.  This shows that a plausible slip in the oracle
(a flipped comparison, a wrong tie-break, an off-by-one in the rank rule, a
strict/inclusive mix-up in the counts or the checker, a dropped or misplaced
ReLU or a transposed operand in the indexer scores, a reversed or index-keyed
ordered output) would not go unnoticed.
"""
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle_index_scores as score_pins
from tests import test_oracle_order as order_pins
from tests import test_oracle_pins as pins

MUTANTS = {
    "order_flipped": ("if (v[a] > v[b]) return true;", "if (v[a] < v[b]) return true;"),
    "tie_break_high_index": ("return a < b;", "return a > b;"),
    "sentinel_zero": ("o[i] = (i < L) ? (int32_t)i : -1;", "o[i] = (i < L) ? (int32_t)i : 0;"),
    "checker_strict_ties": ("min_sel < max_rest) err = 4;", "min_sel <= max_rest) err = 4;"),
    "checker_no_dup_check": ("if (seen[(size_t)x]) {", "if (false) {"),
    "rank_floor": ("int64_t rk = (targets[j] * ns + L - 1) / L;",
                   "int64_t rk = (targets[j] * ns) / L;"),
    "count_strict": ("c0 += (v[i] >= t[0]);", "c0 += (v[i] > t[0]);"),
    "sample_offset": ("for (int64_t i = 0; i < L; i += stride) samp.push_back(v[i]);",
                      "for (int64_t i = 1; i < L; i += stride) samp.push_back(v[i]);"),
    "boundary_off_by_one": ("const float b = vals[(size_t)K];", "const float b = vals[(size_t)K - 1];"),
    "len_not_clamped_high": ("if (v > n_alloc) v = n_alloc;", ""),
    "score_no_relu": ("acc += wj * (dot > 0.0 ? dot : 0.0);", "acc += wj * dot;"),
    "score_relu_after_sum": ("acc += wj * (dot > 0.0 ? dot : 0.0);", "acc += wj * dot;\n        if (j == H - 1 && acc < 0.0) acc = 0.0;"),
    "score_w_transposed": ("const double wj = (double)w[t * H + j];", "const double wj = (double)w[j * T + t];"),
    "score_k_wrong_row": ("bf16_to_double(k[sidx * D + d]);", "bf16_to_double(k[t * D + d]);"),
    "score_magnitude_signed": ("mag += std::fabs(wj) * adot;", "mag += wj * adot;"),
    "order_reversed": ("std::sort(idx.begin(), idx.end(), Before{v});",
                       "std::sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) "
                       "{ return Before{v}(b, a); });"),
    "order_by_index": ("std::sort(idx.begin(), idx.end(), Before{v});",
                       "std::sort(idx.begin(), idx.end());"),
    "order_sentinels_first": (
        "for (int64_t i = 0; i < K; ++i) o[i] = i < (int64_t)idx.size() ? idx[(size_t)i] : -1;",
        "for (int64_t i = 0; i < K; ++i) o[i] = i < K - (int64_t)idx.size() ? -1 : "
        "idx[(size_t)(i - (K - (int64_t)idx.size()))];"),
}


def _run_all_pins():
    for case in pins.CONTRACT_CASES:
        pins.test_golden_contract_cases(case)
    for dist in ("continuous", "few_values", "with_inf"):
        pins.test_brute_force_tiny_rows(dist)
    for L in (0, 1, 2047, 2048, 2049):
        pins.test_sentinel_rule_closed_form(L)
    pins.test_row_lens_are_clamped()
    pins.test_boundary_values_match_sorted_row()
    pins.test_checker_rejects_duplicate()
    pins.test_checker_rejects_out_of_range_and_negative()
    pins.test_checker_rejects_swapped_smaller_for_larger()
    pins.test_checker_rejects_sentinel_in_long_row()
    pins.test_checker_rejects_missing_sentinel_and_missing_index()
    for c in pins.THR:
        pins.test_threshold_closed_forms(c)
    pins.test_threshold_paths_hand_built_tau1_and_recovery()
    pins.test_threshold_paths_sentinel_and_direct()
    pins.test_certification_invariants_random_rows()
    score_pins.test_golden_case()
    score_pins.test_one_hot_closed_form()
    score_pins.test_invariances()
    score_pins.test_dense_product_tiny()
    for case in order_pins.ORDER_CASES:
        order_pins.test_golden_order_cases(case)
    order_pins.test_distinct_values_follow_argsort()
    order_pins.test_invariants_on_tied_rows()


def test_unmutated_oracle_passes_every_pin():
    _run_all_pins()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation anchor must appear exactly once"
    mutated = src.replace(old, new)
    cpp = os.path.join(tmp_path, "mutant.cpp")
    lib = os.path.join(tmp_path, "libmutant.so")
    with open(cpp, "w") as f:
        f.write(mutated)
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", cpp, "-o", lib],
                   check=True)
    with oracle.use_library(lib):
        with pytest.raises(AssertionError):
            _run_all_pins()
