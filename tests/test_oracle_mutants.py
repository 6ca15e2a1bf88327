"""Plants plausible mistakes in a temporary copy of the CPU oracle and checks
that the oracle's pins (tests/test_oracle_pins.py) catch every one.

The mistakes are planted only in copies compiled into a temporary directory;
the committed oracle is reloaded afterwards.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sd_oracle.cpp")

MUTANTS = {
    "residual_sign": ("std::max(0.0, p[(size_t)m][(size_t)i] - q[(size_t)m][(size_t)i])",
                      "std::max(0.0, q[(size_t)m][(size_t)i] - p[(size_t)m][(size_t)i])"),
    "residual_unclamped": ("std::max(0.0, p[(size_t)m][(size_t)i] - q[(size_t)m][(size_t)i])",
                           "std::fabs(p[(size_t)m][(size_t)i] - q[(size_t)m][(size_t)i])"),
    "accept_inverted": ("if (!(u <= r[(size_t)j]))", "if (!(u >= r[(size_t)j]))"),
    "ratio_inverted": ("r[(size_t)j] = qd > 0.0 ? pd / qd", "r[(size_t)j] = qd > 0.0 ? qd / pd"),
    "bonus_wrong_row": ("w = p[(size_t)K];", "w = p[(size_t)K - 1];"),
    "greedy_emits_draft": ("res.token = amax[(size_t)m];",
                           "res.token = m < K ? tokens[m] : amax[(size_t)m];"),
    "cdf_off_by_one": ("      return (int)i;\n    }\n  }\n  int last",
                       "      return (int)std::min(i + 1, w.size() - 1);\n    }\n  }\n  int last"),
    "philox_word_swap": ("const uint32_t n1 = lo1;", "const uint32_t n1 = hi1;"),
    "no_temperature": ("e[i] = std::exp((l[i] - m) / T);", "e[i] = std::exp(l[i] - m);"),
    "keys_keep_drafted": ("if (i == excl ||", "if (false ||"),
    "offsets_inclusive": ("    offsets[b] = acc;\n", "    offsets[b] = acc + tau[b];\n"),
    "tau_off_by_one": ("res.tau = res.n_acc + 1;", "res.tau = res.n_acc;"),
    "argmax_last_tie": ("if (l[(size_t)i] > l[(size_t)best]) best = i;",
                        "if (l[(size_t)i] >= l[(size_t)best]) best = i;"),
    "accept_uses_sample_slot": ("uniform_from_philox(seed, row, (uint32_t)j, 0u)",
                                "uniform_from_philox(seed, row, (uint32_t)j, 1u)"),
    "pack_position_off_by_one": ("p[i] = anchor_pos[b] + 1 + k + i;",
                                 "p[i] = anchor_pos[b] + k + i;"),
    "pack_ctx_off_by_one": ("      c = k + 1;", "      c = k;"),
    "ngram_earliest_match": ("for (int i = n_tok - n - 1; i >= 0; --i) {",
                             "for (int i = 0; i <= n_tok - n - 1; ++i) {"),
    "ngram_matches_itself": ("for (int i = n_tok - n - 1; i >= 0; --i) {",
                             "for (int i = n_tok - n; i >= 0; --i) {"),
    "rollback_keeps_tau_plus_one": ("std::min(std::max(tau[b], 0), appended)",
                                    "std::min(std::max(tau[b] + 1, 0), appended)"),
    "rollback_floor_pages": ("const int still = (n_new + page_size - 1) / page_size;",
                             "const int still = n_new / page_size;"),
    # the guard that decides which sampled decisions are compared exactly
    "guard_upper_edge_only": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                              "*near = (C - target) < kGuard * S;"),
    "guard_lower_edge_only": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                              "*near = (target - prev) < kGuard * S;"),
    "guard_absolute_window": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                              "*near = std::min(C - target, target - prev) < kGuard;"),
    "guard_total_for_target": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                               "*near = std::min(C - S, S - prev) < kGuard * S;"),
    "guard_never_flags_draw": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                               "*near = false;"),
    "guard_flags_every_draw": ("*near = std::min(C - target, target - prev) < kGuard * S;",
                               "*near = true;"),
    "guard_fallthrough_unflagged": ("*near = true;  // the draw fell",
                                    "*near = false;  // the draw fell"),
    "guard_accept_window_wide": ("std::fabs(u - r[(size_t)j]) < kGuard",
                                 "std::fabs(u - r[(size_t)j]) < 10 * kGuard"),
    "finite_allows_posinf": ("if (std::isnan(v) || v == std::numeric_limits<double>::infinity()) return true;",
                             "if (std::isnan(v)) return true;"),
    "finite_allows_all_neg_inf": ("  return !any_finite;\n}", "  return false;\n}"),
    "finite_reads_every_draft_row": ("if (T > 0.0 || (fc.keys_at && fc.keys_at[j] > 0))",
                                     "if (true)"),
    "finite_skips_bonus_row": ("if (!bad && fc.bonus && fc.keys_at && fc.keys_at[K] > 0)",
                               "if (false)"),
    "guard_accept_never": ("if (res.guard_pos < 0 && std::fabs(u - r[(size_t)j]) < kGuard)",
                           "if (false)"),
}

FAST_PINS = [
    pins.test_guard_flags_decisions_near_a_boundary,
    pins.test_guard_flags_draws_near_a_cdf_edge,
    pins.test_finite_check_flags_exactly_the_rows_read,
    pins.test_worked_example_greedy,
    pins.test_bonus_when_all_greedy_drafts_match,
    pins.test_greedy_argmax_ties_match_torch_first_occurrence,
    lambda o: pins.test_losslessness_exact_enumeration_V4_K2(o, 0.7),
    pins.test_identical_models_accept_everything,
    pins.test_probabilities_match_torch_softmax_float64,
    pins.test_outcome_keys_match_stable_sort_brute_force,
    pins.test_key_counts_from_d3d_preparation_table,
    pins.test_d3d_pack_worked_example,
    pins.test_d3d_pack_hit_block_continues_confirmed_text,
    pins.test_ngram_draft_worked_example,
    pins.test_ngram_draft_matches_substring_search,
    pins.test_kv_rollback_worked_example,
    pins.test_kv_rollback_matches_entry_sets,
    pins.test_hit_test_brute_force,
    pins.test_compaction_brute_force,
    pins.test_invalid_rows_and_degenerate_K0,
    pins.test_philox_known_answers,
]


def _caught(lib_module):
    for pin in FAST_PINS:
        try:
            pin(lib_module)
        except AssertionError:
            return True
    # the Monte-Carlo pin is slower: only reached when every fast pin passed
    try:
        pins.test_chi_square_V8_one_million_rounds(lib_module)
    except AssertionError:
        return True
    return False


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "sd_oracle_mutant.cpp"
    mutated.write_text(src.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off",
                    str(mutated), "-o", str(so)], check=True)
    try:
        oracle.load_library(str(so))
        assert _caught(oracle), f"planted mistake '{name}' passed every pin"
    finally:
        oracle.load_library(oracle.build())
