"""The pins are sharp: each plausible mistake planted in a copy of the
oracle's C source (a transposed operand, a wrong sign, a wrong row, a dropped
stop, a dropped temperature, a broken constant, a reversed tie order) makes at
least one pin of test_oracle_pins fail.  Mutants are compiled to a temporary
library; the committed oracle is untouched."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_enumeration as enum
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spv_oracle.c")

MUTANTS = {
    "accept_transposed": ("int acc = (p > 0) && ((double)r[i] * q <= p);",
                          "int acc = (p > 0) && ((double)r[i] * p <= q);",
                          ["test_acceptance_rate_is_one_minus_tvd", "test_target_above_draft_always_accepts",
                           "test_enumeration_designed_thresholds"]),
    "residual_sign": ("double d = w[x] - prob(dj, x, T, Md[k], Sd[k]);",
                      "double d = prob(dj, x, T, Md[k], Sd[k]) - w[x];",
                      ["test_residual_fallback_is_exact"]),
    "bonus_wrong_row": ("const float *tb = tgt + (size_t)gamma * V;",
                        "const float *tb = tgt + (size_t)(gamma - 1) * V;",
                        ["test_bonus_is_distributed_as_last_target_row"]),
    "no_first_rejection_stop": ("if (i < k) { /* decisions", "if (1) { /* decisions",
                                ["test_expected_tokens_per_iteration", "test_output_length_and_padding",
                                 "test_enumeration_arbitrary_pairs"]),
    "temperature_dropped": ("return exp((double)z[x] / T - M) / S;", "return exp((double)z[x] - M) / S;",
                            ["test_acceptance_rate_is_one_minus_tvd"]),
    "trial_accept_inverted": ("if (q <= (1.0 - v) * p) { emitted = x; break; }",
                              "if (p <= (1.0 - v) * q) { emitted = x; break; }",
                              ["test_residual_distribution_on_forced_rejection", "test_trial_acceptance_enumerated"]),
    "block_race_weight": ("arr[b] = Wb > 0 ? expo(key, s_block, trial, pos, (uint64_t)b) / Wb : INFINITY;",
                          "arr[b] = Wb > 0 ? expo(key, s_block, trial, pos, (uint64_t)b) * Wb : INFINITY;",
                          ["test_first_token_is_distributed_as_target", "test_bonus_is_distributed_as_last_target_row"]),
    "sub_block_race_weight": ("arr[j] = Ws > 0 ? expo(key, s_sub, trial, pos, (uint64_t)j) / Ws : INFINITY;",
                              "arr[j] = Ws > 0 ? expo(key, s_sub, trial, pos, (uint64_t)j) : INFINITY;",
                              ["test_first_token_is_distributed_as_target",
                               "test_bonus_is_distributed_as_last_target_row"]),
    "token_race_weight": ("arr[x - s0] = w[x] > 0 ? expo(key, s_tok, trial, pos, (uint64_t)(x - s0)) / w[x] : INFINITY;",
                          "arr[x - s0] = w[x] > 0 ? expo(key, s_tok, trial, pos, (uint64_t)(x - s0)) : INFINITY;",
                          ["test_first_token_is_distributed_as_target", "test_bonus_is_distributed_as_last_target_row"]),
    "philox_constant": ("uint64_t p0 = (uint64_t)0xD2511F53u * c0;", "uint64_t p0 = (uint64_t)0xD2511F55u * c0;",
                        ["test_philox_known_answer_vectors"]),
    "fanout_tie_order": ("return (x->id > y->id) - (x->id < y->id);", "return (x->id < y->id) - (x->id > y->id);",
                         ["test_fanout_vs_numpy_lexsort"]),
    "greedy_last_tie": ("if (best < 0 || v > bv) { best = x; bv = v; }", "if (best < 0 || v >= bv) { best = x; bv = v; }",
                        ["test_greedy_matches_numpy_argmax"]),
    "cache_wrong_position": ("if (pos == k && cache_ids[slot] == t_star) return slot;",
                             "if (pos == k + 1 && cache_ids[slot] == t_star) return slot;",
                             ["test_cache_full_fanout_always_hits", "test_cache_hit_rate_closed_form"]),
    "cache_slot_within_position": ("if (pos == k && cache_ids[slot] == t_star) return slot;",
                                   "if (pos == k && cache_ids[slot] == t_star) return j;",
                                   ["test_cache_full_fanout_always_hits",
                                    "test_cache_slot_first_entry_of_the_outcome_position"]),
    "filter_not_renormalised": ("    for (int j = 0; j < n; ++j) probs_out[j] /= s;\n",
                                "\n",
                                ["test_filter_row_vs_torch_topk_softmax"]),
    "top_p_cut_one_late": ("if (after >= top_p) {", "if (before >= top_p) {", ["test_filter_top_p_closed_form"]),
    "filtered_residual_sign": ("wx = wx - qx > 0 ? wx - qx : 0.0;", "wx = qx - wx > 0 ? qx - wx : 0.0;",
                               ["test_filtered_residual_on_forced_rejection"]),
    "filtered_race_weight": ("expo(seq_key, SPVO_STREAM_FILTERED, 0, (uint32_t)k, (uint64_t)x) / wx",
                             "expo(seq_key, SPVO_STREAM_FILTERED, 0, (uint32_t)k, (uint64_t)x) * wx",
                             ["test_filtered_first_token_and_bonus_are_exact"]),
    "filtered_accept_transposed": ("int stands = (p > 0) && ((double)r[i] * q <= p);",
                                   "int stands = (p > 0) && ((double)r[i] * p <= q);",
                                   ["test_filtered_acceptance_rate_is_one_minus_tvd"]),
    "saguaro_accept_transposed": ("int holds = (p > 0) && ((double)r[i] * q <= p);",
                                  "int holds = (p > 0) && ((double)r[i] * p <= q);",
                                  ["test_saguaro_preserves_the_target_distribution"]),
    "saguaro_bonus_wrong_row": ("const float *last = tgt + (size_t)gamma * V;",
                                "const float *last = tgt + (size_t)(gamma - 1) * V;",
                                ["test_saguaro_C1_is_plain_chain"]),
    "saguaro_trial_accept_inverted": ("if (q <= (1.0 - v) * p) {\n                emitted = x;",
                                      "if (p <= (1.0 - v) * q) {\n                emitted = x;",
                                      ["test_saguaro_preserves_the_target_distribution"]),
    "saguaro_weight_inverted": ("return exp((double)z[x] / T - M) * (inS[x] ? invC : 1.0) / S;",
                                "return exp((double)z[x] / T - M) * (inS[x] ? 1.0 / invC : 1.0) / S;",
                                ["test_saguaro_draft_probabilities"]),
    "saguaro_normaliser_unweighted": ("exp((double)d[x] / T - M) * (inS[(size_t)i * V + x] ? invC : 1.0));",
                                      "exp((double)d[x] / T - M));",
                                      ["test_saguaro_draft_probabilities"]),
    "tree_shift_by_one": ("            s += Nm;\n", "            s += 1.0;\n", ["test_tree_root_acceptance_closed_form"]),
    "tree_residual_unnormalised": ("(px - s * qx) / Nm : 0.0);", "(px - s * qx) : 0.0);",
                                   ["test_tree_root_acceptance_closed_form"]),
    "tree_greedy_last_child": ("if (parent[c] == u && tok[c] == a) { next = c; break; }",
                               "if (parent[c] == u && tok[c] == a) { next = c; }",
                               ["test_tree_greedy_walk"]),
    "tree_bonus_wrong_row": ("        if (nkids == 0) { /* leaf: the bonus token from p_u */\n",
                             "        if (nkids == 0) { /* leaf: the bonus token from p_u */\n"
                             "            for (int x = 0; x < V; ++x) w[x] = prob(tgt, x, T, Mt, St);\n",
                             ["test_tree_path_is_the_chain"]),
    "tree_draw_ignores_shift": ("emitted = tree_trials(w, du, V, T, Md, Sd, s, seq_key,",
                                "emitted = tree_trials(w, du, V, T, Md, Sd, 1.0, seq_key,",
                                ["test_tree_first_token_is_exact"]),
    "accept_margin_transposed": ("double m = (q > 0) ? fabs((double)r[i] - p / q) : INFINITY;",
                                 "double m = (q > 0) ? fabs((double)r[i] - q / p) : INFINITY;",
                                 ["test_accept_margin_is_the_ratio_gap"]),
    "accept_margin_off_path": ("        if (i < k) { /* decisions up to the first rejection decide the output */\n"
                               "            double m = (q > 0) ? fabs((double)r[i] - p / q) : INFINITY;\n"
                               "            note_margin(&margin, m);\n",
                               "        double m = (q > 0) ? fabs((double)r[i] - p / q) : INFINITY;\n"
                               "        note_margin(&margin, m);\n"
                               "        if (i < k) { /* decisions up to the first rejection decide the output */\n",
                               ["test_margin_counts_only_the_decisions_on_the_output_path"]),
    "race_margin_linear_gap": ("else m = log(a2) - log(a1);", "else m = a2 - a1;",
                               ["test_race_margin_is_the_log_gap_of_the_two_earliest_arrivals"]),
    "trial_margin_wrong_side": ("note_margin(&margin, fabs((1.0 - v) - q / p));\n            if (q <= (1.0 - v) * p) { emitted = x; break; }",
                                "note_margin(&margin, fabs(v - q / p));\n            if (q <= (1.0 - v) * p) { emitted = x; break; }",
                                ["test_trial_margin_is_the_gap_of_one_minus_v_to_q_over_p"]),
    "accept_ignores_draft": ("int acc = (p > 0) && ((double)r[i] * q <= p);",
                             "int acc = (p > 0) && ((double)r[i] <= p);",
                             ["test_enumeration_designed_thresholds"]),
    "fanout_formula": ("return (double)F0 * pow(a, (double)k / (1.0 + r));", "return (double)F0 * pow(a, (double)k / r);",
                       ["test_fanout_sizes_golden"]),
}


def _calls(name):
    fn = getattr(pins, name, None) or getattr(enum, name)
    if name == "test_enumeration_designed_thresholds":
        return [lambda: fn(1, 4, 0), lambda: fn(2, 3, 2)]
    if name == "test_enumeration_arbitrary_pairs":
        return [lambda: fn(1, 5, 4096, 11)]
    if name == "test_trial_acceptance_enumerated":
        return [lambda: fn(5, 21)]
    if name == "test_acceptance_rate_is_one_minus_tvd":
        return [lambda: fn(1.0), lambda: fn(0.6)]
    if name == "test_fanout_vs_numpy_lexsort":
        return [lambda: fn(None), lambda: fn(8)]
    if name == "test_filter_row_vs_torch_topk_softmax":
        return [lambda: fn(1.0)]
    if name == "test_tree_root_acceptance_closed_form":
        return [lambda: fn(2), lambda: fn(4)]
    if name == "test_tree_first_token_is_exact":
        return [lambda: fn(3), lambda: fn(4)]
    if name == "test_saguaro_draft_probabilities":
        return [lambda: fn(2.0), lambda: fn(8.0)]
    if name == "test_filtered_acceptance_rate_is_one_minus_tvd":
        return [lambda: fn(10), lambda: fn(40)]
    return [fn]


# A planted mistake can leave a chi-square cell with no expected mass (scipy
# then warns of a division by zero); the pin fails all the same.
@pytest.mark.filterwarnings("ignore:invalid value encountered in divide:RuntimeWarning")
@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tmp_path, monkeypatch):
    old, new, tests = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found for {mutant}"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-o", str(lib), str(msrc), "-lm"])
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: str(lib))
    caught = []
    for name in tests:
        for call in _calls(name):
            try:
                call()
            except AssertionError:
                caught.append(name)
                break
    monkeypatch.setattr(oracle, "_lib", None)
    assert caught, f"mutant {mutant} survived {tests}"
