"""The oracle's pins must catch plausible mistakes.

Each case copies oracle/sd_oracle.c, plants one mistake (a wrong comparison,
a flipped sign, a dropped term, an off-by-one index, swapped operands),
builds it with gcc and runs the pins of tests/test_oracle_pins.py that
should notice.  The test passes only if at least one of them fails on the
planted mistake.  Nothing here touches a GPU.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = [
    # (id, text in sd_oracle.c, replacement, nth occurrence, pins)
    ("accept_direction", "ok = (r <= rho);", "ok = (r >= rho);", 1,
     ["test_beta_closed_form_and_empirical_accept_rate"]),
    ("ratio_swapped", "double rho = accept_ratio(p[x], q[x]);",
     "double rho = accept_ratio(q[x], p[x]);", 1,
     ["test_beta_closed_form_and_empirical_accept_rate",
      "test_worked_residual_examples"]),
    ("residual_sign", "double d = p[j] - q[j];", "double d = q[j] - p[j];", 1,
     ["test_first_token_marginal_is_p", "test_worked_residual_examples"]),
    ("residual_no_clamp", "w[j] = d > 0.0 ? d : 0.0;", "w[j] = d;", 1,
     ["test_worked_residual_examples", "test_first_token_marginal_is_p"]),
    ("temperature_dropped",
     "p[j] = exp((logit_at(base, dtype, off + (size_t)j) - m) / T);",
     "p[j] = exp((logit_at(base, dtype, off + (size_t)j) - m));", 1,
     ["test_first_token_marginal_is_p"]),
    ("bonus_row_off_by_one",
     "if (!softmax_row(target, dtype, ((size_t)b * G1 + gamma) * V, V, T,",
     "if (!softmax_row(target, dtype, ((size_t)b * G1 + gamma - 1) * V, V, T,",
     1, ["test_bruteforce_enumeration",
         "test_second_token_conditional_with_prefix_dependent_target"]),
    ("cdf_unnormalised", "double target = u * N;", "double target = u;", 1,
     ["test_worked_residual_examples", "test_first_token_marginal_is_p"]),
    ("residual_wrong_position_draft",
     "!softmax_row(draft, dtype, ((size_t)b * gamma + i) * V, V, T, q)",
     "!softmax_row(draft, dtype, ((size_t)b * gamma + 0) * V, V, T, q)", 1,
     ["test_second_token_conditional_with_prefix_dependent_target",
      "test_bruteforce_enumeration"]),
    ("greedy_tie_highest", "if (z > bv) { bv = z; best = j; }",
     "if (z >= bv) { bv = z; best = j; }", 1,
     ["test_greedy_is_id_equality_with_argmax"]),
    ("kcand_tie_highest_k", "if (n > best_n) { best_n = n; best_k = k; }",
     "if (n >= best_n) { best_n = n; best_k = k; }", 1,
     ["test_kcand_selection_is_max_streak_lowest_k"]),
    ("kcand_shared_draft_row_wrong",
     "!softmax_row(draft, dtype, DROW(b, j), V, T, q)) {",
     "!softmax_row(draft, dtype, DROW(b, 0), V, T, q)) {", 1,
     ["test_kcand_max_streak_law_bruteforce"]),
    ("tree_no_residual_update", "p[j] = d > 0.0 ? d : 0.0;\n            S += p[j];",
     "S += (d > 0.0 ? d : 0.0);", 1,
     ["test_tree_iid_siblings_lossless"]),
    ("tree_final_uniform_slot", "sample_icdf(p, V, (double)U[0],",
     "sample_icdf(p, V, (double)U[1],", 1,
     ["test_tree_chain_equals_linear", "test_tree_iid_siblings_lossless"]),
    ("fanout_exponent", "w[k] = pow(a, (double)k / (1.0 + r));",
     "w[k] = pow(a, (double)k / r);", 1,
     ["test_fanout_schedule_golden_and_theorem12"]),
    ("fanout_cap_sign",
     "pow(1.0 - a, -1.0 / (1.0 + r));", "pow(1.0 - a, 1.0 / (1.0 + r));", 1,
     ["test_fanout_schedule_golden_and_theorem12"]),
    ("hits_position_off_by_one", "for (int k = 0; k < n; ++k) off += F[k];",
     "for (int k = 0; k <= n && k < K; ++k) off += F[k];", 1,
     ["test_cache_hits_golden"]),
    ("hits_outcome_token_off_by_one",
     "const int32_t t = tokens[(size_t)b * (K + 1) + n];",
     "const int32_t t = tokens[(size_t)b * (K + 1) + (n > 0 ? n - 1 : 0)];",
     1, ["test_cache_hits_golden",
         "test_cache_hit_rate_equals_top_f_mass_when_p_equals_q"]),
    ("flag_without_margin", "if (m < ORC_BAND) ++*flagged;", "++*flagged;",
     1, ["test_accept_test_counts_and_flags_planted"]),
    ("flag_band_too_narrow", "if (m < ORC_BAND) ++*flagged;",
     "if (m < 1e-6) ++*flagged;", 1,
     ["test_accept_test_counts_and_flags_planted"]),
    ("nucleus_range_band_sign", "if (f < top_p + ORC_BAND) hi = i + 1;",
     "if (f < top_p - ORC_BAND) hi = i + 1;", 1,
     ["test_filtered_keep_ranges_and_forced_cuts"]),
    ("nucleus_forced_count_ignored",
     "if (forced >= 1) keep = forced < k ? forced : k;",
     "if (forced >= 1 && 0) keep = forced < k ? forced : k;", 1,
     ["test_filtered_keep_ranges_and_forced_cuts"]),
    ("nucleus_one_too_many", "if (f < top_p) keep = i + 1;",
     "if (f < top_p) keep = i + 2 < k ? i + 2 : k;", 1,
     ["test_filtered_sampling_golden"]),
    ("nucleus_not_renormalised_over_top_k", "double f = before / mk;",
     "double f = before;", 1,
     ["test_filtered_sampling_golden"]),
    ("filter_kept_not_renormalised",
     "for (int i = 0; i < keep; ++i) kept[i] = p[e[i].idx] / S;",
     "for (int i = 0; i < keep; ++i) kept[i] = p[e[i].idx];", 1,
     ["test_filtered_sampling_golden",
      "test_filtered_first_token_marginal_is_filtered_p"]),
    ("topk_tie_order", "return (a->idx > b->idx) - (a->idx < b->idx);",
     "return (a->idx < b->idx) - (a->idx > b->idx);", 1,
     ["test_fanout_topk_against_stable_sort_and_ties"]),
    ("det_accept_direction", "if ((double)U[v] <= rho) { next = v; break; }",
     "if ((double)U[v] >= rho) { next = v; break; }", 1,
     ["test_tree_det_golden", "test_tree_det_topk_siblings_lossless"]),
    ("det_rejected_token_kept", "p[x] = 0.0;", "p[x] = p[x];", 1,
     ["test_tree_det_golden", "test_tree_det_quadrature_bruteforce"]),
    ("det_not_renormalised", "for (int j = 0; j < V; ++j) p[j] /= S;",
     "for (int j = 0; j < V; ++j) p[j] /= 1.0;", 2,
     ["test_tree_det_topk_siblings_lossless",
      "test_tree_det_quadrature_bruteforce"]),
    ("det_child_reads_root_row",
     "size_t off = ((size_t)b * N + cur) * (size_t)V;",
     "size_t off = ((size_t)b * N + 0) * (size_t)V;", 2,
     ["test_tree_det_two_level_joint_is_p", "test_tree_det_golden"]),
    ("trie_duplicate_below_its_twin", "dup[v] = 1;\n          tr[v]",
     "dup[v] = 1; par[v] = same;\n          tr[v]", 1,
     ["test_kcand_trie_golden",
      "test_kcand_trie_lossless_first_and_second_token"]),
    ("trie_target_row_off_by_one", "tr[v] = k * G1 + j + 1;",
     "tr[v] = k * G1 + j;", 1,
     ["test_kcand_trie_one_candidate_equals_linear",
      "test_kcand_trie_lossless_first_and_second_token"]),
    ("trie_final_uniform_slot", "U[0] = u[gamma];", "U[0] = u[0];", 1,
     ["test_kcand_trie_one_candidate_equals_linear"]),
    ("presto_rho_sign",
     "double s = lq[j] + (lambda == 0.0 ? 0.0 : lambda * r);",
     "double s = lq[j] - (lambda == 0.0 ? 0.0 : lambda * r);", 1,
     ["test_presto_golden", "test_presto_score_is_the_kl_minimiser"]),
    ("presto_path_score_dropped", "all[nc].s = fs[w] + row[i].s;",
     "all[nc].s = row[i].s;", 1,
     ["test_presto_golden", "test_presto_construction_invariants"]),
    ("presto_parent_slot", "parent[v] = old_fn[all[i].w];",
     "parent[v] = old_fn[0];", 1,
     ["test_presto_golden", "test_presto_construction_invariants"]),
    ("scan_reads_past_rejection", "if (!ok) { rejected = 1; break; }",
     "if (!ok) { rejected = 1; continue; }", 1,
     ["test_rows_after_the_decision_are_never_read"]),
    ("greedy_scan_reads_past_rejection", "if (!ok) break;",
     "if (!ok) continue;", 1,
     ["test_rows_after_the_decision_are_never_read"]),
    ("kcand_scan_reads_past_rejection", "if (!ok) break;",
     "if (!ok) continue;", 2,
     ["test_kcand_rows_after_each_scan_are_never_read"]),
    ("tree_reads_leaf_draft_row",
     "if (has_child && !softmax_row(draft, dtype, off, V, T, q)) {",
     "if (!softmax_row(draft, dtype, off, V, T, q)) {", 1,
     ["test_tree_rows_off_the_path_are_never_read"]),
    ("masked_token_invalidates_row", "if (isnan(z) || z == INFINITY) return 0;",
     "if (isnan(z) || isinf(z)) return 0;", 1,
     ["test_minus_infinity_is_a_token_of_probability_zero"]),
    ("softmax_no_max_subtraction",
     "p[j] = exp((logit_at(base, dtype, off + (size_t)j) - m) / T);",
     "p[j] = exp(logit_at(base, dtype, off + (size_t)j) / T);", 1,
     ["test_softmax_shift_invariance"]),
    ("fork_floor", "int k = k_max - (int)ceil(y);",
     "int k = k_max - (int)floor(y);", 1,
     ["test_branch_fork_golden"]),
    ("fork_confidence_complement", "qx = (x >= 0 && x < V) ? q[x] : 0.0;",
     "qx = (x >= 0 && x < V) ? 1.0 - q[x] : 0.0;", 1,
     ["test_branch_fork_golden",
      "test_branch_fork_topk_is_a_stable_sort_and_k_law"]),
]


def _build_mutant(src, pattern, repl, nth, outdir, name):
    idx = -1
    for _ in range(nth):
        idx = src.index(pattern, idx + 1)
    mutated = src[:idx] + repl + src[idx + len(pattern):]
    cpath = os.path.join(outdir, name + ".c")
    so = os.path.join(outdir, name + ".so")
    with open(cpath, "w") as f:
        f.write(mutated)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared",
                           "-ffp-contract=off", cpath, "-o", so, "-lm"])
    return so


def _run_pin(name):
    fn = getattr(pins, name)
    params = {
        "test_first_token_marginal_is_p": [dict(T=1.0), dict(T=0.7)],
        "test_bruteforce_enumeration": [dict(V=3, gamma=3),
                                        dict(V=5, gamma=2)],
        "test_tree_chain_equals_linear": [dict(T=1.0)],
        "test_kcand_trie_one_candidate_equals_linear": [dict(T=1.0)],
        "test_softmax_shift_invariance": [dict(T=1.0)],
        "test_rows_after_the_decision_are_never_read": [dict(T=1.0),
                                                        dict(T=0.0)],
        "test_minus_infinity_is_a_token_of_probability_zero": [dict(T=1.0)],
        "test_kcand_rows_after_each_scan_are_never_read": [dict(T=1.0),
                                                           dict(T=0.0)],
        "test_tree_rows_off_the_path_are_never_read": [
            dict(rule="sibling", T=1.0), dict(rule="det", T=1.0)],
        "test_filtered_first_token_marginal_is_filtered_p": [
            dict(top_k=5, top_p=1.0), dict(top_k=4, top_p=0.6)],
    }.get(name, [dict()])
    for kw in params:
        fn(**kw)


@pytest.mark.parametrize("mid,pattern,repl,nth,catchers", MUTANTS,
                         ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mid, pattern, repl, nth, catchers):
    with open(oracle._SRC) as f:
        src = f.read()
    assert pattern in src, "mutation site vanished: " + mid
    with tempfile.TemporaryDirectory() as d:
        so = _build_mutant(src, pattern, repl, nth, d, mid)
        caught = []
        with oracle.swapped_library(so):
            for name in catchers:
                try:
                    _run_pin(name)
                except AssertionError:
                    caught.append(name)
    assert caught, "no pin caught the planted mistake " + mid
