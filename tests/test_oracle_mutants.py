"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each one.

Each mutant is an edited copy of the oracle's C source compiled into a temporary library
(on the CPU; nothing here touches the product or a GPU).  The pins of
test_oracle_visibility / test_oracle_rope / test_oracle_attn are then run against the
mutant, and at least one of them must fail.  This shows the pins are not vacuous: a
dropped term, a wrong sign, an off-by-one index or a wrong exponent would not go
unnoticed.
"""
import pytest

import oracle
from tests import test_oracle_accept as TAC
from tests import test_oracle_tree_build as TTB
from tests import test_oracle_attn as TA
from tests import test_oracle_rope as TR
from tests import test_oracle_visibility as TV

MUTANTS = {
    "rope_sign": ("const double y0 = x0 * c - x1 * s;", "const double y0 = x0 * c + x1 * s;"),
    "rope_freq": ("(2.0 * (double)k) / (double)d_rope", "((double)k) / (double)d_rope"),
    "rope_pos_no_prefix": ("const double pos = (double)prefix_len[b] + (double)depth[r];",
                           "const double pos = (double)depth[r];"),
    "score_drops_rope": ("for (int r = 0; r < DR; ++r) dot += (double)qR[r] * (double)kr[r];",
                         "(void)kr;"),
    "score_no_scale": ("s[j] = scale * dot;", "s[j] = dot;"),
    "mask_tree_bit_off_by_one": ("ok[j] = (j < P) ? 1 : vrow[j - P];",
                                 "ok[j] = (j < P) ? 1 : vrow[(j - P + 1) % Q];"),
    "mask_drops_last_prefix_key": ("ok[j] = (j < P) ? 1 : vrow[j - P];",
                                   "ok[j] = (j + 1 < P) ? 1 : (j < P ? 0 : vrow[j - P]);"),
    "mask_all_tree_visible": ("ok[j] = (j < P) ? 1 : vrow[j - P];", "ok[j] = 1;"),
    "lse_without_max": ("lse[qrow] = m + log(l);", "lse[qrow] = log(l);"),
    "no_normalisation": ("const double p = exp(s[j] - m) / l;",
                         "const double p = exp(s[j] - m);"),
    "vis_misses_self": ("int k = i, steps = 0;",
                        "int k = i ? par[i] : 0, steps = i ? 1 : 0;"),
    "vis_depth_off_by_one": ("depth[(int64_t)b * Q + i] = steps;",
                             "depth[(int64_t)b * Q + i] = steps + 1;"),
    "tree_slot_wrong": ("tvo_row(&c, b, (int64_t)prefix_len[b] + i)",
                        "tvo_row(&c, b, (int64_t)prefix_len[b] + i - 1 + (i == 0))"),
    "value_uses_kpe_row": ("const float* ck = c_kv + tvo_row(&c, b, j) * ckv_stride;",
                           "const float* ck = c_kv + tvo_row(&c, b, j > 0 ? j - 1 : 0) * ckv_stride;"),
}

PINS = [
    TV.test_brute_force_all_trees_q6, TV.test_chain_is_lower_triangular,
    TV.test_star_sees_root_and_self,
    TR.test_position_zero_is_identity, lambda: TR.test_matches_complex_multiplication(64),
    TR.test_d2_is_plane_rotation, TR.test_pair0_rotates_by_position_radians_and_norm_kept,
    TR.test_golden_worked_example,
    lambda: TA.test_matches_sdpa_with_networkx_mask(True, "random"),
    TA.test_chain_tree_is_causal_attention, TA.test_root_row_and_q1_are_single_query_decode,
    TA.test_zero_query_is_mean_and_lse_is_log_count,
    TA.test_dominant_score_selects_row_and_ones_give_one, TA.test_golden_worked_example,
    TA.test_full_step_chain_equals_rope_then_causal_attention,
]


# planted mistakes in the acceptance / compaction oracle (tree_oracle.c)
TREE_MUTANTS = {
    "argmax_ties_to_largest": ("if (x[v] > x[best]) best = v;", "if (x[v] >= x[best]) best = v;"),
    "accept_compares_child_target": ("if (par[c] == cur && tok[c] == tgt[cur]) {",
                                     "if (par[c] == cur && tok[c] == tgt[c]) {"),
    "accept_any_node_not_child": ("if (par[c] == cur && tok[c] == tgt[cur]) {",
                                  "if (c > cur && tok[c] == tgt[cur]) {"),
    "accept_largest_child": ("next = c; /* the smallest qualifying child */\n          break;",
                             "next = c; /* the smallest qualifying child */"),
    "bonus_from_root": ("emit[a] = tgt[cur]; /* bonus token */", "emit[a] = tgt[0];"),
    "compact_dst_off_by_one": ("b, P + d);", "b, P + d + 1);"),
    "compact_prefix_misses_root": ("new_prefix_len[b] = (int32_t)(P + 1 + a);",
                                   "new_prefix_len[b] = (int32_t)(P + a);"),
    "compact_skips_k_pe": ("memcpy(k_pe + dst * kpe_stride, k_pe + src * kpe_stride,",
                           "if (0) memcpy(k_pe + dst * kpe_stride, k_pe + src * kpe_stride,"),
}

# planted mistakes in the best-first tree builder (tree_oracle.c)
BUILD_MUTANTS = {
    "ties_deeper_first": ("if (a->depth != b->depth) return a->depth < b->depth;",
                          "if (a->depth != b->depth) return a->depth > b->depth;"),
    "ties_path_reversed": ("if (a->path[i] != b->path[i]) return a->path[i] < b->path[i];",
                           "if (a->path[i] != b->path[i]) return a->path[i] > b->path[i];"),
    "child_logprob_off_by_one_depth": ("c.score = w.score + lpb[(int64_t)w.depth * K + k];",
                                       "c.score = w.score + lpb[(int64_t)(w.depth - 1) * K + k];"),
    "only_first_child": ("        for (int k = 0; k < K; ++k) {\n          tro_cand c = w;",
                         "        for (int k = 0; k < 1; ++k) {\n          tro_cand c = w;"),
    "parent_is_grandparent": ("          c.parent = i;", "          c.parent = w.parent;"),
    "token_from_wrong_depth": ("tks[i] = tkb[(int64_t)(w.depth - 1) * K + w.rank];",
                               "tks[i] = tkb[(int64_t)(w.depth > 1 ? w.depth - 2 : 0) * K + w.rank];"),
}

BUILD_PINS = [
    lambda: TTB.test_brute_force(3, 3, 10), lambda: TTB.test_brute_force(4, 2, 15),
    TTB.test_ties_follow_depth_then_rank_path, TTB.test_closed_forms, TTB.test_structure,
    TTB.test_golden_worked_example,
]


@pytest.mark.parametrize("name", sorted(BUILD_MUTANTS))
def test_build_pins_catch_planted_mistake(name, tmp_path):
    src = oracle.source_text("tree")
    old, new = BUILD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found for {name}"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  which="tree")
    failures = 0
    with oracle.use_library(path):
        for pin in BUILD_PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError):
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


def test_unmutated_build_oracle_passes_all_pins():
    for pin in BUILD_PINS:
        pin()


TREE_PINS = [
    TAC.test_argmax_matches_numpy_and_takes_smallest_index_on_ties,
    TAC.test_brute_force_all_six_node_trees, TAC.test_chain_accepts_up_to_first_mismatch,
    TAC.test_star_accepts_at_most_one_and_duplicate_siblings_take_smallest_index,
    TAC.test_speculative_output_equals_autoregressive_output, TAC.test_golden_worked_example,
    lambda: TAC.test_compaction_equals_out_of_place_gather(False),
    lambda: TAC.test_compaction_equals_out_of_place_gather(True),
]


@pytest.mark.parametrize("name", sorted(TREE_MUTANTS))
def test_tree_pins_catch_planted_mistake(name, tmp_path):
    src = oracle.source_text("tree")
    old, new = TREE_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found for {name}"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"),
                                  which="tree")
    failures = 0
    with oracle.use_library(path):
        for pin in TREE_PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError):
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


def test_unmutated_tree_oracle_passes_all_pins():
    for pin in TREE_PINS:
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = oracle.source_text()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor not found for {name}"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    failures = 0
    with oracle.use_library(path):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError):
                failures += 1
    assert failures > 0, f"no pin caught mutant {name}"


def test_unmutated_oracle_passes_all_pins():
    for pin in PINS:
        pin()
