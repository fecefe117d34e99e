"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle.c into a temporary directory, plants one mistake (a dropped term, a wrong index
or sign, an inverted tie rule), builds it, points the oracle binding at that build and asserts that the
named pin now FAILS.  The committed oracle.c is never modified.
"""
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_accept as TA
from tests import test_oracle_attn as TT
from tests import test_oracle_attn_bwd as TB
from tests import test_oracle_compact as TC
from tests import test_oracle_expand as TE
from tests import test_oracle_fp4 as TF
from tests import test_oracle_loss as TL

MUTANTS = {
    "gqa_head_modulo": (
        "int G = Hq / Hkv, hk = h / G;", "int G = Hq / Hkv, hk = h % Hkv;",
        lambda: TT.test_attn_matches_sdpa_with_dense_mask(TT.CASES[2])),
    "ancestors_without_self": (
        "for (int a = i; a >= 0; a = par[a]) on[a] = 1;", "for (int a = par[i]; a >= 0; a = par[a]) on[a] = 1;",
        TT.test_chain_equals_causal_attention),
    "no_max_subtraction_scale": (
        "s[j] = scale * acc;", "s[j] = acc;", TT.test_single_node_is_plain_decode_attention),
    "argmax_last_occurrence": (
        "if (best < 0 || z > bv) { bv = z; best = k; }", "if (best < 0 || z >= bv) { bv = z; best = k; }",
        TA.test_greedy_duplicate_siblings_first_wins_and_ties_take_first_index),
    "accept_with_p_not_p_over_q": (
        "u128 lhs = (u128)uniforms[(size_t)b * T + c] * wqx * Sres;",
        "u128 lhs = (u128)uniforms[(size_t)b * T + c] * Sq * Sres;",
        lambda: TA.test_prob_chain_marginals_follow_target(1.0)),
    "bonus_ignores_residual": (
        "wres[kk] = a > s ? (uint64_t)((a - s) / Sq) : 0u;", "(void)s; (void)a;",
        TA.test_onehot_tree_marginals_follow_target),
    "grad_drops_rejected_delta": (
        "g[tok[c]] += 1.0 / expm1(a);", "(void)a;", TL.test_gradient_matches_central_finite_differences),
    "rejection_term_uses_log_q": (
        "rej += -log1mexp(a);", "rej += a;",
        TL.test_binary_vocab_rejection_is_cross_entropy_on_the_other_token),
    "compact_destination_off_by_one": (
        "memcpy(base + (size_t)(1 + j) * row,", "memcpy(base + (size_t)j * row,",
        lambda: TC.test_path_nodes_see_a_causal_prefix_after_compaction("bf16", (3, 2, 2), 13)),
    "expand_ties_take_last_token": (
        "if (best < 0 || z > bz) { best = j; bz = z; }", "if (best < 0 || z >= bz) { best = j; bz = z; }",
        lambda: TE.test_row_proposals_match_stable_sort_and_log_softmax("bf16", 3000, 3, 2)),
    "expand_score_drops_parent_path": (
        "cand[s * k + q].score = (double)front_score[r] + ((double)bz - lse);",
        "cand[s * k + q].score = ((double)bz - lse);",
        lambda: TE.test_selection_equals_brute_force_over_all_children(12, 5, 5)),
    "attn_bwd_drops_delta": (
        "double ds = p * (dp - delta);", "double ds = p * dp;",
        lambda: TB.test_backward_matches_autograd_through_sdpa_with_dense_mask("f32", (3, 2, 2), 13)),
    "attn_bwd_value_grad_uses_q": (
        "dv[row * D + d] += p * g[d];", "dv[row * D + d] += p * qv[d];",
        TB.test_backward_matches_central_finite_differences),
    "fp4_high_nibble_first": (
        "unsigned kc = (k[(base + i) / 2] >> (4 * (i & 1))) & 15,",
        "unsigned kc = (k[(base + i) / 2] >> (4 * (1 - (i & 1)))) & 15,",
        lambda: TF.test_fp4_attention_equals_attention_on_independently_decoded_caches((3, 2, 2), 13)),
    "fx_poly_drops_cubic": (
        "p = fmaf(p, f, C_P3);", "p = fmaf(p, f, 0.0f);", TA.test_fx_exp2_polynomial_error_bound),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_catches_planted_mistake(name, tmp_path):
    old, new, pin = MUTANTS[name]
    src = (oracle.HERE / "oracle.c").read_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    (tmp_path / "oracle.c").write_text(src.replace(old, new))
    shutil.copy(oracle.HERE / "oracle.h", tmp_path / "oracle.h")
    so = tmp_path / f"mut_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fopenmp",
                    str(tmp_path / "oracle.c"), "-o", str(so), "-lm"], check=True)
    prev = oracle.use(so)
    try:
        with pytest.raises(AssertionError):
            pin()
    finally:
        oracle.restore(prev)
