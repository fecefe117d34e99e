"""Pins for the oracle's one-level draft tree expansion (CPU only).

Expected values come from library routines and brute force: torch's stable sort (descending logit, lower
token id first) and log_softmax in float64 for the per-row proposals; and, when k >= n_keep, a brute-force
selection over EVERY (frontier slot, token) pair of the level, which must agree with the two-stage
top-k-then-prune result.  A level-by-level build must reproduce the budgeted level sizes and a valid tree.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def logits_f64(e):
    return W.decode_f32(e.logits, e.logit_dt).astype(np.float64)


def run(e):
    r = oracle.tree_expand(e.logits, e.front_score, V=e.V, k=e.k, n_keep=e.n_keep, logit_dt=e.logit_dt)
    assert r["rc"] == 0
    return r


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V,k,ties", [(50, 4, 0), (1000, 8, 0), (3000, 3, 2), (64, 16, 5)])
def test_row_proposals_match_stable_sort_and_log_softmax(dt, V, k, ties):
    e = W.make_expand(1, B=3, n_front=5, V=V, k=k, n_keep=7, logit_dt=dt, ties=ties)
    r = run(e)
    z = torch.from_numpy(logits_f64(e))
    order = torch.sort(-z, dim=-1, stable=True).indices[..., :k].numpy()
    lp = torch.log_softmax(z, dim=-1)
    np.testing.assert_array_equal(r["topk_token"], order)
    np.testing.assert_allclose(r["topk_logprob"], np.take_along_axis(lp.numpy(), order, -1), rtol=0, atol=1e-12)
    assert (r["status"] == 0).all()


@pytest.mark.parametrize("n_front,k,n_keep", [(1, 4, 4), (4, 3, 3), (12, 5, 5), (24, 2, 2), (6, 8, 1)])
def test_selection_equals_brute_force_over_all_children(n_front, k, n_keep):
    e = W.make_expand(7, B=4, n_front=n_front, V=400, k=k, n_keep=n_keep, logit_dt="bf16")
    r = run(e)
    z = logits_f64(e)
    lp = torch.log_softmax(torch.from_numpy(z), dim=-1).numpy()
    for b in range(e.B):
        # every child of the level: score, frontier slot, token; ranked by score, slot, then token
        cand = [(-(float(e.front_score[b, s]) + lp[b, s, t]), s, t) for s in range(n_front) for t in range(e.V)]
        cand.sort()
        kept = cand[:n_keep]
        # listed by (slot, position in the slot's row order: larger logit first, lower token first)
        kept.sort(key=lambda c: (c[1], -z[b, c[1], c[2]], c[2]))
        np.testing.assert_array_equal(r["child_parent"][b], [c[1] for c in kept])
        np.testing.assert_array_equal(r["child_token"][b], [c[2] for c in kept])
        np.testing.assert_allclose(r["child_score"][b], [-c[0] for c in kept], rtol=0, atol=1e-12)


def test_children_are_consistent_with_row_proposals():
    e = W.make_expand(9, B=5, n_front=12, V=2000, k=2, n_keep=17, logit_dt="bf16")
    r = run(e)
    for b in range(e.B):
        par = r["child_parent"][b]
        assert (np.diff(par) >= 0).all()
        for i, s in enumerate(par):
            ranks = np.nonzero(r["topk_token"][b, s] == r["child_token"][b, i])[0]
            assert len(ranks) == 1
            assert r["child_score"][b, i] == pytest.approx(e.front_score[b, s] + r["topk_logprob"][b, s, ranks[0]],
                                                            abs=1e-12)
        # survivors beat every dropped candidate
        all_scores = (e.front_score[b][:, None].astype(np.float64) + r["topk_logprob"][b]).ravel()
        kept = np.sort(r["child_score"][b])
        assert kept[0] >= np.sort(all_scores)[::-1][e.n_keep - 1] - 1e-12


def test_level_by_level_build_gives_the_budgeted_tree():
    T, branching = 60, (4, 3, 2, 2, 1, 1)
    levels = W.expansion_levels(T, branching)
    B = 3
    parent = [[-1] for _ in range(B)]
    front_ids = [[0] for _ in range(B)]
    score = np.zeros((B, 1), np.float32)
    for d, (n_front, k, n_keep) in enumerate(levels):
        e = W.make_expand(100 + d, B=B, n_front=n_front, V=500, k=k, n_keep=n_keep, logit_dt="bf16")
        e.front_score = score
        r = run(e)
        new_ids = []
        for b in range(B):
            ids = []
            for s in r["child_parent"][b]:
                parent[b].append(front_ids[b][s])
                ids.append(len(parent[b]) - 1)
            new_ids.append(ids)
        front_ids = new_ids
        score = r["child_score"].astype(np.float32)
    for b in range(B):
        p = np.asarray(parent[b], np.int32)
        assert len(p) == T and oracle.tree_check(p) == 0
        st, depth = oracle.tree_depth(p)
        assert np.bincount(depth).tolist() == W.level_sizes(T, branching)


def test_nonfinite_rows_fail_their_request_only():
    e = W.make_expand(3, B=3, n_front=2, V=100, k=2, n_keep=3, logit_dt="f32")
    e.logits = e.logits.copy()
    e.front_score = e.front_score.copy()
    e.logits[0, 1, 7] = np.inf
    e.front_score[2, 0] = np.nan
    r = run(e)
    assert list(r["status"]) == [5, 0, 5]
    assert (r["child_token"][[0, 2]] == -1).all() and (r["child_token"][1] >= 0).all()
