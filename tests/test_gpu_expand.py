"""GPU parity of sv_tree_expand against the oracle.

Integer outputs are compared exactly where they are unique: the proposed tokens of every row (decided by
comparing logits, no rounding involved) and, whenever the oracle's scores separate the n_keep-th and the
next candidate by more than the float32 error of a log-probability, the surviving children.  Closer than
that, several selections are correct, so the test checks that the GPU's survivors are a valid choice under
the oracle's exact scores.  Log-probabilities and scores must be within 1e-4 (float32 logsumexp over up to
152K terms against float64)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

TOL = 1e-4


def run_expand(e):
    B, NF, k, nk = e.B, e.n_front, e.k, e.n_keep
    i32 = dict(dtype=torch.int32, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    out = dict(topk_token=torch.full((B, NF, k), -9, **i32), topk_logprob=torch.full((B, NF, k), float("nan"), **f32),
               child_parent=torch.full((B, max(nk, 1)), -9, **i32), child_token=torch.full((B, max(nk, 1)), -9, **i32),
               child_score=torch.full((B, max(nk, 1)), float("nan"), **f32), status=torch.full((B,), -9, **i32))
    sv.tree_expand(dev(e.logits).view(B, NF, e.V), dev(e.front_score), k, nk, out["topk_token"], out["topk_logprob"],
                   out["child_parent"], out["child_token"], out["child_score"], status=out["status"])
    torch.cuda.synchronize()
    res = {kk: v.cpu().numpy() for kk, v in out.items()}
    for kk in ("child_parent", "child_token", "child_score"):
        res[kk] = res[kk][:, :nk]
    return res


def check(e):
    ref = oracle.tree_expand(e.logits, e.front_score, V=e.V, k=e.k, n_keep=e.n_keep, logit_dt=e.logit_dt)
    assert ref["rc"] == 0
    got = run_expand(e)
    np.testing.assert_array_equal(got["status"], ref["status"])
    np.testing.assert_array_equal(got["topk_token"], ref["topk_token"])
    ok = ref["status"] == 0
    np.testing.assert_allclose(got["topk_logprob"][ok], ref["topk_logprob"][ok], rtol=0, atol=TOL)
    assert (got["topk_logprob"][~ok] == -np.inf).all() and (got["child_token"][~ok] == -1).all()
    exact = 0
    for b in np.nonzero(ok)[0]:
        # the oracle's float64 score of every candidate (slot, rank)
        cand = e.front_score[b][:, None].astype(np.float64) + ref["topk_logprob"][b]
        flat = np.sort(cand.ravel())[::-1]
        nk = e.n_keep
        gap = np.inf if nk in (0, flat.size) else flat[nk - 1] - flat[nk]
        if gap > 4 * TOL:
            np.testing.assert_array_equal(got["child_parent"][b], ref["child_parent"][b])
            np.testing.assert_array_equal(got["child_token"][b], ref["child_token"][b])
            np.testing.assert_allclose(got["child_score"][b], ref["child_score"][b], rtol=0, atol=TOL)
            exact += 1
        else:
            # a valid selection: distinct candidates in (slot, rank) order, none beaten by a dropped one
            par, tok = got["child_parent"][b], got["child_token"][b]
            ranks = np.array([int(np.nonzero(ref["topk_token"][b, s] == t)[0][0]) for s, t in zip(par, tok)])
            keys = par * e.k + ranks
            assert (np.diff(keys) > 0).all()
            kept = cand.ravel()[keys]
            dropped = np.delete(cand.ravel(), keys)
            assert dropped.size == 0 or kept.min() >= dropped.max() - 4 * TOL
            np.testing.assert_allclose(got["child_score"][b], kept, rtol=0, atol=TOL)
    return exact


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V", [40, 1000, 1001, 40000])
@pytest.mark.parametrize("n_front,k,n_keep", [(1, 4, 4), (4, 3, 12), (12, 2, 17), (24, 2, 17), (64, 16, 100),
                                              (7, 1, 3), (5, 5, 0)])
def test_expand_parity(dt, V, n_front, k, n_keep):
    if k > V:
        pytest.skip("k > V")
    e = W.make_expand(V + 13 * n_front + k, B=5, n_front=n_front, V=V, k=k, n_keep=n_keep, logit_dt=dt)
    check(e)


@pytest.mark.parametrize("ties", [1, 3])
@pytest.mark.parametrize("V", [64, 5000])
def test_expand_equal_logits_take_the_lower_token(ties, V):
    e = W.make_expand(ties * 7 + V, B=4, n_front=6, V=V, k=4, n_keep=9, logit_dt="bf16", ties=ties)
    check(e)


def test_expand_nonfinite_fails_only_its_request():
    e = W.make_expand(3, B=4, n_front=3, V=3000, k=2, n_keep=4, logit_dt="f32")
    e.logits = e.logits.copy()
    e.front_score = e.front_score.copy()
    e.logits[0, 2, 2999] = np.nan
    e.logits[1, 0, 5] = -np.inf
    e.front_score[3, 1] = np.inf
    got = run_expand(e)
    assert list(got["status"]) == [5, 5, 0, 5]
    check(e)


@pytest.mark.parametrize("level", range(6))
def test_expand_llama3_tree_levels_full_size(level):
    """Every level of the Llama3-shaped 60-node tree (4/3/2/2/1/1) at full size: 8 requests, V = 128256."""
    n_front, k, n_keep = W.expansion_levels(60, (4, 3, 2, 2, 1, 1))[level]
    e = W.make_expand(200 + level, B=8, n_front=n_front, V=128256, k=k, n_keep=n_keep, logit_dt="bf16")
    check(e)


def test_expand_qwen3_chain_step_full_size():
    """A lookahead step of the Qwen3-shaped chain batch: 32 requests, top-1 over V = 151936."""
    e = W.make_expand(300, B=32, n_front=1, V=151936, k=1, n_keep=1, logit_dt="bf16", sigma=2.5)
    check(e)
