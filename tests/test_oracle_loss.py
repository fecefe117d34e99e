"""Pins for the oracle's online-training loss (CPU only).

The loss is the acceptance cross-entropy on accepted draft tokens plus the rejection term
-log(1 - q(token)) on rejected ones, averaged over the N*(T-1) non-root nodes.  Checked against central
finite differences (fp64, V=8), the zero row-sum of a softmax gradient, torch's cross_entropy when no
branch is rejected, and the V=2 identity -log(1 - q_x) = -log q_other.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def small_batch(seed, N=3, T=9, V=8, tree=(2, 2, 2)):
    lb = W.make_loss(seed, N=N, T=T, V=V, tree=tree, accept_frac=0.45)
    z = W.bf16_to_f32(lb.logits).astype(np.float64)
    return lb, z


def test_gradient_matches_central_finite_differences():
    lb, z = small_batch(1)
    res = oracle.loss_f64(z, lb.tokens, lb.parent, lb.labels, V=lb.V)
    assert (res["status"] == 0).all()
    h = 1e-6
    num = np.zeros_like(z)
    for r in range(z.shape[0]):
        for k in range(z.shape[1]):
            zp = z.copy(); zp[r, k] += h
            zm = z.copy(); zm[r, k] -= h
            lp = oracle.loss_f64(zp, lb.tokens, lb.parent, lb.labels, V=lb.V, want_grad=False)["loss"]
            lm = oracle.loss_f64(zm, lb.tokens, lb.parent, lb.labels, V=lb.V, want_grad=False)["loss"]
            num[r, k] = (lp - lm) / (2 * h)
    np.testing.assert_allclose(res["grad"], num, atol=1e-8, rtol=1e-6)


def test_gradient_rows_sum_to_zero_and_leaves_are_zero():
    lb = W.make_loss(2, N=4, T=32, V=300, tree=(4, 3, 2, 1, 1))
    res = oracle.loss_w(lb)
    g = res["grad"]
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-14)
    has_child = np.zeros(lb.N * lb.T, bool)
    for n in range(lb.N):
        for c in range(1, lb.T):
            has_child[n * lb.T + lb.parent[n, c]] = True
    assert (g[~has_child] == 0).all() and (res["row_loss"][~has_child] == 0).all()
    assert np.abs(g[has_child]).max() > 0


def test_no_rejection_reduces_to_cross_entropy():
    N, T, V = 5, 7, 50
    lb = W.make_loss(3, N=N, T=T, V=V, tree="chain")
    tokens = lb.tokens.copy()
    tokens[:, 1:] = lb.labels[:, :-1]          # every draft token is its parent's label
    z = W.bf16_to_f32(lb.logits).astype(np.float64)
    res = oracle.loss(lb.logits, tokens, lb.parent, lb.labels, V=V)
    rows = np.array([n * T + p for n in range(N) for p in range(T - 1)])
    tgt = np.array([lb.labels[n, p] for n in range(N) for p in range(T - 1)], np.int64)
    ce = F.cross_entropy(torch.from_numpy(z[rows]), torch.from_numpy(tgt), reduction="sum").item()
    assert res["sums"][1] == 0.0
    assert res["loss"] == pytest.approx(ce / (N * (T - 1)), rel=1e-12)
    zt = torch.from_numpy(z[rows]).requires_grad_(True)
    (F.cross_entropy(zt, torch.from_numpy(tgt), reduction="sum") / (N * (T - 1))).backward()
    np.testing.assert_allclose(res["grad"][rows], zt.grad.numpy(), atol=1e-14)


def test_binary_vocab_rejection_is_cross_entropy_on_the_other_token():
    N, T, V = 6, 2, 2
    rng = np.random.default_rng(4)
    z = rng.standard_normal((N * T, V)) * 2
    parent = np.tile(W.chain_tree(T), (N, 1))
    labels = rng.integers(0, 2, size=(N, T)).astype(np.int32)
    tokens = np.zeros((N, T), np.int32)
    tokens[:, 1] = 1 - labels[:, 0]            # always rejected
    res = oracle.loss_f64(z, tokens, parent, labels, V=V)
    rows = np.arange(N) * T
    ce = F.cross_entropy(torch.from_numpy(z[rows]), torch.from_numpy(labels[:, 0].astype(np.int64)),
                         reduction="none").numpy()
    np.testing.assert_allclose(res["row_rej"][rows], ce, rtol=1e-12)
    assert res["sums"][0] == 0.0


def test_bf16_entry_equals_f64_entry_on_decoded_logits():
    lb, z = small_batch(5, N=4, T=12, V=40, tree=(3, 2, 1))
    a = oracle.loss_w(lb)
    b = oracle.loss_f64(z, lb.tokens, lb.parent, lb.labels, V=lb.V)
    np.testing.assert_array_equal(a["grad"], b["grad"])
    np.testing.assert_array_equal(a["sums"], b["sums"])


def test_rejection_term_is_finite_when_q_is_near_one():
    N, T, V = 1, 2, 4
    z = np.array([[60.0, 0.0, 0.0, 0.0], [0, 0, 0, 0]])
    res = oracle.loss_f64(z, np.array([[0, 0]], np.int32), W.chain_tree(2)[None], np.array([[1, 0]], np.int32),
                          V=V)
    # q(0) rounds to 1 in fp64; the clamp q <= 1 - 1e-6 keeps the term at -log(1e-6)
    assert res["row_rej"][0] == pytest.approx(-np.log(-np.expm1(-1e-6)), rel=1e-9)
    assert np.isfinite(res["grad"]).all()


def test_loss_status_codes():
    lb = W.make_loss(6, N=3, T=6, V=20, tree=(2, 2))
    parent = lb.parent.copy(); parent[1, 3] = 4
    tokens = lb.tokens.copy(); tokens[2, 2] = 20
    res = oracle.loss(lb.logits, tokens, parent, lb.labels, V=lb.V)
    assert list(res["status"]) == [0, 2, 1]
    assert (res["row_loss"][6:] == 0).all()
