"""GPU parity of sv_loss against the oracle: per-row losses and the batch sums within 1e-3 relative, the
bf16 gradient within 1e-2 of each row's largest entry, status codes exact; small shapes with ragged
vocabularies and the full online-training batch."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import run_loss

pytestmark = pytest.mark.gpu


def check_rows(got_rows, ref_rows):
    np.testing.assert_allclose(got_rows, ref_rows, rtol=1e-3, atol=1e-5)


def check_grad(g, ref):
    scale = np.abs(ref).max(axis=1, keepdims=True)
    assert (np.abs(g - ref) <= 1e-2 * scale + 1e-8).all()


@pytest.mark.parametrize("V", [8, 300, 4096, 50000])
@pytest.mark.parametrize("tree,T", [("chain", 6), ((4, 3, 2, 1, 1), 32), ((2, 2, 2, 2, 2, 1), 64), ((3,), 4)])
def test_loss_parity_small(V, tree, T):
    if tree == (3,) and V < 4:
        pytest.skip()
    lb = W.make_loss(V + T, N=5, T=T, V=max(V, T + 2) if tree != "chain" else V, tree=tree)
    ref = oracle.loss_w(lb)
    got = run_loss(lb)
    np.testing.assert_array_equal(got["status"], ref["status"])
    check_rows(got["row_loss"], ref["row_loss"])
    np.testing.assert_allclose(got["sums"][:2], ref["sums"][:2], rtol=1e-3, atol=1e-6)
    assert got["sums"][2] == ref["sums"][2]
    check_grad(got["grad"], ref["grad"])


def test_loss_single_node_traces_have_no_terms():
    lb = W.make_loss(1, N=3, T=1, V=64, tree="chain")
    got = run_loss(lb)
    assert (got["sums"] == 0).all() and (got["row_loss"] == 0).all() and (got["grad"] == 0).all()


def test_loss_status_codes_and_no_grad_mode():
    lb = W.make_loss(2, N=4, T=9, V=512, tree=(2, 2, 2))
    lb.parent = lb.parent.copy()
    lb.tokens = lb.tokens.copy()
    lb.parent[1, 5] = 7
    lb.tokens[3, 2] = 512
    ref = oracle.loss_w(lb)
    got = run_loss(lb)
    assert list(got["status"]) == [0, 2, 0, 1] == list(ref["status"])
    check_rows(got["row_loss"], ref["row_loss"])
    check_grad(got["grad"], ref["grad"])
    nog = run_loss(lb, want_grad=False)
    np.testing.assert_array_equal(nog["row_loss"], got["row_loss"])


def test_loss_batch_full_size():
    lb = W.make_workload("loss_batch", seed=0)
    got = run_loss(lb)
    ref = oracle.loss_w(lb, want_grad=False)
    assert (got["status"] == 0).all()
    check_rows(got["row_loss"], ref["row_loss"])
    np.testing.assert_allclose(got["sums"][:2], ref["sums"][:2], rtol=1e-3)
    # gradient on a subset of traces: the oracle's scale 1/n_terms is rescaled from the subset to the batch
    sub = [0, 17, 40, 63]
    rows = np.concatenate([np.arange(n * lb.T, (n + 1) * lb.T) for n in sub])
    part = W.LossBatch(N=len(sub), T=lb.T, V=lb.V, logits=lb.logits[rows], tokens=lb.tokens[sub],
                       parent=lb.parent[sub], labels=lb.labels[sub])
    rp = oracle.loss_w(part)
    check_grad(got["grad"][rows], rp["grad"] * (len(sub) / lb.N))
