"""GPU parity of sv_accept against the oracle: every output bit-exact (accept_len, path, out_tokens, bonus,
argmax, status), greedy and stochastic, small shapes with ragged vocabularies and every named workload at
full size."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import run_accept

pytestmark = pytest.mark.gpu

KEYS = ("status", "accept_len", "path", "out_tokens", "bonus", "argmax")


def compare(g, o):
    for k in KEYS:
        if g.get(k) is None:
            continue
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)


AUTO = object()


def check(w, temperature=None, draft=AUTO):
    t = w.temperature if temperature is None else temperature
    d = w.draft_logits if draft is AUTO else draft
    d = d if t > 0 else None
    ref = oracle.accept(w.target_logits, w.tokens, w.parent, V=w.V, logit_dt=w.logit_dt, temperature=t, draft=d,
                        uniforms=w.uniforms)
    got = run_accept(w.target_logits, w.tokens, w.parent, V=w.V, temperature=t, draft=d, uniforms=w.uniforms)
    compare(got, ref)
    return got


TREES = [("chain", 8), ((3, 2, 2), 13), ("star", 10), ((2, 2, 2, 2, 1), 25), ((4, 3, 2, 2, 1, 1, 1), 64)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V", [16, 1000, 4096, 40000])
@pytest.mark.parametrize("tree,T", TREES)
def test_greedy_parity(dt, V, tree, T):
    if tree == "star" and T > V:
        pytest.skip("star needs V >= T")
    w = W.make_verify(V + T, B=23, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree=tree, mode="greedy",
                      force_p=0.7, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("mode", ["prob", "onehot"])
@pytest.mark.parametrize("temp", [1.0, 0.7, 1e-3])
@pytest.mark.parametrize("V,dt", [(16, "f32"), (1000, "bf16"), (4096, "bf16"), (50000, "bf16")])
@pytest.mark.parametrize("tree,T", [("chain", 6), ((3, 2, 2), 13), ("star", 5)])
def test_stochastic_parity(mode, temp, V, dt, tree, T):
    w = W.make_verify(V * 7 + T, B=19, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree=tree,
                      mode="prob" if mode == "prob" else "onehot", temperature=temp, force_p=0.7, sigma=2.0,
                      with_attn=False)
    g = check(w, temperature=temp, draft=w.draft_logits if mode == "prob" else None)
    assert (g["status"] == 0).all()


def test_single_node_trees():
    for t in (0.0, 1.0):
        w = W.make_verify(3, B=9, T=1, Hq=1, Hkv=1, D=8, L=(0, 0), V=777, logit_dt="bf16", tree="chain",
                          mode="greedy" if t == 0 else "onehot", temperature=t, with_attn=False)
        g = check(w, temperature=t, draft=None)
        assert (g["accept_len"] == 0).all()


def test_status_codes_bad_tree_token_nonfinite():
    w = W.make_verify(4, B=6, T=7, Hq=1, Hkv=1, D=8, L=(0, 0), V=300, logit_dt="f32", tree=(2, 2, 1), mode="onehot",
                      temperature=1.0, with_attn=False)
    w.parent = w.parent.copy()
    w.tokens = w.tokens.copy()
    w.target_logits = w.target_logits.copy()
    w.parent[1, 3] = 5                 # not topological
    w.parent[2, 0] = 0                 # root must have parent -1
    w.tokens[3, 4] = 300               # token out of range
    w.target_logits[4, 2, 17] = np.nan
    w.target_logits[5, 6, 0] = -np.inf
    for t in (0.0, 1.0):
        g = check(w, temperature=t, draft=None)
        assert list(g["status"]) == [0, 2, 2, 1, 5, 5]
        assert (g["accept_len"][1:] == -1).all()


@pytest.mark.parametrize("name", ["tiny_chain", "llama3_8b_tree"])
def test_named_greedy_workloads_full_size(name):
    w = W.make_workload(name, seed=0, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()
    if w.B > 1:
        assert g["accept_len"].mean() > 0


def test_qwen3_stochastic_full_size():
    w = W.make_workload("qwen3_8b_stochastic", seed=0, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("temp", [0.0, 0.7])
def test_fp8_long_context_accept_full_size(temp):
    w = W.make_workload("fp8_long_context", seed=0, with_attn=False, mode="greedy" if temp == 0 else "onehot",
                        temperature=temp)
    g = check(w, temperature=temp, draft=None)
    assert (g["status"] == 0).all()
