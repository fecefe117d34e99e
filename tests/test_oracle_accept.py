"""Pins for the oracle's acceptance walk (CPU only).

Greedy: longest matching prefix, brute-force enumeration of root-to-node paths, first-occurrence
argmax, the expected acceptance length of a 0.7-match chain, the definition of acceptance length and
the worked timeline from the TIDE overview.  Stochastic: chi-square tests that the emitted tokens follow
the target distribution (10^6 draws, V=16), the closed-form first-step acceptance rate sum_x min(p,q),
and the degenerate cases (p = q, one-hot p, low temperature = greedy).  Fixed point: the contract's
exp2 polynomial and weights against float64 exp.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest
from scipy import stats

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W

GOLDEN = Path(__file__).resolve().parent / "golden"


def children(parent):
    ch = [[] for _ in parent]
    for i in range(1, len(parent)):
        ch[parent[i]].append(i)
    return ch


def softmax64(z, temp=1.0):
    z = np.asarray(z, np.float64) / temp
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


# ================================================================================================ fixed point
def test_fx_exp2_polynomial_error_bound():
    f = np.linspace(-0.5, 0.5, 2_000_001, dtype=np.float32)
    p = oracle.fx_exp2(f).astype(np.float64)
    rel = np.abs(p / np.exp2(f.astype(np.float64)) - 1.0)
    assert rel.max() <= 2.0 ** -21
    assert oracle.fx_exp2(np.array([0.0], np.float32))[0] == 1.0


def test_fx_weight_matches_exp_within_contract_error():
    y = np.linspace(-17.0, 0.0, 500_001, dtype=np.float32)
    w = oracle.fx_weight(y, 0.0).astype(np.float64)
    ref = 2.0 ** 24 * np.exp(y.astype(np.float64))
    assert np.all(np.abs(w - ref) <= ref * 2.0 ** -19 + 1.0)
    assert oracle.fx_weight(np.array([3.5], np.float32), 3.5)[0] == 2 ** 24
    # below 2^-24 of the maximum the weight is zero
    assert oracle.fx_weight(np.array([-16.7, -30.0, -1e30], np.float32), 0.0).tolist() == [0, 0, 0]


# ================================================================================================ greedy
def greedy_inputs(seed, B, T, V, tree, force_p, dt="f32"):
    return W.make_verify(seed, B=B, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, q_dt="f32", kv_dt="f32",
                         logit_dt=dt, tree=tree, mode="greedy", force_p=force_p, with_attn=False)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_greedy_chain_is_longest_matching_prefix(dt):
    w = greedy_inputs(1, 300, 8, 50, "chain", 0.75, dt)
    res = oracle.accept_w(w)
    zf = W.decode_f32(w.target_logits, dt)
    am = np.argmax(zf, axis=-1)     # numpy argmax: first occurrence
    for b in range(w.B):
        n = 0
        while n + 1 < w.T and w.tokens[b, n + 1] == am[b, n]:
            n += 1
        assert res["accept_len"][b] == n
        assert list(res["path"][b, :n]) == list(range(1, n + 1))
        assert res["bonus"][b] == am[b, n]
        assert res["out_tokens"][b, n] == am[b, n]
    np.testing.assert_array_equal(res["argmax"], am)


def test_greedy_tree_matches_brute_force_path_enumeration():
    w = greedy_inputs(2, 200, 20, 64, (3, 3, 2, 2), 0.8)
    res = oracle.accept_w(w)
    am = np.argmax(w.target_logits, axis=-1)
    for b in range(w.B):
        par = w.parent[b]
        best = [0]
        for node in range(1, w.T):          # every root-to-node path
            pth = [node]
            while par[pth[-1]] != 0:
                pth.append(par[pth[-1]])
            pth = pth[::-1]
            ok = all(w.tokens[b, c] == am[b, par[c]] for c in pth)
            if ok and len(pth) + 1 > len(best):
                best = [0] + pth
        n = len(best) - 1
        assert res["accept_len"][b] == n
        assert list(res["path"][b, :n]) == best[1:]
        assert all(x == -1 for x in res["path"][b, n:])
        assert res["bonus"][b] == am[b, best[-1]]
        assert list(res["out_tokens"][b, : n + 1]) == [w.tokens[b, c] for c in best[1:]] + [am[b, best[-1]]]


def test_greedy_duplicate_siblings_first_wins_and_ties_take_first_index():
    V = 8
    parent = np.array([[-1, 0, 0, 1, 2]], np.int32)
    z = np.zeros((1, 5, V), np.float32)
    z[0, 0, [3, 5]] = 2.0        # tie: argmax must be 3 (first occurrence)
    z[0, 1, 6] = 1.0
    z[0, 2, 4] = 1.0
    tokens = np.array([[0, 3, 3, 6, 4]], np.int32)   # both children of root carry 3; node 1 wins
    res = oracle.accept(z, tokens, parent, V=V, logit_dt="f32")
    assert res["argmax"][0, 0] == 3
    assert res["accept_len"][0] == 2 and list(res["path"][0, :2]) == [1, 3]


def test_greedy_expected_accept_length_of_point_seven_chain():
    """5-draft chain, each draft equal to the target argmax w.p. 0.7: E[len] = sum_k 0.7^k."""
    w = greedy_inputs(3, 6000, 6, 1024, "chain", 0.7)
    res = oracle.accept_w(w)
    lens = res["accept_len"].astype(np.float64)
    expect = sum(0.7 ** k for k in range(1, 6))
    assert abs(lens.mean() - expect) < 4 * lens.std() / math.sqrt(len(lens))


def test_accept_length_definition_golden():
    g = json.loads((GOLDEN / "accept_length_definition.json").read_text())
    for key, want_match in (("chain_all_match", True), ("chain_none_match", False)):
        T = g[key]["T"]
        V = 16
        z = np.zeros((1, T, V), np.float32)
        z[0, :, 5] = 1.0
        tokens = np.full((1, T), 5 if want_match else 6, np.int32)
        res = oracle.accept(z, tokens, W.chain_tree(T)[None], V=V, logit_dt="f32")
        assert res["accept_len"][0] == g[key]["accept_len"]
        assert int((res["out_tokens"][0] >= 0).sum()) == g[key]["emitted_tokens"]


def test_worked_timeline_golden():
    """TIDE overview: 10 tokens, 4 drafts per step, 2 accepted per step -> about 2x fewer target passes."""
    g = json.loads((GOLDEN / "timeline.json").read_text())
    gamma, need, acc = g["draft_tokens_per_step"], g["tokens_to_generate"], g["accepted_per_step"]
    T, V = gamma + 1, 32
    rng = np.random.default_rng(0)
    emitted, passes = 0, 0
    while emitted < need:
        z = rng.standard_normal((1, T, V)).astype(np.float32)
        am = np.argmax(z, axis=-1)[0]
        tokens = np.zeros((1, T), np.int32)
        for k in range(1, T):
            tokens[0, k] = am[k - 1] if k <= acc else (am[k - 1] + 1) % V
        res = oracle.accept(z, tokens, W.chain_tree(T)[None], V=V, logit_dt="f32")
        assert res["accept_len"][0] == acc
        emitted += int(res["accept_len"][0]) + 1      # accepted drafts + the target's own token
        passes += 1
    assert passes == math.ceil(need / (acc + 1))
    assert need / passes >= g["speedup_about"] * 0.95 - 1e-9   # ~2x fewer target passes than plain decode


def test_accept_status_codes():
    V = 8
    z = np.random.default_rng(0).standard_normal((4, 3, V)).astype(np.float32)
    parent = np.tile(W.chain_tree(3), (4, 1))
    tokens = np.ones((4, 3), np.int32)
    parent[1, 2] = 5
    tokens[2, 1] = V
    z[3, 2, 4] = np.nan
    res = oracle.accept(z, tokens, parent, V=V, logit_dt="f32")
    assert list(res["status"]) == [0, 2, 1, 5]
    assert list(res["accept_len"][1:]) == [-1, -1, -1]
    assert res["argmax"][3, 2] == -1
    assert (res["path"][1:] == -1).all() and (res["out_tokens"][1:] == -1).all()


# ================================================================================================ stochastic
def chi2_ok(samples, p, alpha=1e-3):
    counts = np.bincount(samples, minlength=len(p)).astype(np.float64)
    exp = p * counts.sum()
    chi = ((counts - exp) ** 2 / exp).sum()
    return stats.chi2.sf(chi, len(p) - 1) > alpha, chi


def run_batched(target_row_logits, draft_row_logits, parent, draw_tokens, n, temp, seed, chunk=250_000):
    """Replicate fixed per-node logits over n requests with fresh draft tokens and uniforms."""
    rng = np.random.default_rng(seed)
    outs = []
    T, V = target_row_logits.shape
    for start in range(0, n, chunk):
        B = min(chunk, n - start)
        tgt = np.broadcast_to(target_row_logits, (B, T, V)).copy()
        dr = None if draft_row_logits is None else np.broadcast_to(draft_row_logits, (B, T, V)).copy()
        tokens = draw_tokens(rng, B)
        u = rng.integers(0, 2 ** 32, size=(B, T), dtype=np.uint32)
        res = oracle.accept(tgt, tokens, np.broadcast_to(parent, (B, T)).copy(), V=V, logit_dt="f32",
                            temperature=temp, draft=dr, uniforms=u, want_argmax=False)
        assert (res["status"] == 0).all()
        res["tokens"] = tokens
        outs.append(res)
    return {k: np.concatenate([o[k] for o in outs]) for k in ("accept_len", "out_tokens", "tokens", "path")}


def sample_rows(rng, probs, B):
    """B draws from a categorical distribution by inverse CDF."""
    c = np.cumsum(probs)
    return np.minimum(np.searchsorted(c, rng.random(B) * c[-1], side="right"), len(probs) - 1)


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_prob_chain_marginals_follow_target(temp):
    V, T, n = 16, 3, 1_000_000
    rng = np.random.default_rng(10)
    zp = (1.5 * rng.standard_normal((T, V))).astype(np.float32)
    zq = (0.8 * zp + 0.9 * rng.standard_normal((T, V))).astype(np.float32)
    p, q = softmax64(zp, temp), softmax64(zq, temp)

    def draw(r, B):
        t = np.zeros((B, T), np.int32)
        for k in range(1, T):
            t[:, k] = sample_rows(r, q[k - 1], B)
        return t

    out = run_batched(zp, zq, W.chain_tree(T), draw, n, temp, 11)
    ok, chi = chi2_ok(out["out_tokens"][:, 0], p[0])
    assert ok, chi
    sel = out["accept_len"] >= 1
    ok, chi = chi2_ok(out["out_tokens"][sel, 1], p[1])
    assert ok, chi
    # closed form: first-step acceptance probability = sum_x min(p(x), q(x)) = 1 - TV(p, q)
    a = np.minimum(p[0], q[0]).sum()
    rate = sel.mean()
    assert abs(rate - a) < 4 * math.sqrt(a * (1 - a) / n)


def test_prob_siblings_iid_from_draft_follow_target():
    """Three i.i.d. draft siblings under the root (duplicates allowed): the first emitted token ~ p."""
    V, T, n = 16, 4, 1_000_000
    rng = np.random.default_rng(20)
    zp = (1.5 * rng.standard_normal((T, V))).astype(np.float32)
    zq = (1.5 * rng.standard_normal((T, V))).astype(np.float32)
    p, q = softmax64(zp), softmax64(zq)

    def draw(r, B):
        t = np.zeros((B, T), np.int32)
        for k in range(1, T):
            t[:, k] = sample_rows(r, q[0], B)
        return t

    out = run_batched(zp, zq, W.star_tree(T), draw, n, 1.0, 21)
    ok, chi = chi2_ok(out["out_tokens"][:, 0], p[0])
    assert ok, chi


def test_onehot_tree_marginals_follow_target():
    """One-hot proposals (no draft distribution), distinct siblings: sampling without replacement keeps
    the emitted token ~ p at every depth."""
    V, n = 16, 1_000_000
    parent = np.array([-1, 0, 0, 0, 1, 1], np.int32)
    T = len(parent)
    rng = np.random.default_rng(30)
    zp = (1.2 * rng.standard_normal((T, V))).astype(np.float32)
    p = softmax64(zp, 0.7)
    fixed = np.array([0, int(np.argmax(p[0])), 3, 9, int(np.argmax(p[1])), 2], np.int32)

    def draw(r, B):
        return np.broadcast_to(fixed, (B, T)).copy()

    out = run_batched(zp, None, parent, draw, n, 0.7, 31)
    ok, chi = chi2_ok(out["out_tokens"][:, 0], p[0])
    assert ok, chi
    sel = (out["accept_len"] >= 1) & (out["path"][:, 0] == 1)
    ok, chi = chi2_ok(out["out_tokens"][sel, 1], p[1])
    assert ok, chi


def test_p_equals_q_always_accepts():
    V, T, B = 32, 6, 2000
    rng = np.random.default_rng(40)
    z = rng.standard_normal((B, T, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, T)).astype(np.int32)
    u = rng.integers(0, 2 ** 32, size=(B, T), dtype=np.uint32)
    res = oracle.accept(z, tokens, np.tile(W.chain_tree(T), (B, 1)), V=V, logit_dt="f32", temperature=1.0,
                        draft=z.copy(), uniforms=u)
    # only tokens with zero fixed-point weight in both p and q can be rejected
    assert (res["accept_len"] == T - 1).mean() > 0.99


def test_one_hot_target_is_deterministic():
    V, T, B = 32, 4, 500
    rng = np.random.default_rng(41)
    z = rng.standard_normal((B, T, V)).astype(np.float32)
    star = rng.integers(0, V, size=(B, T))
    for b in range(B):
        for r in range(T):
            z[b, r, star[b, r]] = 40.0
    zq = rng.standard_normal((B, T, V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, T)).astype(np.int32)
    match = rng.random((B, T)) < 0.6
    tokens[:, 1:] = np.where(match[:, 1:], star[:, :-1], tokens[:, 1:])
    u = rng.integers(0, 2 ** 32, size=(B, T), dtype=np.uint32)
    res = oracle.accept(z, tokens, np.tile(W.chain_tree(T), (B, 1)), V=V, logit_dt="f32", temperature=1.0,
                        draft=zq, uniforms=u)
    greedy = oracle.accept(z, tokens, np.tile(W.chain_tree(T), (B, 1)), V=V, logit_dt="f32")
    for key in ("accept_len", "path", "out_tokens", "bonus"):
        np.testing.assert_array_equal(res[key], greedy[key])


def test_low_temperature_onehot_equals_greedy():
    w = greedy_inputs(50, 400, 20, 64, (3, 2, 2, 2), 0.7, "bf16")
    zf = W.bf16_to_f32(w.target_logits).copy()
    am = np.argmax(zf, axis=-1)
    for b in range(w.B):                 # give every row a unique maximum with a gap >= 1
        for r in range(w.T):
            zf[b, r, am[b, r]] = zf[b, r].max() + 1.0
    tgt = W.f32_to_bf16(zf)
    u = np.random.default_rng(51).integers(0, 2 ** 32, size=(w.B, w.T), dtype=np.uint32)
    sto = oracle.accept(tgt, w.tokens, w.parent, V=w.V, logit_dt="bf16", temperature=1e-3, uniforms=u)
    gr = oracle.accept(tgt, w.tokens, w.parent, V=w.V, logit_dt="bf16")
    for key in ("accept_len", "path", "out_tokens", "bonus"):
        np.testing.assert_array_equal(sto[key], gr[key])


def test_stochastic_requires_uniforms():
    z = np.zeros((1, 2, 4), np.float32)
    res = oracle.accept(z, np.zeros((1, 2), np.int32), W.chain_tree(2)[None], V=4, logit_dt="f32",
                        temperature=1.0)
    assert res["rc"] == 1
