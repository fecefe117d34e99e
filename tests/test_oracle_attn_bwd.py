"""Pins for the oracle's tree-attention backward (CPU only).

Expected gradients come by routes other than the oracle's chain-rule loops: torch autograd through
scaled_dot_product_attention with an explicit dense boolean mask (float64, a library routine), central
finite differences of <dO, O> through the oracle's own forward, and two closed forms that hold for any
softmax attention: the gradient w.r.t. the keys sums to zero over the positions (the softmax Jacobian
annihilates constants), and the gradient w.r.t. the values sums to dO (the weights sum to one).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.test_oracle_attn import closure_mask, decode


def batch(seed, tree, T, dt="f32", B=3, Hq=4, Hkv=2, D=16, L=(0, 20)):
    w = W.make_verify(seed, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, L=L, V=32, q_dt=dt, kv_dt=dt, logit_dt="f32", tree=tree,
                      mode="greedy", with_attn=True)
    s_g, = W.rng_streams(seed + 1000, 1)
    g = s_g.standard_normal(size=w.q.shape, dtype=np.float32)
    dout = W.encode(g, dt)
    return w, dout


def autograd_reference(w, dout):
    B, T, Hq, D = w.q.shape
    G = w.Hq // w.Hkv
    q = torch.from_numpy(decode(w.q, w.q_dt)).requires_grad_(True)
    k = torch.from_numpy(decode(w.k, w.kv_dt)).requires_grad_(True)
    v = torch.from_numpy(decode(w.v, w.kv_dt)).requires_grad_(True)
    g = torch.from_numpy(decode(dout, w.q_dt))
    total = 0.0
    for b in range(B):
        L = int(w.kv_len[b])
        mask = np.zeros((T, L + T), dtype=bool)
        mask[:, :L] = True
        mask[:, L:] = closure_mask(w.parent[b])
        qb = q[b].permute(1, 0, 2)
        kb = k[b, :, : L + T].repeat_interleave(G, dim=0)
        vb = v[b, :, : L + T].repeat_interleave(G, dim=0)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=torch.from_numpy(mask))
        total = total + (o * g[b].permute(1, 0, 2)).sum()
    total.backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("tree,T", [("chain", 6), ((3, 2, 2), 13), ("star", 5), ((4, 3, 2, 2, 1, 1), 30)])
def test_backward_matches_autograd_through_sdpa_with_dense_mask(dt, tree, T):
    w, dout = batch(T * 7 + len(dt), tree, T, dt)
    dq, dk, dv, st, rc = oracle.tree_attn_bwd(w.q, w.k, w.v, w.kv_len, w.parent, dout, Hq=w.Hq, Hkv=w.Hkv,
                                              q_dt=w.q_dt, kv_dt=w.kv_dt)
    assert rc == 0 and (st == 0).all()
    gq, gk, gv = autograd_reference(w, dout)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, gk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, gv, rtol=0, atol=1e-11)


def test_backward_matches_central_finite_differences():
    """d <dO, O> / d x by central differences of the oracle's float64 forward on float32 inputs."""
    w, dout = batch(3, (2, 2), 5, "f32", B=1, Hq=2, Hkv=1, D=4, L=(3, 3))
    dq, dk, dv, st, rc = oracle.tree_attn_bwd(w.q, w.k, w.v, w.kv_len, w.parent, dout, Hq=w.Hq, Hkv=w.Hkv,
                                              q_dt="f32", kv_dt="f32")
    g = dout.astype(np.float64)

    def loss(q, k, v):
        o, _, _, _ = oracle.tree_attn(q, k, v, w.kv_len, w.parent, Hq=w.Hq, Hkv=w.Hkv, q_dt="f32", kv_dt="f32")
        return float(np.sum(o * g))

    h = 2.0 ** -10
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        base = {"q": w.q, "k": w.k, "v": w.v}
        x = base[name]
        idx = list(np.ndindex(x.shape))
        if name != "q":
            idx = [i for i in idx if i[2] < int(w.kv_len[0]) + w.T]
        for ix in idx:
            xp, xm = x.copy(), x.copy()
            xp[ix] += h
            xm[ix] -= h
            args_p = dict(base, **{name: xp})
            args_m = dict(base, **{name: xm})
            fd = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
            assert abs(fd - grad[ix]) < 2e-5 * max(1.0, abs(fd)), (name, ix, fd, grad[ix])


@pytest.mark.parametrize("tree,T", [((3, 2, 2), 13), ((4, 3, 2, 2, 1, 1, 1), 64)])
def test_key_gradient_sums_to_zero_and_value_gradient_sums_to_dout(tree, T):
    w, dout = batch(11, tree, T, "bf16", B=2, Hq=6, Hkv=2, D=8, L=(5, 40))
    dq, dk, dv, st, rc = oracle.tree_attn_bwd(w.q, w.k, w.v, w.kv_len, w.parent, dout, Hq=w.Hq, Hkv=w.Hkv,
                                              q_dt="bf16", kv_dt="bf16")
    g = decode(dout, "bf16")                                   # [B,T,Hq,D]
    G = w.Hq // w.Hkv
    for b in range(w.B):
        for hk in range(w.Hkv):
            np.testing.assert_allclose(dk[b, hk].sum(axis=0), 0.0, atol=1e-12)
            want = g[b, :, hk * G:(hk + 1) * G].sum(axis=(0, 1))
            np.testing.assert_allclose(dv[b, hk].sum(axis=0), want, rtol=0, atol=1e-11)
        L = int(w.kv_len[b])
        assert not dk[b, :, L + T:].any() and not dv[b, :, L + T:].any()


def test_bad_requests_get_zero_gradients_and_a_status():
    w, dout = batch(5, (2, 2), 7, "f32", B=3)
    parent = w.parent.copy()
    kv_len = w.kv_len.copy()
    parent[0, 3] = 6
    kv_len[2] = w.kv_cap
    dq, dk, dv, st, rc = oracle.tree_attn_bwd(w.q, w.k, w.v, kv_len, parent, dout, Hq=w.Hq, Hkv=w.Hkv,
                                              q_dt="f32", kv_dt="f32")
    assert list(st) == [2, 0, 1]
    assert not dq[[0, 2]].any() and not dk[[0, 2]].any() and dq[1].any()
