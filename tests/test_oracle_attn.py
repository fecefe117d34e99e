"""Pins for the oracle's tree-masked attention (CPU only).

Each check reaches the expected value by a different route than the oracle's own ancestor walk and
fp64 loops: torch's scaled_dot_product_attention with an explicit dense mask built by a boolean
matrix closure, torch's built-in causal mask, hand-written expectations for star trees, and invariants.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def decode(a, dt, scale=None):
    if dt == "f32":
        x = np.asarray(a, np.float64)
    elif dt == "bf16":
        x = W.bf16_to_f32(a).astype(np.float64)
    else:  # e4m3 through the generator's own value table (independent of the oracle's bit decoder)
        a = np.asarray(a, np.uint8)
        mag = W._E4M3_POS[np.minimum(a & 0x7F, 126)]
        x = np.where(a & 0x80, -mag, mag)
    if scale is not None:
        x = x * np.asarray(scale, np.float64)[None, :, None, None]
    return x


def closure_mask(parent):
    """reach[i, j] = 1 iff j is i or an ancestor of i, by boolean matrix closure of the parent edges."""
    T = len(parent)
    R = np.eye(T, dtype=bool)
    A = np.zeros((T, T), dtype=bool)
    for i in range(1, T):
        A[i, parent[i]] = True
    while True:
        R2 = R | ((R.astype(np.int64) @ A.astype(np.int64)) > 0)
        if (R2 == R).all():
            return R
        R = R2


def sdpa_reference(w, sm_scale=None):
    """torch SDPA (fp64, CPU) with an explicit [T, L+T] boolean mask per request."""
    B, T, Hq, D = w.q.shape
    G = w.Hq // w.Hkv
    q = torch.from_numpy(decode(w.q, w.q_dt))
    k = torch.from_numpy(decode(w.k, w.kv_dt, w.k_scale))
    v = torch.from_numpy(decode(w.v, w.kv_dt, w.v_scale))
    outs, lses = [], []
    for b in range(B):
        L = int(w.kv_len[b])
        mask = np.zeros((T, L + T), dtype=bool)
        mask[:, :L] = True
        mask[:, L:] = closure_mask(w.parent[b])
        m = torch.from_numpy(mask)
        qb = q[b].permute(1, 0, 2)                                   # [Hq, T, D]
        kb = k[b, :, : L + T].repeat_interleave(G, dim=0)            # [Hq, L+T, D]
        vb = v[b, :, : L + T].repeat_interleave(G, dim=0)
        scale = sm_scale if sm_scale else 1.0 / np.sqrt(D)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=m, scale=scale)
        s = (qb @ kb.transpose(-1, -2)) * scale
        lse = torch.logsumexp(s.masked_fill(~m, float("-inf")), dim=-1)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(lse.permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


CASES = [
    # B, T, Hq, Hkv, D, L, tree, dtypes
    (2, 6, 4, 1, 16, (0, 9), "chain", ("f32", "f32")),
    (2, 13, 4, 2, 32, (3, 40), (3, 2, 2), ("bf16", "bf16")),
    (3, 9, 8, 2, 16, (1, 20), (4, 2), ("bf16", "e4m3")),
    (1, 1, 2, 2, 8, (5, 5), "chain", ("f32", "f32")),
    (2, 17, 6, 3, 16, (0, 0), (2, 2, 2, 1), ("f32", "bf16")),
    (2, 20, 2, 1, 64, (60, 70), "star", ("bf16", "bf16")),
]


@pytest.mark.parametrize("case", CASES)
def test_attn_matches_sdpa_with_dense_mask(case):
    B, T, Hq, Hkv, D, L, tree, (qdt, kvdt) = case
    w = W.make_verify(7, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, L=L, V=64, q_dt=qdt, kv_dt=kvdt, tree=tree)
    out, lse, st, rc = oracle.tree_attn_w(w)
    assert rc == 0 and (st == 0).all()
    ref_o, ref_lse = sdpa_reference(w)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-10)


def test_sm_scale_override():
    w = W.make_verify(3, B=1, T=5, Hq=2, Hkv=1, D=16, L=(7, 7), V=8, q_dt="f32", kv_dt="f32", tree=(2, 2))
    out, lse, _, _ = oracle.tree_attn_w(w, sm_scale=0.3)
    ref_o, ref_lse = sdpa_reference(w, sm_scale=0.3)
    np.testing.assert_allclose(out, ref_o, atol=1e-10)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-10)


def test_chain_equals_causal_attention():
    """A chain tree is ordinary causal attention over prefix + drafts (torch's is_causal mask)."""
    w = W.make_verify(11, B=2, T=7, Hq=4, Hkv=2, D=32, L=(5, 30), V=8, q_dt="f32", kv_dt="f32", tree="chain")
    out, _, _, _ = oracle.tree_attn_w(w)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        L = int(w.kv_len[b])
        n = L + w.T
        k = torch.from_numpy(w.k[b, :, :n].astype(np.float64)).repeat_interleave(G, 0)
        v = torch.from_numpy(w.v[b, :, :n].astype(np.float64)).repeat_interleave(G, 0)
        # full-length queries: prefix rows are arbitrary (their outputs are discarded), tree rows are q
        qf = torch.zeros(w.Hq, n, w.D, dtype=torch.float64)
        qf[:, L:] = torch.from_numpy(w.q[b].astype(np.float64)).permute(1, 0, 2)
        o = F.scaled_dot_product_attention(qf, k, v, is_causal=True)
        np.testing.assert_allclose(out[b], o[:, L:].permute(1, 0, 2).numpy(), atol=1e-10)


def test_star_tree_sees_prefix_root_and_self():
    w = W.make_verify(5, B=1, T=6, Hq=2, Hkv=1, D=16, L=(9, 9), V=8, q_dt="f32", kv_dt="f32", tree="star")
    out, _, _, _ = oracle.tree_attn_w(w)
    L = int(w.kv_len[0])
    for i in range(w.T):
        pos = list(range(L)) + [L] + ([L + i] if i else [])
        for h in range(w.Hq):
            q = w.q[0, i, h].astype(np.float64)
            K = w.k[0, 0, pos].astype(np.float64)
            V = w.v[0, 0, pos].astype(np.float64)
            s = K @ q / np.sqrt(w.D)
            p = np.exp(s - s.max())
            np.testing.assert_allclose(out[0, i, h], (p / p.sum()) @ V, atol=1e-12)


def test_single_node_is_plain_decode_attention():
    w = W.make_verify(2, B=3, T=1, Hq=4, Hkv=4, D=16, L=(1, 50), V=8, q_dt="f32", kv_dt="f32", tree="chain")
    out, _, _, _ = oracle.tree_attn_w(w)
    for b in range(w.B):
        n = int(w.kv_len[b]) + 1
        o = F.scaled_dot_product_attention(torch.from_numpy(w.q[b].astype(np.float64)).permute(1, 0, 2),
                                           torch.from_numpy(w.k[b, :, :n].astype(np.float64)),
                                           torch.from_numpy(w.v[b, :, :n].astype(np.float64)))
        np.testing.assert_allclose(out[b], o.permute(1, 0, 2).numpy(), atol=1e-12)


def test_prefix_permutation_invariance():
    w = W.make_verify(9, B=1, T=8, Hq=4, Hkv=2, D=16, L=(33, 33), V=8, q_dt="f32", kv_dt="f32", tree=(3, 2))
    out, lse, _, _ = oracle.tree_attn_w(w)
    perm = np.random.default_rng(0).permutation(33)
    w.k = w.k.copy()
    w.v = w.v.copy()
    w.k[:, :, :33] = w.k[:, :, perm]
    w.v[:, :, :33] = w.v[:, :, perm]
    out2, lse2, _, _ = oracle.tree_attn_w(w)
    np.testing.assert_allclose(out2, out, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)


def test_row_subset_matches_full():
    w = W.make_verify(4, B=2, T=9, Hq=4, Hkv=2, D=16, L=(3, 12), V=8, q_dt="bf16", kv_dt="bf16", tree=(2, 2, 1))
    out, lse, _, _ = oracle.tree_attn_w(w)
    rows = np.array([[0, 0, 0], [1, 8, 3], [1, 4, 2]], np.int32)
    o2, l2, _, _ = oracle.tree_attn_w(w, rows=rows)
    for b, i, h in rows:
        np.testing.assert_array_equal(o2[b, i, h], out[b, i, h])
        assert l2[b, i, h] == lse[b, i, h]
    assert np.isnan(o2[0, 1, 0]).all()


def test_request_status_codes():
    w = W.make_verify(1, B=3, T=4, Hq=2, Hkv=1, D=8, L=(2, 2), V=8, q_dt="f32", kv_dt="f32", tree="chain")
    w.parent = w.parent.copy()
    w.parent[1, 2] = 2            # not topological
    w.kv_len = w.kv_len.copy()
    w.kv_len[2] = w.kv_cap - 3    # kv_len + T > kv_cap
    _, _, st, rc = oracle.tree_attn_w(w)
    assert rc == 0
    assert list(st) == [0, 2, 1]


def test_tree_check_and_depth():
    assert oracle.tree_check(np.array([-1, 0, 0, 1, 3])) == 0
    assert oracle.tree_check(np.array([0, 0])) == 2
    assert oracle.tree_check(np.array([-1, 1])) == 2
    assert oracle.tree_check(np.array([-1, 0, 5])) == 2
    st, d = oracle.tree_depth(np.array([-1, 0, 0, 1, 3, 2]))
    assert st == 0 and list(d) == [0, 1, 1, 2, 3, 2]


def test_duplicate_sampled_rows_are_race_free():
    """Sampled rows may repeat (random draws); every copy must equal the full computation."""
    w = W.make_verify(12, B=2, T=16, Hq=8, Hkv=2, D=64, L=(300, 400), V=64, q_dt="bf16", kv_dt="bf16",
                      tree=(3, 2, 2))
    out, lse, _, _ = oracle.tree_attn_w(w)
    rows = np.tile(np.array([[0, 3, 1], [1, 15, 7], [1, 0, 0]], np.int32), (64, 1))
    o2, l2, _, _ = oracle.tree_attn_w(w, rows=rows)
    for b, i, h in rows[:3]:
        np.testing.assert_array_equal(o2[b, i, h], out[b, i, h])
        assert l2[b, i, h] == lse[b, i, h]
