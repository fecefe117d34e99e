"""GPU parity of sv_tree_attn_bwd against the oracle's float64 backward.

The GPU runs its own forward (sv_tree_attn) for out and lse, then the backward with the upstream gradient
dout; the oracle recomputes everything in float64 from q, k, v.  Tolerance, per request and per tensor:
max |g - g_ref| <= tol * max |g_ref| + 1e-6 with tol = 2e-2 for bf16 inputs (out is rounded to bf16 before
delta = <dout, out> is formed, the same 2e-2 the forward is held to) and 2e-3 for fp32 inputs (fp32
accumulation over up to a few thousand positions).  dk / dv are compared on [0, kv_len + T), the positions
the call writes."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def run_bwd(w, dout):
    q, k, v = dev(w.q), dev(w.k), dev(w.v)
    kl, par = dev(w.kv_len), dev(w.parent)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
    sv.tree_attn(q, k, v, kl, par, out, lse=lse)
    dq = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.full(k.shape, float("nan"), dtype=torch.float32, device="cuda")
    dv = torch.full(v.shape, float("nan"), dtype=torch.float32, device="cuda")
    st = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    sv.tree_attn_bwd(q, k, v, kl, par, out, lse, dev(dout), dq, dk, dv, status=st)
    torch.cuda.synchronize()
    return dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), st.cpu().numpy()


def check(w, dout):
    rq, rk, rv, rst, rc = oracle.tree_attn_bwd(w.q, w.k, w.v, w.kv_len, w.parent, dout, Hq=w.Hq, Hkv=w.Hkv,
                                               q_dt=w.q_dt, kv_dt=w.kv_dt)
    assert rc == 0
    gq, gk, gv, gst = run_bwd(w, dout)
    np.testing.assert_array_equal(gst, rst)
    tol = 2e-2 if w.q_dt == "bf16" else 2e-3
    for b in range(w.B):
        if rst[b] != 0:
            assert not gq[b].any()
            continue
        n = int(w.kv_len[b]) + w.T
        for name, g, r in (("dq", gq[b], rq[b]), ("dk", gk[b][:, :n], rk[b][:, :n]), ("dv", gv[b][:, :n], rv[b][:, :n])):
            err = np.max(np.abs(g - r))
            assert err <= tol * np.max(np.abs(r)) + 1e-6, (name, b, err, np.max(np.abs(r)))
    return gst


def make(seed, *, B, T, Hq, Hkv, D, L, dt, tree):
    w = W.make_verify(seed, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, L=L, V=32, q_dt=dt, kv_dt=dt, logit_dt="f32", tree=tree,
                      mode="greedy", with_attn=True, junk="nan")
    s_g, = W.rng_streams(seed + 1000, 1)
    dout = W.encode(s_g.standard_normal(size=w.q.shape, dtype=np.float32), dt)
    return w, dout


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("D,Hq,Hkv", [(32, 4, 4), (64, 8, 2), (128, 32, 8), (128, 16, 1)])
@pytest.mark.parametrize("tree,T", [("chain", 6), ((3, 2, 2), 13), ((4, 3, 2, 2, 1, 1, 1), 64), ("star", 9)])
def test_attn_bwd_parity(dt, D, Hq, Hkv, tree, T):
    w, dout = make(D + Hq + T, B=3, T=T, Hq=Hq, Hkv=Hkv, D=D, L=(0, 150), dt=dt, tree=tree)
    assert (check(w, dout) == 0).all()


def test_attn_bwd_statuses():
    w, dout = make(4, B=3, T=7, Hq=4, Hkv=2, D=64, L=(10, 40), dt="bf16", tree=(2, 2, 1))
    w.parent = w.parent.copy()
    w.kv_len = w.kv_len.copy()
    w.parent[0, 2] = 5
    w.kv_len[2] = w.kv_cap
    assert list(check(w, dout)) == [2, 0, 1]


def test_attn_bwd_llama3_shape_two_requests():
    """Two requests of the Llama3-shaped batch at full per-request size (60-node tree, 32/8 heads, D=128,
    bf16, prefixes of 2048..8192)."""
    w, dout = make(0, B=2, T=60, Hq=32, Hkv=8, D=128, L=(2048, 8192), dt="bf16", tree=(4, 3, 2, 2, 1, 1))
    assert (check(w, dout) == 0).all()


@pytest.mark.parametrize("Hq,Hkv,tree,T", [(8, 8, (3, 2, 2), 13), (64, 8, (4, 3, 2, 2, 1, 1, 1), 64),
                                          (16, 2, "chain", 6)])
def test_attn_bwd_tensor_core_groups(Hq, Hkv, tree, T):
    # the tensor-core kernels (bf16, D = 128) at group sizes 1, 8 and 8 with 512 query rows per kv head (four
    # 128-row tiles), prefixes that end inside a tile, NaN junk past every tree block
    w, dout = make(Hq * T, B=2, T=T, Hq=Hq, Hkv=Hkv, D=128, L=(1, 700), dt="bf16", tree=tree)
    assert (check(w, dout) == 0).all()


def test_attn_bwd_tensor_core_statuses():
    w, dout = make(5, B=3, T=13, Hq=16, Hkv=4, D=128, L=(100, 400), dt="bf16", tree=(3, 2, 2))
    w.parent = w.parent.copy()
    w.kv_len = w.kv_len.copy()
    w.parent[1, 3] = 7
    w.kv_len[2] = -1
    assert list(check(w, dout)) == [0, 2, 1]
