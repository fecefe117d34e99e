"""Pins for the paged form of the oracle's tree attention (CPU only): reading the cache through a random
page table must give exactly (bit for bit) the attention over the contiguous cache it was scattered from,
for every page size; bad page ids and a capacity overrun are reported per request."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


@pytest.mark.parametrize("kv_dt", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("P", [1, 16, 64])
def test_paged_equals_contiguous(kv_dt, P):
    w = W.make_verify(P + 3, B=4, T=13, Hq=4, Hkv=2, D=16, L=(0, 90), V=32, q_dt="bf16", kv_dt=kv_dt,
                      logit_dt="f32", tree=(3, 2, 2), mode="greedy", with_attn=True)
    kp, table = W.to_pages(7, w.k, w.kv_len, w.T, P)
    vp, _ = W.to_pages(7, w.v, w.kv_len, w.T, P)
    ref, ref_lse, ref_st, _ = oracle.tree_attn_w(w)
    got, lse, st, rc = oracle.tree_attn_paged(w.q, kp, vp, table, w.kv_len, w.parent, Hq=w.Hq, Hkv=w.Hkv,
                                              q_dt=w.q_dt, kv_dt=kv_dt, k_scale=w.k_scale, v_scale=w.v_scale)
    assert rc == 0 and (st == 0).all() and (ref_st == 0).all()
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(lse, ref_lse)


def test_paged_statuses():
    w = W.make_verify(1, B=3, T=6, Hq=2, Hkv=1, D=8, L=(10, 40), V=32, q_dt="f32", kv_dt="f32", logit_dt="f32",
                      tree="chain", mode="greedy", with_attn=True)
    kp, table = W.to_pages(2, w.k, w.kv_len, w.T, 8)
    table = table.copy()
    table[0, 0] = kp.shape[0]                    # a page id past the pool
    kv_len = w.kv_len.copy()
    kv_len[2] = table.shape[1] * 8               # kv_len + T beyond the table's capacity
    out, lse, st, rc = oracle.tree_attn_paged(w.q, kp, kp, table, kv_len, w.parent, Hq=2, Hkv=1, q_dt="f32",
                                              kv_dt="f32")
    assert list(st) == [1, 0, 1]
    assert not out[0].any() and not out[2].any() and out[1].any()
