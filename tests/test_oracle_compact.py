"""Pins for the oracle's KV compaction after acceptance (CPU only).

The expected values come from the attention definition, not from the compaction's own copy loop: a node
on the accepted path attends to the prefix, the root and its ancestors, which after compaction are the
contiguous positions [0, L + depth]; so the tree attention of that node over the ORIGINAL cache must equal
plain causal attention (a chain tree) over the COMPACTED cache.  Identity cases and status codes complete
the pins.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def verify_batch(seed, tree, T, kv_dt="bf16", B=6, Hq=4, Hkv=2, D=16, L=(0, 40)):
    return W.make_verify(seed, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, L=L, V=64, q_dt="f32" if kv_dt == "f32" else "bf16",
                         kv_dt=kv_dt, logit_dt="f32", tree=tree, mode="greedy", with_attn=True)


@pytest.mark.parametrize("kv_dt", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("tree,T", [((3, 2, 2), 13), ((4, 3, 2, 2, 1, 1), 40), ("star", 7)])
def test_path_nodes_see_a_causal_prefix_after_compaction(kv_dt, tree, T):
    w = verify_batch(11, tree, T, kv_dt)
    acc, path = W.random_root_paths(5, w.parent, stop_p=0.2)
    k2, v2, new_len, st, rc = oracle.kv_compact(w.k, w.v, w.kv_len, w.parent, acc, path, kv_dt=kv_dt)
    assert rc == 0 and (st == 0).all()
    assert (new_len == w.kv_len + 1 + acc).all()
    before, _, _, _ = oracle.tree_attn_w(w)
    # queries of the path nodes, placed on a chain: chain node j+1 carries path node path[j]'s query
    q_chain = np.array(w.q, copy=True)
    for b in range(w.B):
        for j in range(acc[b]):
            q_chain[b, j + 1] = w.q[b, path[b, j]]
    chain = np.stack([W.chain_tree(T) for _ in range(w.B)])
    after, _, _, _ = oracle.tree_attn(q_chain, k2, v2, w.kv_len, chain, Hq=w.Hq, Hkv=w.Hkv, q_dt=w.q_dt,
                                      kv_dt=kv_dt, k_scale=w.k_scale, v_scale=w.v_scale)
    checked = 0
    for b in range(w.B):
        np.testing.assert_allclose(after[b, 0], before[b, 0], rtol=0, atol=1e-12)   # the root itself
        for j in range(acc[b]):
            np.testing.assert_allclose(after[b, j + 1], before[b, path[b, j]], rtol=0, atol=1e-12)
            checked += 1
    assert checked > 0


def test_prefix_and_tail_positions_are_untouched():
    w = verify_batch(3, (3, 2, 2), 13)
    acc, path = W.random_root_paths(8, w.parent, stop_p=0.1)
    k2, v2, new_len, st, rc = oracle.kv_compact(w.k, w.v, w.kv_len, w.parent, acc, path, kv_dt="bf16")
    for b in range(w.B):
        lo = int(w.kv_len[b]) + 1
        hi = lo + int(acc[b])
        for src, dst in ((w.k, k2), (w.v, v2)):
            np.testing.assert_array_equal(dst[b, :, :lo], src[b, :, :lo])
            np.testing.assert_array_equal(dst[b, :, hi:], src[b, :, hi:])


def test_chain_with_everything_accepted_is_the_identity():
    w = verify_batch(4, "chain", 9)
    acc = np.full(w.B, 8, np.int32)
    path = np.tile(np.arange(-1, 8, dtype=np.int32), (w.B, 1))
    path[:, :8] = np.arange(1, 9)
    path[:, 8] = -1
    k2, v2, new_len, st, rc = oracle.kv_compact(w.k, w.v, w.kv_len, w.parent, acc, path, kv_dt="bf16")
    assert (st == 0).all() and (new_len == w.kv_len + 9).all()
    np.testing.assert_array_equal(k2, w.k)
    np.testing.assert_array_equal(v2, w.v)


def test_nothing_accepted_keeps_the_root_only():
    w = verify_batch(5, (2, 2), 7)
    acc = np.zeros(w.B, np.int32)
    path = np.full((w.B, 7), -1, np.int32)
    k2, v2, new_len, st, rc = oracle.kv_compact(w.k, w.v, w.kv_len, w.parent, acc, path, kv_dt="bf16")
    assert (st == 0).all() and (new_len == w.kv_len + 1).all()
    np.testing.assert_array_equal(k2, w.k)


def test_failed_or_inconsistent_requests_are_left_alone():
    w = verify_batch(6, (3, 2, 2), 13, B=5)
    acc, path = W.random_root_paths(2, w.parent, stop_p=0.0)       # full-depth paths
    acc = acc.copy()
    path = path.copy()
    parent = w.parent.copy()
    kv_len = w.kv_len.copy()
    acc[0] = -1                      # a failed verification
    path[1, 1] = path[1, 0]          # not a walk down the tree
    parent[2, 4] = 9                 # not topological
    kv_len[3] = w.kv_cap - 12        # kv_len + T > kv_cap
    k2, v2, new_len, st, rc = oracle.kv_compact(w.k, w.v, kv_len, parent, acc, path, kv_dt="bf16")
    assert list(st) == [1, 1, 2, 1, 0]
    assert (new_len[:4] == kv_len[:4]).all() and new_len[4] == kv_len[4] + 1 + acc[4]
    np.testing.assert_array_equal(k2[:4], w.k[:4])
    np.testing.assert_array_equal(v2[:4], w.v[:4])
