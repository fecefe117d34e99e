"""GPU parity of sv_kv_compact against the oracle: every byte of both caches, new_kv_len and status must be
identical (the call moves bytes, so the bar is bit-exactness), on ragged small shapes, every kv dtype,
failed requests, and the tree blocks of the Llama3-shaped and FP8 long-context batches at full size."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu


def run_compact(k, v, kv_len, parent, accept_len, path):
    kd, vd = dev(k), dev(v)
    B = parent.shape[0]
    new_len = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    status = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    sv.kv_compact(kd, vd, dev(kv_len), dev(parent), dev(accept_len), dev(path), new_len, status=status)
    torch.cuda.synchronize()
    as_np = lambda t: t.cpu().numpy().view(k.dtype)
    return as_np(kd), as_np(vd), new_len.cpu().numpy(), status.cpu().numpy()


def check(k, v, kv_len, parent, accept_len, path, kv_dt):
    rk, rv, rlen, rst, rc = oracle.kv_compact(k, v, kv_len, parent, accept_len, path, kv_dt=kv_dt)
    assert rc == 0
    gk, gv, glen, gst = run_compact(k, v, kv_len, parent, accept_len, path)
    np.testing.assert_array_equal(gst, rst)
    np.testing.assert_array_equal(glen, rlen)
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)
    return gst


@pytest.mark.parametrize("kv_dt,D", [("f32", 64), ("bf16", 128), ("bf16", 72), ("e4m3", 128), ("e4m3", 16)])
@pytest.mark.parametrize("tree,T", [("chain", 9), ((3, 2, 2), 13), ("star", 6), ((4, 3, 2, 2, 1, 1, 1), 64)])
def test_compact_parity(kv_dt, D, tree, T):
    w = W.make_verify(T * 31 + D, B=11, T=T, Hq=3, Hkv=3, D=D, L=(0, 90), V=64, q_dt="bf16", kv_dt=kv_dt,
                      logit_dt="f32", tree=tree, mode="greedy", with_attn=True)
    acc, path = W.random_root_paths(T + D, w.parent, stop_p=0.25)
    st = check(w.k, w.v, w.kv_len, w.parent, acc, path, kv_dt)
    assert (st == 0).all()


def test_compact_statuses_leave_failed_requests_untouched():
    w = W.make_verify(5, B=6, T=13, Hq=2, Hkv=2, D=64, L=(3, 50), V=64, kv_dt="bf16", logit_dt="f32",
                      tree=(3, 2, 2), mode="greedy", with_attn=True)
    acc, path = W.random_root_paths(1, w.parent, stop_p=0.0)
    acc, path, parent, kv_len = acc.copy(), path.copy(), w.parent.copy(), w.kv_len.copy()
    acc[0] = -1
    path[1, 1] = path[1, 0]
    parent[2, 4] = 9
    kv_len[3] = w.kv_cap - 12
    acc[4] = 13                      # more than T - 1
    st = check(w.k, w.v, kv_len, parent, acc, path, "bf16")
    assert list(st) == [1, 1, 2, 1, 1, 0]


def test_compact_after_oracle_acceptance_llama3_shape_full_size():
    """The Llama3-shaped batch at full size (8 requests, 8 kv heads, D=128 bf16, prefixes up to 8192), with
    the accepted paths the oracle's greedy acceptance gives on the batch's own logits."""
    w = W.make_workload("llama3_8b_tree", seed=0)
    acc = oracle.accept_w(w)
    assert (acc["status"] == 0).all()
    st = check(w.k, w.v, w.kv_len, w.parent, acc["accept_len"], acc["path"], "bf16")
    assert (st == 0).all()


def test_compact_fp8_long_context_full_size_tree_blocks():
    """FP8 long-context shape at full size (128 requests, 8 kv heads, D=128 e4m3, kv_cap 32832).  The call
    only touches positions kv_len .. kv_len+T-1, so the oracle runs on those tree blocks (cropped, kv_len 0)
    and the rest of each cache must stay exactly as it was (zero here)."""
    B, T, Hkv, D = 128, 64, 8, 128
    s_len, s_blk, s_tree = W.rng_streams(77, 3)
    kv_len = s_len.integers(8192, 32768, size=B, endpoint=True).astype(np.int32)
    cap = 32768 + T
    parent = np.stack([W.make_tree(s_tree, T, (4, 3, 2, 2, 1, 1, 1)) for _ in range(B)])
    acc, path = W.random_root_paths(78, parent, stop_p=0.15)
    blk_k = s_blk.integers(0, 256, size=(B, Hkv, T, D), dtype=np.uint8)
    blk_v = s_blk.integers(0, 256, size=(B, Hkv, T, D), dtype=np.uint8)
    kd = torch.zeros((B, Hkv, cap, D), dtype=torch.uint8, device="cuda")
    vd = torch.zeros_like(kd)
    for b in range(B):
        L = int(kv_len[b])
        kd[b, :, L:L + T] = torch.from_numpy(blk_k[b]).cuda()
        vd[b, :, L:L + T] = torch.from_numpy(blk_v[b]).cuda()
    new_len = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    status = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    sv.kv_compact(kd, vd, dev(kv_len), dev(parent), dev(acc), dev(path), new_len, status=status)
    torch.cuda.synchronize()
    rk, rv, rlen, rst, rc = oracle.kv_compact(blk_k, blk_v, np.zeros(B, np.int32), parent, acc, path, kv_dt="e4m3")
    assert rc == 0 and (rst == 0).all()
    np.testing.assert_array_equal(status.cpu().numpy(), rst)
    np.testing.assert_array_equal(new_len.cpu().numpy(), kv_len + 1 + acc)
    for b in range(B):
        L = int(kv_len[b])
        np.testing.assert_array_equal(kd[b, :, L:L + T].cpu().numpy(), rk[b])
        np.testing.assert_array_equal(vd[b, :, L:L + T].cpu().numpy(), rv[b])
        kd[b, :, L:L + T] = 0
        vd[b, :, L:L + T] = 0
    assert int(torch.count_nonzero(kd)) == 0 and int(torch.count_nonzero(vd)) == 0
