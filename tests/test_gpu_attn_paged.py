"""GPU parity of sv_tree_attn_paged: the attention over caches scattered into a page pool in random order
(unused pool pages hold NaN) against the oracle over the same pages, within the forward's tolerance
(2e-2 max-abs for bf16 / fp32 inputs, 6e-2 for e4m3 caches); for fp32 inputs, bit-identical to the contiguous
call, which runs the same CUDA-core arithmetic.  bf16 / e4m3 pools with D = 128 run on the tensor-core kernel
(TMA boxes gathered page by page, pages of 8 to 512 rows); D = 64 and fp32 on the CUDA-core kernel."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev, host_f32, run_attn

pytestmark = pytest.mark.gpu

NAN = {"f32": np.float32(np.nan), "bf16": np.uint16(0x7FC0), "e4m3": np.uint8(0x7F)}


def run_paged(w, kp, vp, table):
    q = dev(w.q)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
    st = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    sv.tree_attn_paged(q, dev(kp), dev(vp), dev(table), dev(w.kv_len), dev(w.parent), out, k_scale=dev(w.k_scale),
                       v_scale=dev(w.v_scale), lse=lse, status=st)
    torch.cuda.synchronize()
    return host_f32(out, w.q_dt), lse.cpu().numpy().astype(np.float64), st.cpu().numpy()


def pages(w, P, seed):
    kp, table = W.to_pages(seed, w.k, w.kv_len, w.T, P, junk=NAN[w.kv_dt])
    vp, _ = W.to_pages(seed, w.v, w.kv_len, w.T, P, junk=NAN[w.kv_dt])
    return kp, vp, table


@pytest.mark.parametrize("kv_dt", ["f32", "bf16", "e4m3"])
@pytest.mark.parametrize("P", [8, 16, 64, 128, 256, 512])
@pytest.mark.parametrize("D,Hq,Hkv,tree,T", [(128, 32, 8, (4, 3, 2, 2, 1, 1), 60), (64, 8, 2, "chain", 6),
                                             (128, 16, 2, (3, 2, 2), 13)])
def test_paged_parity(kv_dt, P, D, Hq, Hkv, tree, T):
    q_dt = "f32" if kv_dt == "f32" else "bf16"
    w = W.make_verify(P + D + T, B=4, T=T, Hq=Hq, Hkv=Hkv, D=D, L=(0, 700), V=32, q_dt=q_dt, kv_dt=kv_dt,
                      logit_dt="f32", tree=tree, mode="greedy", with_attn=True, junk="nan")
    kp, vp, table = pages(w, P, P + T)
    ref, ref_lse, ref_st, _ = oracle.tree_attn_paged(w.q, kp, vp, table, w.kv_len, w.parent, Hq=Hq, Hkv=Hkv, q_dt=q_dt,
                                                     kv_dt=kv_dt, k_scale=w.k_scale, v_scale=w.v_scale)
    out, lse, st = run_paged(w, kp, vp, table)
    np.testing.assert_array_equal(st, ref_st)
    tol = 6e-2 if kv_dt == "e4m3" else 2e-2
    assert np.max(np.abs(out - ref)) <= tol
    assert np.max(np.abs(lse - ref_lse)) <= 1e-3


def test_paged_fp32_is_bitwise_the_contiguous_call():
    w = W.make_verify(5, B=3, T=13, Hq=8, Hkv=2, D=64, L=(100, 400), V=32, q_dt="f32", kv_dt="f32", logit_dt="f32",
                      tree=(3, 2, 2), mode="greedy", with_attn=True, junk="nan")
    kp, vp, table = pages(w, 32, 1)
    out_p, lse_p, st_p = run_paged(w, kp, vp, table)
    out_c, lse_c, st_c = run_attn(w)
    assert (st_p == 0).all() and (st_c == 0).all()
    np.testing.assert_array_equal(out_p, out_c)
    np.testing.assert_array_equal(lse_p, lse_c)


def test_paged_statuses():
    w = W.make_verify(6, B=3, T=6, Hq=4, Hkv=1, D=64, L=(10, 60), V=32, q_dt="bf16", kv_dt="bf16", logit_dt="f32",
                      tree="chain", mode="greedy", with_attn=True)
    kp, vp, table = pages(w, 16, 3)
    table = table.copy()
    table[0, 1] = kp.shape[0] + 5
    w.kv_len = w.kv_len.copy()
    w.kv_len[2] = table.shape[1] * 16
    out, lse, st = run_paged(w, kp, vp, table)
    assert list(st) == [1, 0, 1]
    assert not out[0].any() and not out[2].any()


@pytest.mark.parametrize("kv_dt", ["bf16", "e4m3"])
def test_paged_tensor_core_statuses(kv_dt):
    # a page id outside the pool and a capacity overrun on the tensor-core path: status 1 and zero outputs, the
    # other request exact
    w = W.make_verify(8, B=3, T=13, Hq=16, Hkv=2, D=128, L=(100, 600), V=32, q_dt="bf16", kv_dt=kv_dt, logit_dt="f32",
                      tree=(3, 2, 2), mode="greedy", with_attn=True, junk="nan")
    kp, vp, table = pages(w, 64, 4)
    table = table.copy()
    table[0, 1] = kp.shape[0] + 5
    w.kv_len = w.kv_len.copy()
    w.kv_len[2] = table.shape[1] * 64
    out, lse, st = run_paged(w, kp, vp, table)
    assert list(st) == [1, 0, 1]
    assert not out[0].any() and not out[2].any()
    ref, ref_lse, ref_st, _ = oracle.tree_attn_paged(w.q, kp, vp, table, w.kv_len, w.parent, Hq=w.Hq, Hkv=w.Hkv,
                                                     q_dt="bf16", kv_dt=kv_dt, k_scale=w.k_scale, v_scale=w.v_scale)
    assert list(ref_st) == [1, 0, 1]
    assert np.abs(out[1] - ref[1]).max() <= (6e-2 if kv_dt == "e4m3" else 2e-2)


def test_paged_tensor_core_full_size_sampled():
    # the Llama3-shaped batch in 128-row pages on the tensor-core kernel; the oracle checks sampled rows
    w = W.make_workload("llama3_8b_tree", seed=0)
    kp, vp, table = pages(w, 128, 9)
    out, lse, st = run_paged(w, kp, vp, table)
    assert (st == 0).all()
    rng = np.random.default_rng(3)
    rows = np.stack([rng.integers(0, w.B, 256), rng.integers(0, w.T, 256), rng.integers(0, w.Hq, 256)], 1).astype(np.int32)
    ref, ref_lse, _, _ = oracle.tree_attn_w(w, rows=rows)
    b, i, h = rows.T
    assert np.abs(out[b, i, h] - ref[b, i, h]).max() <= 2e-2
    assert np.abs(lse[b, i, h] - ref_lse[b, i, h]).max() <= 1e-3
