"""GPU parity of sv_tree_attn_fp4 (FP4 caches in the NVFP4 layout: E2M1 codes, E4M3 block scales per 16
elements, fp32 head scales) against the oracle's attention over the same codes, float64.

Tolerance: max-abs 2e-2 on the output (the bf16 bar).  The oracle and the kernel see the same quantised cache
values, and each of them (a 2-bit-mantissa code times a 4-bit-mantissa scale) is exactly an f16 value, so the
kernel's only roundings are those of the bf16 path: Q to f16 (exact for these inputs), P to f16, fp32 sums and
the bf16 output.  The log-sum-exp within 1e-3.  Cache rows past each tree block hold NaN block scales and random
codes, which must not reach the output."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev, host_f32

pytestmark = pytest.mark.gpu


def fp4_batch(seed, B, T, Hq, Hkv, L, tree):
    kv_cap = (L[1] + T + 1) // 2 * 2          # the FP4 call wants an even capacity (two scale rows per TMA row)
    w = W.make_verify(seed, B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, L=L, V=16, q_dt="bf16", kv_dt="f32", logit_dt="f32",
                      tree=tree, mode="greedy", kv_cap=kv_cap)
    kc, kb, ks = W.encode_nvfp4(w.k)
    vc, vb, vs = W.encode_nvfp4(w.v)
    junk = np.arange(w.kv_cap)[None, None, :] >= (w.kv_len[:, None, None] + T)      # [B, 1, cap]
    kb = np.where(junk[..., None], np.uint8(0x7F), kb)      # NaN block scales past the tree block
    vb = np.where(junk[..., None], np.uint8(0x7F), vb)
    return w, (kc, vc, kb, vb, ks, vs)


def run_fp4(w, c):
    kc, vc, kb, vb, ks, vs = c
    q = dev(w.q)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
    st = torch.full((w.B,), -9, dtype=torch.int32, device="cuda")
    sv.tree_attn_fp4(q, dev(kc), dev(vc), dev(kb), dev(vb), dev(ks), dev(vs), dev(w.kv_len), dev(w.parent), out, lse=lse,
                     status=st)
    torch.cuda.synchronize()
    return host_f32(out, "bf16"), lse.cpu().numpy().astype(np.float64), st.cpu().numpy()


CASES = [
    # B, T, Hq, Hkv, L, tree: one tile, split mode (<= 128 query rows per kv head), pair mode (240 rows), two units
    # per kv head (512 rows), G = 3 (Q written by the softmax warps), empty prefixes and ragged tails
    (2, 1, 4, 4, (0, 0), "chain"),
    (3, 6, 8, 2, (100, 300), "chain"),
    (2, 13, 16, 2, (1, 700), (3, 2, 2)),
    (2, 60, 32, 8, (900, 1500), (4, 3, 2, 2, 1, 1)),
    (1, 64, 64, 8, (2000, 2100), (4, 3, 2, 2, 1, 1, 1)),
    (2, 11, 9, 3, (90, 400), (3, 2, 2)),
]


@pytest.mark.parametrize("case", CASES)
def test_fp4_parity(case):
    B, T, Hq, Hkv, L, tree = case
    w, c = fp4_batch(700 + sum(L) + T, B, T, Hq, Hkv, L, tree)
    out, lse, st = run_fp4(w, c)
    kc, vc, kb, vb, ks, vs = c
    ref, ref_lse, ref_st, rc = oracle.tree_attn_e2m1(w.q, kc, vc, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq,
                                                     q_dt="bf16")
    assert rc == 0
    np.testing.assert_array_equal(st, ref_st)
    assert (st == 0).all()
    assert np.isfinite(out).all()
    err = np.abs(out - ref).max()
    assert err <= 2e-2, err
    assert np.abs(lse - ref_lse).max() <= 1e-3


def test_fp4_statuses():
    w, c = fp4_batch(11, 3, 7, 8, 2, (10, 200), (2, 2))
    w.parent = w.parent.copy()
    w.kv_len = w.kv_len.copy()
    w.parent[0, 3] = 6
    w.kv_len[1] = w.kv_cap - 3
    out, lse, st = run_fp4(w, c)
    assert list(st) == [2, 1, 0]
    assert not out[:2].any() and not lse[:2].any()


def test_fp4_odd_capacity_is_refused():
    w, c = fp4_batch(3, 1, 1, 4, 4, (0, 0), "chain")
    kc, vc, kb, vb, ks, vs = c
    q = dev(w.q)
    with pytest.raises(sv.SVError) as e:
        sv.tree_attn_fp4(q, dev(kc[:, :, :1]).contiguous(), dev(vc[:, :, :1]).contiguous(), dev(kb[:, :, :1]).contiguous(),
                         dev(vb[:, :, :1]).contiguous(), dev(ks), dev(vs), dev(w.kv_len), dev(w.parent), torch.empty_like(q))
    assert e.value.code == sv.ERR_UNSUPPORTED
