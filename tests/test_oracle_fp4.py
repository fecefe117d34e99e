"""Pins for the oracle's FP4 (E2M1) KV caches (CPU only).

The caches are decoded a second way, in numpy from the OCP E2M1 magnitude list (0, 0.5, 1, 1.5, 2, 3, 4, 6)
and the generator's E4M3 value table, with the packing stated in the header (two codes a byte, the even
element in the low nibble; one E4M3 block scale per 16 elements of a row; an fp32 scale per kv head).  With
power-of-two head scales every decoded value is exact in float32, so the FP4 attention must equal the plain
float32-cache attention on the decoded values to rounding of the float64 sums.  Swapping the nibbles or
shifting the block mapping changes the output, so both conventions are pinned."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def decode_fp4(packed, bcode, hs):
    B, H, cap, half = packed.shape
    codes = np.stack([packed & 15, packed >> 4], axis=-1).reshape(B, H, cap, 2 * half)
    mag = W.E2M1_POS[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    bval = W._E4M3_POS[np.minimum(bcode & 0x7F, 126)]
    bval = np.where(bcode & 0x80, -bval, bval)
    return val * np.repeat(bval, 16, axis=-1) * np.asarray(hs, np.float64)[None, :, None, None]


def batch(seed, tree, T, D=32):
    w = W.make_verify(seed, B=3, T=T, Hq=4, Hkv=2, D=D, L=(5, 70), V=32, q_dt="f32", kv_dt="f32", logit_dt="f32",
                      tree=tree, mode="greedy", with_attn=True)
    kp, kb, ks = W.encode_nvfp4(w.k, pow2_head_scale=True)
    vp, vb, vs = W.encode_nvfp4(w.v, pow2_head_scale=True)
    return w, (kp, vp, kb, vb, ks, vs)


@pytest.mark.parametrize("tree,T", [((3, 2, 2), 13), ("chain", 6), ((4, 3, 2, 2, 1, 1), 30)])
def test_fp4_attention_equals_attention_on_independently_decoded_caches(tree, T):
    w, (kp, vp, kb, vb, ks, vs) = batch(T, tree, T)
    out, lse, st, rc = oracle.tree_attn_e2m1(w.q, kp, vp, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32")
    assert rc == 0 and (st == 0).all()
    kd = decode_fp4(kp, kb, ks).astype(np.float32)
    vd = decode_fp4(vp, vb, vs).astype(np.float32)
    assert np.array_equal(kd.astype(np.float64), decode_fp4(kp, kb, ks))    # exact in float32
    ref, ref_lse, _, _ = oracle.tree_attn(w.q, kd, vd, w.kv_len, w.parent, Hq=w.Hq, Hkv=w.Hkv, q_dt="f32", kv_dt="f32")
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_nibble_order_and_block_mapping_are_pinned():
    w, (kp, vp, kb, vb, ks, vs) = batch(2, (3, 2, 2), 13)
    base, _, _, _ = oracle.tree_attn_e2m1(w.q, kp, vp, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32")
    swapped = ((vp & 15) << 4 | (vp >> 4)).astype(np.uint8)
    out_s, _, _, _ = oracle.tree_attn_e2m1(w.q, kp, swapped, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32")
    rolled = np.roll(vb, 1, axis=-1)
    out_r, _, _, _ = oracle.tree_attn_e2m1(w.q, kp, vp, kb, rolled, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32")
    assert np.abs(out_s - base).max() > 1e-3 and np.abs(out_r - base).max() > 1e-3


def test_e2m1_encoding_rounds_to_nearest_even_and_saturates():
    x = np.array([0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.3, -6.5])
    codes = W.f32_to_e2m1_codes(x)
    mag = W.E2M1_POS[codes & 7]
    vals = np.where(codes & 8, -mag, mag)
    # 0.25 -> 0 (tie, even code 0); 0.75 -> 1.0 (tie between codes 1 and 2: even code 2); 1.25 -> 1.0;
    # 1.75 -> 2.0; 2.5 -> 2.0; 3.5 -> 4.0; 5.0 -> 4.0; saturation at 6
    np.testing.assert_array_equal(vals, [0.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.5, -6.0])


def test_fp4_statuses():
    w, (kp, vp, kb, vb, ks, vs) = batch(4, (2, 2), 7)
    parent = w.parent.copy()
    kv_len = w.kv_len.copy()
    parent[0, 3] = 6
    kv_len[1] = w.kv_cap
    out, lse, st, rc = oracle.tree_attn_e2m1(w.q, kp, vp, kb, vb, ks, vs, kv_len, parent, Hq=w.Hq, q_dt="f32")
    assert list(st) == [2, 1, 0]


def test_fp4_sampled_rows_equal_the_full_computation():
    # the sampled-row form (used by the full-size GPU parity tests) computes exactly the listed rows
    w, (kp, vp, kb, vb, ks, vs) = batch(5, (3, 2, 2), 13)
    full, full_lse, _, _ = oracle.tree_attn_e2m1(w.q, kp, vp, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32")
    rows = np.array([[2, 12, 3], [0, 0, 0], [2, 5, 1], [1, 7, 2]], np.int32)
    out, lse, st, rc = oracle.tree_attn_e2m1(w.q, kp, vp, kb, vb, ks, vs, w.kv_len, w.parent, Hq=w.Hq, q_dt="f32",
                                             rows=rows)
    assert rc == 0
    b, i, h = rows.T
    np.testing.assert_array_equal(out[b, i, h], full[b, i, h])
    np.testing.assert_array_equal(lse[b, i, h], full_lse[b, i, h])
    mask = np.ones(lse.shape, bool)
    mask[b, i, h] = False
    assert np.isnan(lse[mask]).all()
