"""GPU parity of sv_tree_attn against the oracle (float64): element by element on small shapes that span
several KV tiles with ragged tails, and on sampled (request, node, head) rows of the named workloads at
full size.  Tolerances: max-abs 2e-2 for bf16 outputs, 6e-2 with FP8 E4M3 KV, 1e-4 for float32 outputs
(fp32 arithmetic throughout)."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev, host_f32, run_attn

pytestmark = pytest.mark.gpu


def tol(w):
    if w.kv_dt == "e4m3":
        return 6e-2
    return 2e-2 if w.q_dt == "bf16" else 1e-4


def check_full(w, sm_scale=0.0):
    out, lse, st = run_attn(w, sm_scale)
    ref_o, ref_l, ref_st, _ = oracle.tree_attn_w(w, sm_scale=sm_scale)
    np.testing.assert_array_equal(st, ref_st)
    ok = ref_st == 0
    err = np.abs(out[ok] - ref_o[ok]).max()
    assert err <= tol(w), err
    assert np.abs(lse[ok] - ref_l[ok]).max() <= (1e-3 if w.q_dt == "bf16" else 1e-5)
    return out, st


def check_sampled(w, n_rows=384, seed=0):
    out, lse, st = run_attn(w)
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, w.B, n_rows), rng.integers(0, w.T, n_rows), rng.integers(0, w.Hq, n_rows)], 1)
    # every node of one whole request too (all tree depths, all heads)
    b0 = int(rng.integers(0, w.B))
    extra = np.array([[b0, i, h] for i in range(w.T) for h in range(0, w.Hq, max(1, w.Hq // 8))])
    rows = np.concatenate([rows, extra]).astype(np.int32)
    ref_o, ref_l, ref_st, _ = oracle.tree_attn_w(w, rows=rows)
    assert (st == 0).all() and (ref_st == 0).all()
    b, i, h = rows.T
    err = np.abs(out[b, i, h] - ref_o[b, i, h]).max()
    assert err <= tol(w), err
    assert np.abs(lse[b, i, h] - ref_l[b, i, h]).max() <= (1e-3 if w.q_dt == "bf16" else 1e-5)


SMALL = [
    # B, T, Hq, Hkv, D, L, tree, q_dt, kv_dt
    (2, 6, 4, 1, 64, (0, 0), "chain", "f32", "f32"),
    (3, 6, 4, 1, 64, (100, 300), "chain", "f32", "f32"),
    (2, 13, 8, 2, 128, (1, 517), (3, 2, 2), "bf16", "bf16"),
    (2, 60, 32, 8, 128, (120, 700), (4, 3, 2, 2, 1, 1), "bf16", "bf16"),
    (3, 9, 16, 2, 128, (200, 333), (4, 2), "bf16", "e4m3"),
    (1, 64, 8, 8, 64, (0, 100), (4, 3, 2, 2, 1, 1, 1), "bf16", "bf16"),
    (2, 1, 8, 1, 128, (1, 1000), "chain", "bf16", "bf16"),
    (2, 20, 4, 2, 64, (31, 33), "star", "f32", "bf16"),
    (2, 7, 6, 3, 96, (50, 90), (2, 2, 1), "bf16", "bf16"),
    # tensor-core path with Q loaded by the 3D TMA box (G = 1 in split mode, G = 16 with 320 rows per kv
    # head: a pair unit and a split-mode unit), and with Q written by the softmax warps because G does not divide the
    # 128-row M tile (G = 3 in split mode; G = 6 in pair mode)
    (2, 40, 4, 4, 128, (70, 400), (4, 3, 2), "bf16", "bf16"),
    (2, 20, 32, 2, 128, (64, 300), (4, 2, 2), "bf16", "bf16"),
    (2, 11, 9, 3, 128, (90, 400), (3, 2, 2), "bf16", "bf16"),
    (2, 30, 12, 2, 128, (130, 600), (3, 3, 2, 2), "bf16", "bf16"),
]


@pytest.mark.parametrize("case", SMALL)
def test_attn_parity_small(case):
    B, T, Hq, Hkv, D, L, tree, qdt, kvdt = case
    w = W.make_verify(sum(L) + T, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, L=L, V=64, q_dt=qdt, kv_dt=kvdt, tree=tree)
    check_full(w)


def test_attn_ignores_nan_junk_beyond_the_tree():
    w = W.make_verify(5, B=3, T=9, Hq=8, Hkv=2, D=128, L=(60, 260), V=64, q_dt="bf16", kv_dt="bf16", tree=(3, 2),
                      junk="nan", kv_cap=400)
    out, _ = check_full(w)
    assert np.isfinite(out).all()


def test_attn_sm_scale_override():
    w = W.make_verify(6, B=2, T=6, Hq=4, Hkv=2, D=64, L=(40, 80), V=64, q_dt="f32", kv_dt="f32", tree=(2, 2))
    check_full(w, sm_scale=0.05)


def test_attn_status_codes():
    w = W.make_verify(7, B=4, T=5, Hq=4, Hkv=2, D=64, L=(10, 20), V=64, q_dt="bf16", kv_dt="bf16", tree=(2, 2))
    w.parent = w.parent.copy()
    w.kv_len = w.kv_len.copy()
    w.parent[1, 4] = 4
    w.kv_len[2] = w.kv_cap - 2
    w.kv_len[3] = -1
    out, lse, st = run_attn(w)
    assert list(st) == [0, 2, 1, 1]
    assert (out[1:] == 0).all() and (lse[1:] == 0).all()


@pytest.mark.parametrize("name", ["tiny_chain"])
def test_named_small_workload_full(name):
    check_full(W.make_workload(name, seed=0))


@pytest.mark.parametrize("name", ["llama3_8b_tree", "qwen3_8b_stochastic"])
def test_named_workloads_full_size_sampled(name):
    check_sampled(W.make_workload(name, seed=0))


# E4M3 caches with bf16 Q and D = 128 run on the tensor cores (e4m3 -> f16 conversion in shared memory):
# ragged prefixes, trees up to 64 nodes, and config-5 head shapes, with NaN junk past every tree block.
FP8_TC = [
    # B, T, Hq, Hkv, L, tree
    (1, 1, 4, 4, (0, 0), "chain"),
    (2, 6, 8, 2, (100, 300), "chain"),
    (3, 13, 16, 2, (1, 700), (3, 2, 2)),
    (2, 60, 32, 8, (2048, 3000), (4, 3, 2, 2, 1, 1)),
    (2, 64, 64, 8, (8192, 9000), (4, 3, 2, 2, 1, 1, 1)),
    (2, 11, 9, 3, (90, 400), (3, 2, 2)),        # G = 3: the softmax warps write Q (rounded to f16)
    (2, 20, 32, 2, (64, 300), (4, 2, 2)),       # 320 rows per kv head: one pair unit and one split unit
]


@pytest.mark.parametrize("case", FP8_TC)
def test_attn_fp8_tensor_core_parity(case):
    B, T, Hq, Hkv, L, tree = case
    w = W.make_verify(300 + sum(L) + T, B=B, T=T, Hq=Hq, Hkv=Hkv, D=128, L=L, V=64, q_dt="bf16", kv_dt="e4m3",
                      tree=tree, junk="nan")
    if B * T * Hq > 4000:
        check_sampled(w)
    else:
        out, _ = check_full(w)
        assert np.isfinite(out).all()


def test_fp8_long_context_attention_sampled():
    # config-5 requests (T=64, 64/8 heads, e4m3 KV, L in [8192, 32768]) at 16 requests drawn on the host
    check_sampled(W.make_workload("fp8_long_context", seed=0, B=16))


def test_fp8_long_context_full_batch_sampled_rows():
    # the whole 128-request batch in the launch configuration the bench times (drawn on the GPU by the generator's
    # device recipe); the oracle recomputes sampled rows of 12 requests, the first and last included, and every
    # node of one of them at 8 heads
    w = W.make_workload("fp8_long_context", seed=0, device="cuda")
    out, lse, st = run_attn(w)
    assert (st == 0).all()
    rng = np.random.default_rng(7)
    reqs = sorted({0, w.B - 1, *[int(x) for x in rng.choice(w.B, 10, replace=False)]})
    h = W.host_requests(w, reqs, with_logits=False)
    rows = [[j, int(rng.integers(0, w.T)), int(rng.integers(0, w.Hq))] for j in range(len(reqs)) for _ in range(24)]
    rows += [[1, i, hh] for i in range(w.T) for hh in range(0, w.Hq, 8)]
    rows = np.array(rows, np.int32)
    ref_o, ref_l, ref_st, _ = oracle.tree_attn_w(h, rows=rows)
    assert (ref_st == 0).all()
    j, i, hh = rows.T
    b = np.asarray(reqs)[j]
    err = np.abs(out[b, i, hh] - ref_o[j, i, hh]).max()
    assert err <= 6e-2, err
    assert np.abs(lse[b, i, hh] - ref_l[j, i, hh]).max() <= 1e-3


def test_attn_workspace_any_content_and_reuse():
    # The partial results of units that cross CTA range boundaries, and the records the merge kernel reads, live
    # in the workspace: a workspace of arbitrary bytes works on its first call, and reusing it, with calls of
    # another shape in between, gives bit-identical results.  Short prefixes make almost every unit span several
    # CTAs.
    import torch
    from speculative_decoding_tree_verify_gb300 import sv

    def call(w, ws):
        q, k, v = dev(w.q), dev(w.k), dev(w.v)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        sv.tree_attn(q, k, v, dev(w.kv_len), dev(w.parent), out, lse=lse, status=st, workspace=ws)
        torch.cuda.synchronize()
        return host_f32(out, w.q_dt), lse.cpu().numpy(), st.cpu().numpy()

    w1 = W.make_verify(11, B=4, T=60, Hq=32, Hkv=8, D=128, L=(300, 1500), V=64, q_dt="bf16", kv_dt="bf16",
                       tree=(4, 3, 2, 2, 1, 1))
    w2 = W.make_verify(12, B=5, T=13, Hq=8, Hkv=2, D=128, L=(100, 900), V=64, q_dt="bf16", kv_dt="bf16",
                       tree=(3, 2, 2))
    n = max(sv.workspace_size(sv.OP_TREE_ATTN, w.B, w.T, w.Hq, w.Hkv, w.D, w.kv_cap, 0) for w in (w1, w2))
    g = torch.Generator(device="cuda").manual_seed(5)
    ref = {}
    for w in (w1, w2):
        o, l, s, _ = oracle.tree_attn_w(w)
        ref[id(w)] = (o, l, s)
    for fill in ("random", "ones", "zeros"):
        if fill == "random":
            ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
        else:
            ws = torch.full((n,), 255 if fill == "ones" else 0, dtype=torch.uint8, device="cuda")
        first = {}
        for rep in range(3):
            for w in (w1, w2):
                out, lse, st = call(w, ws)
                o, l, s = ref[id(w)]
                np.testing.assert_array_equal(st, s)
                assert np.abs(out - o).max() <= 2e-2, (fill, rep)
                assert np.abs(lse - l).max() <= 1e-3, (fill, rep)
                if rep == 0:
                    first[id(w)] = (out, lse)
                else:
                    assert np.array_equal(out, first[id(w)][0]) and np.array_equal(lse, first[id(w)][1])
