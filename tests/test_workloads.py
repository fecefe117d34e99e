"""The synthetic-input recipe (CPU only): the named workloads have the shapes, tree level sizes, length
ranges and statistical structure the configurations state, and the helper generators produce valid inputs.
The generators hold none of the method's arithmetic; these checks pin what they draw."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W


def depths(parent):
    st, d = oracle.tree_depth(parent)
    assert st == 0
    return d


@pytest.mark.parametrize("T,branching,levels", [(60, (4, 3, 2, 2, 1, 1), [1, 4, 12, 24, 17, 1, 1]),
                                                (64, (4, 3, 2, 2, 1, 1, 1), [1, 4, 12, 24, 20, 1, 1, 1]),
                                                (32, (4, 3, 2, 1, 1), [1, 4, 12, 13, 1, 1])])
def test_tree_level_sizes_of_the_named_trees(T, branching, levels):
    assert W.level_sizes(T, branching) == levels
    (rng,) = W.rng_streams(3, 1)
    for _ in range(5):
        p = W.make_tree(rng, T, branching)
        assert oracle.tree_check(p) == 0
        assert np.bincount(depths(p)).tolist() == levels
        # breadth-first numbering: depth never decreases with the node id
        assert (np.diff(depths(p)) >= 0).all()


def test_llama3_shaped_batch():
    """The recipe of the Llama3-shaped batch at a smaller vocabulary (the forced-argmax rate and the length
    range do not depend on it); the full-size shape is drawn once at 2 requests."""
    full = W.make_workload("llama3_8b_tree", seed=0, with_attn=False, B=2)
    assert full.target_logits.shape == (2, 60, 128256) and full.target_logits.dtype == np.uint16
    w = W.make_workload("llama3_8b_tree", seed=0, with_attn=False, B=40, V=4096)
    assert ((w.kv_len >= 2048) & (w.kv_len <= 8192)).all()
    # at an internal node, one child carries the row's argmax with probability 0.65
    z = W.bf16_to_f32(w.target_logits)
    arg = z.argmax(axis=-1)
    hits = total = 0
    for b in range(w.B):
        ch = W.children_of(w.parent[b])
        for p in range(w.T):
            if ch[p]:
                total += 1
                hits += int(arg[b, p]) in [int(w.tokens[b, c]) for c in ch[p]]
                toks = [int(w.tokens[b, c]) for c in ch[p]]
                assert len(set(toks)) == len(toks)                  # distinct sibling tokens
    assert abs(hits / total - 0.65) < 4 * np.sqrt(0.65 * 0.35 / total)


def test_qwen3_shaped_batch_correlation():
    w = W.make_workload("qwen3_8b_stochastic", seed=0, with_attn=False, B=2)
    zp = W.bf16_to_f32(w.target_logits).astype(np.float64).ravel()
    zq = W.bf16_to_f32(w.draft_logits).astype(np.float64).ravel()
    assert abs(np.corrcoef(zp, zq)[0, 1] - 0.8) < 0.01
    assert abs(zq.std() - 2.5) < 0.02 and abs(zp.std() - 2.5) < 0.02
    assert w.uniforms.shape == (2, 6) and w.temperature == 1.0


def test_loss_batch_accepted_edge_fraction():
    lb = W.make_workload("loss_batch", seed=0, V=2048)      # the edge statistics do not depend on V
    assert lb.logits.shape == (64 * 32, 2048)
    acc = tot = 0
    for n in range(lb.N):
        for j in range(1, lb.T):
            tot += 1
            acc += int(lb.tokens[n, j] == lb.labels[n, lb.parent[n, j]])
    assert abs(acc / tot - 0.45) < 0.05


def test_fp8_long_context_shapes():
    w = W.make_workload("fp8_long_context", seed=0, with_attn=False, B=3, V=4096)
    assert ((w.kv_len >= 8192) & (w.kv_len <= 32768)).all()
    assert np.bincount(depths(w.parent[0])).tolist() == [1, 4, 12, 24, 20, 1, 1, 1]


def test_e4m3_encoding_rounds_to_nearest_and_saturates():
    x = np.array([0.0, 1.0, 1.0625, 1.1875, 448.0, 1000.0, -3.3, 2.0 ** -9, 2.0 ** -10 * 1.5])
    codes = W.f32_to_e4m3(x)
    vals = np.where(codes & 0x80, -1.0, 1.0) * W._E4M3_POS[np.minimum(codes & 0x7F, 126)]
    # 1.0625 is halfway between 1.0 and 1.125: ties to the even code (1.0)
    np.testing.assert_array_equal(vals, [0.0, 1.0, 1.0, 1.25, 448.0, 448.0, -3.25, 2.0 ** -9, 2.0 ** -9])


def test_random_root_paths_are_walks_down_the_tree():
    (rng,) = W.rng_streams(5, 1)
    parent = np.stack([W.make_tree(rng, 40, (4, 3, 2, 2, 1, 1)) for _ in range(50)])
    acc, path = W.random_root_paths(9, parent, stop_p=0.3, full_p=0.2)
    for b in range(50):
        n = int(acc[b])
        up = 0
        for j in range(n):
            assert parent[b, path[b, j]] == up
            up = path[b, j]
        assert (path[b, n:] == -1).all()
    assert acc.min() == 0 and acc.max() >= 3 and (acc <= depths(parent[0]).max() + 1).all()


def test_pages_cover_every_used_position_once():
    (rng,) = W.rng_streams(2, 1)
    cache = rng.standard_normal((3, 2, 70, 4)).astype(np.float32)
    kv_len = np.array([10, 40, 64], np.int32)
    pool, table = W.to_pages(4, cache, kv_len, 6, 16, extra_pages=2, junk=np.float32(np.nan))
    used = table[table >= 0]
    assert len(set(used.tolist())) == len(used) == pool.shape[0] - 2
    for b in range(3):
        for j in range(int(kv_len[b]) + 6):
            np.testing.assert_array_equal(pool[table[b, j // 16], :, j % 16], cache[b, :, j])


def test_expansion_levels_follow_the_level_budget():
    levels = W.expansion_levels(60, (4, 3, 2, 2, 1, 1))
    assert levels == [(1, 4, 4), (4, 3, 12), (12, 2, 24), (24, 2, 17), (17, 1, 1), (1, 1, 1)]
    e = W.make_expand(1, B=2, n_front=4, V=100, k=3, n_keep=12, ties=2)
    assert e.logits.shape == (2, 4, 100) and (e.front_score <= 0).all()
    z = W.bf16_to_f32(e.logits)
    assert ((z == z.max(axis=-1, keepdims=True)).sum(axis=-1) >= 3).all()   # the planted copies of the max
