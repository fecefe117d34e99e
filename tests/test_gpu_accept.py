"""GPU parity of sv_accept against the oracle: every output bit-exact (accept_len, path, out_tokens, bonus,
argmax, status), greedy and stochastic, small shapes with ragged vocabularies and every named workload at
full size."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import run_accept

pytestmark = pytest.mark.gpu

KEYS = ("status", "accept_len", "path", "out_tokens", "bonus", "argmax")


def compare(g, o):
    for k in KEYS:
        if g.get(k) is None:
            continue
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)


AUTO = object()


def check(w, temperature=None, draft=AUTO):
    t = w.temperature if temperature is None else temperature
    d = w.draft_logits if draft is AUTO else draft
    d = d if t > 0 else None
    ref = oracle.accept(w.target_logits, w.tokens, w.parent, V=w.V, logit_dt=w.logit_dt, temperature=t, draft=d,
                        uniforms=w.uniforms)
    got = run_accept(w.target_logits, w.tokens, w.parent, V=w.V, temperature=t, draft=d, uniforms=w.uniforms)
    compare(got, ref)
    return got


TREES = [("chain", 8), ((3, 2, 2), 13), ("star", 10), ((2, 2, 2, 2, 1), 25), ((4, 3, 2, 2, 1, 1, 1), 64)]


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("V", [16, 1000, 4096, 40000])
@pytest.mark.parametrize("tree,T", TREES)
def test_greedy_parity(dt, V, tree, T):
    if tree == "star" and T > V:
        pytest.skip("star needs V >= T")
    w = W.make_verify(V + T, B=23, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree=tree, mode="greedy",
                      force_p=0.7, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("mode", ["prob", "onehot"])
@pytest.mark.parametrize("temp", [1.0, 0.7, 1e-3])
@pytest.mark.parametrize("V,dt", [(16, "f32"), (1000, "bf16"), (4096, "bf16"), (50000, "bf16")])
@pytest.mark.parametrize("tree,T", [("chain", 6), ((3, 2, 2), 13), ("star", 5)])
def test_stochastic_parity(mode, temp, V, dt, tree, T):
    w = W.make_verify(V * 7 + T, B=19, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree=tree,
                      mode="prob" if mode == "prob" else "onehot", temperature=temp, force_p=0.7, sigma=2.0,
                      with_attn=False)
    g = check(w, temperature=temp, draft=w.draft_logits if mode == "prob" else None)
    assert (g["status"] == 0).all()


# Trees of 16 nodes or more: the row kernel leaves the weight sums to the walk, which computes them for the
# rows it visits only (the chains and small trees above take the sums in the row pass).
LAZY_TREES = [((2, 2, 2, 2, 1), 25), ((4, 3, 2, 2, 1, 1, 1), 64), ("star", 16)]


@pytest.mark.parametrize("mode", ["prob", "onehot"])
@pytest.mark.parametrize("temp", [1.0, 1e-3])
@pytest.mark.parametrize("V,dt", [(16, "f32"), (1000, "bf16"), (4099, "f32"), (50000, "bf16")])
@pytest.mark.parametrize("tree,T", LAZY_TREES)
def test_stochastic_parity_walk_sums(mode, temp, V, dt, tree, T):
    if tree == "star" and T > V:
        pytest.skip("star needs V >= T")
    w = W.make_verify(V * 5 + T, B=19, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree=tree,
                      mode=mode, temperature=temp, force_p=0.7, sigma=2.5, with_attn=False)
    g = check(w, temperature=temp, draft=w.draft_logits if mode == "prob" else None)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("mode", ["prob", "onehot"])
def test_stochastic_parity_walk_sums_full_vocabulary(mode):
    V, T = 151936, 25
    w = W.make_verify(V + 5, B=7, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt="bf16", tree=(2, 2, 2, 2, 1),
                      mode=mode, temperature=0.6, force_p=0.7, sigma=2.5, with_attn=False)
    g = check(w, temperature=0.6, draft=w.draft_logits if mode == "prob" else None)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("mode", ["prob", "onehot"])
def test_walk_sums_wide_range_and_statuses(mode):
    """Trees of 25 nodes: rows holding a logit about 4e6 below the rest take the scalar weights in the walk's
    own sum pass; non-finite logits and y overflow fail their request whether or not the walk visits the row."""
    w = W.make_verify(31, B=8, T=25, Hq=1, Hkv=1, D=8, L=(0, 0), V=3000, logit_dt="bf16", tree=(2, 2, 2, 2, 1),
                      mode=mode, temperature=0.9, force_p=0.8, sigma=2.0, with_attn=False)
    w.target_logits = w.target_logits.copy()
    low = W.f32_to_bf16(np.float32(-4.0e6))
    w.target_logits[::2, :, 17] = low
    if mode == "prob":
        w.draft_logits = w.draft_logits.copy()
        w.draft_logits[1::3, :, 2999] = low
    for want in (False, True):
        g = check_opts(w, 0.9, w.draft_logits if mode == "prob" else None, want)
        assert (g["status"] == 0).all()
    w.target_logits[1, 24, 100] = 0x7FC0                                  # NaN in a leaf row
    w.target_logits[2, 0, 5] = 0xFF80                                     # -inf in the root row
    w.target_logits[3, 13, 2047] = W.f32_to_bf16(np.float32(3.0e37))[0]   # y = 3.3e37 / 0.9 stays finite
    w.target_logits[4, 7, 1] = W.f32_to_bf16(np.float32(3.3e38))[0]       # y overflows float32
    g = check_opts(w, 0.9, w.draft_logits if mode == "prob" else None, True)
    assert list(g["status"]) == [0, 5, 5, 0, 5, 0, 0, 0]


@pytest.mark.parametrize("V,dt,temp", [(151936, "bf16", 1.0), (50000, "bf16", 0.8), (4096, "f32", 0.7),
                                       (40003, "bf16", 1.0), (128256, "bf16", 0.3)])
def test_bonus_draw_at_prefix_boundaries_walk_sums(V, dt, temp):
    """Trees of 17 nodes (ONEHOT, the walk computes the sums): the root's only child carries a token whose
    target weight is 0, so it is always rejected and the bonus is drawn from a residual equal to the root's row;
    the slot-0 uniform on a prefix-sum boundary of that row pins the walk's sums and prefix sums to the unit."""
    T = 17
    w = W.make_verify(V + 91, B=48, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree="chain",
                      mode="onehot", temperature=temp, force_p=0.0, sigma=2.5, with_attn=False)   # no forced peaks
    w.target_logits = w.target_logits.copy()
    w.parent = np.full((w.B, T), 1, np.int32)
    w.parent[:, 0] = -1
    w.parent[:, 1] = 0
    w.tokens = w.tokens.copy()
    low = np.ravel(W.f32_to_bf16(np.float32(-4.0e6)))[0] if dt == "bf16" else np.float32(-4.0e6)
    for b in range(w.B):
        x = (7 * b + 5) % V
        w.tokens[b, 1] = x
        w.target_logits[b, 0, x] = low                 # weight 0: the child is rejected whatever its uniform
    w.target_logits[1::4, 0, 3] = low                  # a quarter of the rows span more than 2^21 in y
    u = w.uniforms.copy()
    u[:, 0] = boundary_uniforms(w, temp, V)[:, 0]
    w.uniforms = u
    for want in (False, True):
        g = check_opts(w, temp, None, want)
        assert (g["status"] == 0).all() and (g["accept_len"] == 0).all()


@pytest.mark.parametrize("V,dt,temp", [(151936, "bf16", 1.0), (4096, "f32", 0.7), (40003, "bf16", 0.5)])
def test_bonus_draw_after_duplicate_rejections_walk_sums(V, dt, temp):
    """Trees of 17 nodes (ONEHOT, the walk computes the sums): the root's two children carry the same token x
    (the root row's second-largest logit) with uniforms that reject any token short of all the mass, so x is
    rejected twice and taken out of the residual once; the slot-0 uniform on a prefix-sum boundary of that
    residual (the row with x's weight set to 0) pins the residual's sums to the unit."""
    T = 17
    w = W.make_verify(V + 13, B=40, T=T, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree="chain",
                      mode="onehot", temperature=temp, force_p=0.0, sigma=2.5, with_attn=False)
    w.target_logits = w.target_logits.copy()
    w.parent = np.full((w.B, T), 1, np.int32)
    w.parent[:, 0] = -1
    w.parent[:, 2] = 0
    w.parent[:, 1] = 0
    w.tokens = w.tokens.copy()
    xs = []
    for b in range(w.B):
        z = W.decode_f32(w.target_logits[b, 0], w.logit_dt)
        x = int(np.argsort(z, kind="stable")[-2])
        xs.append(x)
        w.tokens[b, 1] = w.tokens[b, 2] = x
    u = w.uniforms.copy()
    u[:, 1] = u[:, 2] = 0xFFFFFFFF
    resid = W.make_verify(V + 13, B=w.B, T=1, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree="chain",
                          mode="onehot", temperature=temp, with_attn=False)
    resid.target_logits = w.target_logits[:, :1].copy()
    low = np.ravel(W.f32_to_bf16(np.float32(-4.0e6)))[0] if dt == "bf16" else np.float32(-4.0e6)
    for b, x in enumerate(xs):
        resid.target_logits[b, 0, x] = low               # the residual: x's weight 0, the row maximum unchanged
    u[:, 0] = boundary_uniforms(resid, temp, V + 1)[:, 0]
    w.uniforms = u
    for want in (False, True):
        g = check_opts(w, temp, None, want)
        assert (g["status"] == 0).all() and (g["accept_len"] == 0).all()
        assert all(int(g["bonus"][b]) != x for b, x in enumerate(xs))


def test_single_node_trees():
    for t in (0.0, 1.0):
        w = W.make_verify(3, B=9, T=1, Hq=1, Hkv=1, D=8, L=(0, 0), V=777, logit_dt="bf16", tree="chain",
                          mode="greedy" if t == 0 else "onehot", temperature=t, with_attn=False)
        g = check(w, temperature=t, draft=None)
        assert (g["accept_len"] == 0).all()


def test_status_codes_bad_tree_token_nonfinite():
    w = W.make_verify(4, B=6, T=7, Hq=1, Hkv=1, D=8, L=(0, 0), V=300, logit_dt="f32", tree=(2, 2, 1), mode="onehot",
                      temperature=1.0, with_attn=False)
    w.parent = w.parent.copy()
    w.tokens = w.tokens.copy()
    w.target_logits = w.target_logits.copy()
    w.parent[1, 3] = 5                 # not topological
    w.parent[2, 0] = 0                 # root must have parent -1
    w.tokens[3, 4] = 300               # token out of range
    w.target_logits[4, 2, 17] = np.nan
    w.target_logits[5, 6, 0] = -np.inf
    for t in (0.0, 1.0):
        g = check(w, temperature=t, draft=None)
        assert list(g["status"]) == [0, 2, 2, 1, 5, 5]
        assert (g["accept_len"][1:] == -1).all()


@pytest.mark.parametrize("name", ["tiny_chain", "llama3_8b_tree"])
def test_named_greedy_workloads_full_size(name):
    w = W.make_workload(name, seed=0, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()
    if w.B > 1:
        assert g["accept_len"].mean() > 0


def test_qwen3_stochastic_full_size():
    w = W.make_workload("qwen3_8b_stochastic", seed=0, with_attn=False)
    g = check(w)
    assert (g["status"] == 0).all()


@pytest.mark.parametrize("temp", [0.0, 0.7])
def test_fp8_long_context_accept_full_size(temp):
    w = W.make_workload("fp8_long_context", seed=0, with_attn=False, mode="greedy" if temp == 0 else "onehot",
                        temperature=temp)
    g = check(w, temperature=temp, draft=None)
    assert (g["status"] == 0).all()


def check_opts(w, temperature, draft, want_argmax):
    ref = oracle.accept(w.target_logits, w.tokens, w.parent, V=w.V, logit_dt=w.logit_dt, temperature=temperature,
                        draft=draft, uniforms=w.uniforms, want_argmax=want_argmax)
    got = run_accept(w.target_logits, w.tokens, w.parent, V=w.V, temperature=temperature, draft=draft,
                     uniforms=w.uniforms, want_argmax=want_argmax)
    compare(got, ref)
    return got


@pytest.mark.parametrize("want_argmax", [False, True])
@pytest.mark.parametrize("mode", ["prob", "onehot"])
@pytest.mark.parametrize("V", [1000, 50000, 1001, 40003])
def test_stochastic_bf16_with_and_without_argmax(want_argmax, mode, V):
    """bf16 rows whose length keeps them 16-byte aligned take the shared-memory staged kernel (with or
    without the argmax output); other lengths take the generic kernel."""
    w = W.make_verify(V + 3, B=17, T=13, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt="bf16", tree=(3, 2, 2),
                      mode=mode, temperature=0.8, force_p=0.7, sigma=2.5, with_attn=False)
    g = check_opts(w, 0.8, w.draft_logits if mode == "prob" else None, want_argmax)
    assert (g["status"] == 0).all()


def test_stochastic_rows_with_a_very_wide_logit_range():
    """Rows holding a logit about 4e6 below the rest (|t| beyond 2^21) take the scalar contract path of the
    staged kernel; the results must not change."""
    w = W.make_verify(21, B=9, T=6, Hq=1, Hkv=1, D=8, L=(0, 0), V=4096, logit_dt="bf16", tree="chain", mode="prob",
                      temperature=1.0, sigma=2.5, with_attn=False)
    w.target_logits = w.target_logits.copy()
    w.draft_logits = w.draft_logits.copy()
    low = W.f32_to_bf16(np.float32(-4.0e6))
    w.target_logits[::2, :, 17] = low
    w.draft_logits[1::3, :, 4000] = low
    for want in (False, True):
        g = check_opts(w, 1.0, w.draft_logits, want)
        assert (g["status"] == 0).all()


def test_stochastic_bf16_status_codes_and_overflow():
    """NaN and infinite bf16 logits, and finite logits whose y = z / temperature overflows: the request fails
    with SV_ERR_NONFINITE, while the argmax of a finite row is still reported."""
    w = W.make_verify(8, B=5, T=6, Hq=1, Hkv=1, D=8, L=(0, 0), V=2048, logit_dt="bf16", tree="chain", mode="onehot",
                      temperature=0.05, sigma=2.0, with_attn=False)
    w.target_logits = w.target_logits.copy()
    w.target_logits[1, 3, 100] = 0x7FC0                     # NaN
    w.target_logits[2, 0, 5] = 0xFF80                       # -inf
    w.target_logits[3, 5, 2047] = W.f32_to_bf16(np.float32(3.0e37))[0]   # y = 6e38 overflows float32
    g = check_opts(w, 0.05, None, True)
    assert list(g["status"]) == [0, 5, 5, 5, 0]
    assert g["argmax"][3, 5] == 2047 and g["argmax"][1, 3] == -1


def boundary_uniforms(w, temperature, seed, wide_rows=()):
    """Slot-0 uniform of every request placed at a prefix-sum boundary of the row its bonus is drawn from
    (T = 1: the root's row, R = S): alternately just below and exactly at cs[j] * 2^32 / S for a token j in
    the upper half of the mass.  An error of one unit in S moves the threshold across the boundary, and an
    error in any weight before j moves the prefix sum; either changes the drawn token."""
    rng = np.random.default_rng(seed)
    invT = np.float32(1.0 / np.float64(temperature))
    u = np.zeros((w.B, 1), np.uint32)
    for b in range(w.B):
        z = W.decode_f32(w.target_logits[b, 0], w.logit_dt)
        y = (z * invT).astype(np.float32)
        wts = oracle.fx_weight(y, float(y.max())).astype(np.uint64)
        S = int(wts.sum())
        cs = np.cumsum(wts)
        cand = np.nonzero((wts > 0) & (cs * 2 >= S) & (cs < S))[0]
        if cand.size == 0:   # the last token of weight > 0 holds the upper half: any inner boundary
            cand = np.nonzero((wts > 0) & (cs < S))[0]
        j = int(rng.choice(cand))
        up = -(-(int(cs[j]) << 32) // S)               # ceil(cs[j] * 2^32 / S)
        u[b, 0] = up - 1 if b % 2 == 0 else up
        assert 0 < u[b, 0] < 2 ** 32
    return u


@pytest.mark.parametrize("V,dt,temp,mode", [(151936, "bf16", 1.0, "prob"), (151936, "bf16", 0.7, "onehot"),
                                            (50000, "bf16", 0.8, "onehot"), (4096, "f32", 0.7, "onehot"),
                                            (40003, "bf16", 1.0, "onehot"), (128256, "bf16", 0.3, "onehot")])
def test_bonus_draw_at_prefix_boundaries_checks_every_weight(V, dt, temp, mode):
    """Single-node trees: the walk stops at the root at once and draws the bonus from the root's row with
    R = S, so the drawn token pins the row's weight sum and the prefix sums to the unit."""
    w = W.make_verify(V + 77, B=48, T=1, Hq=1, Hkv=1, D=8, L=(0, 0), V=V, logit_dt=dt, tree="chain",
                      mode="prob" if mode == "prob" else "onehot", temperature=temp, sigma=2.5, with_attn=False)
    if mode == "prob":
        w.draft_logits = w.draft_logits.copy()
    w.target_logits = w.target_logits.copy()
    low = W.f32_to_bf16(np.float32(-4.0e6)) if dt == "bf16" else np.float32(-4.0e6)
    w.target_logits[1::4, 0, 3] = low                  # a quarter of the rows span more than 2^21 in y
    w.uniforms = boundary_uniforms(w, temp, V)
    for want in (False, True):
        g = check_opts(w, temp, w.draft_logits if mode == "prob" else None, want)
        assert (g["status"] == 0).all() and (g["accept_len"] == 0).all()
