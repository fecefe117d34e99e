"""Seeded synthetic inputs for speculative tree verification.

This module only *draws* inputs: draft trees (parent arrays), draft tokens, KV caches, logits, labels and
the raw 32-bit uniforms of the acceptance test.  It holds none of the verification arithmetic (no
attention, no acceptance rule, no loss), so it can feed both the CPU oracle and the CUDA library with
the same bytes.

Every tensor comes from its own child stream of ``numpy.random.SeedSequence(seed)`` driving a Philox
bit generator, spawned in a fixed order, so a (workload, seed) pair always produces the same bytes.

Encodings handed to both sides:
  * ``f32``  : float32 array
  * ``bf16`` : uint16 array holding bfloat16 bit patterns (rounded to nearest even from float32)
  * ``e4m3`` : uint8 array holding OCP FP8 E4M3 codes (round to nearest even, saturating at 448), with a
               float32 scale per KV head: real value = decoded code * scale[h].

Tree shape (the pages give node count, depth and branching only; this is the reading used everywhere):
level sizes n_d = min(n_{d-1} * k_d, rem - (depth - d)) with rem starting at T - 1; level d takes n_d
distinct (parent, rank) slots drawn uniformly from the n_{d-1} * k_d candidates; nodes are numbered
breadth-first by (parent, rank), so parent[i] < i and node 0 is the root (the last committed token).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "bf16", "e4m3")


# ----------------------------------------------------------------------------------------------------
# streams and encodings
# ----------------------------------------------------------------------------------------------------
def rng_streams(seed: int, k: int) -> list[np.random.Generator]:
    """k independent Philox streams spawned from one seed, in a fixed order."""
    return [np.random.Generator(np.random.Philox(s)) for s in np.random.SeedSequence(seed).spawn(k)]


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (inputs are finite)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(h) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _e4m3_positive_table() -> np.ndarray:
    # codes 0..126 (0x7F is NaN); value = (8+m) * 2^(e-10) for e >= 1, m * 2^-9 for e == 0
    vals = np.empty(127, np.float64)
    for c in range(127):
        e, m = c >> 3, c & 7
        vals[c] = m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)
    return vals


_E4M3_POS = _e4m3_positive_table()


def f32_to_e4m3(x) -> np.ndarray:
    """float -> E4M3 codes, round to nearest even, saturating to +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 1, 126)
    lo = hi - 1
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi)
    code = np.where(a >= _E4M3_POS[126], 126, code)
    return (code | np.where(x < 0, 0x80, 0)).astype(np.uint8)


# OCP E2M1 magnitudes by code 0..7 (sign in bit 3)
E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def f32_to_e2m1_codes(x) -> np.ndarray:
    """float -> E2M1 codes 0..15, round to nearest (ties to the even code), saturating at +-6."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(E2M1_POS, a, side="left"), 1, 7)
    lo = hi - 1
    d_lo = a - E2M1_POS[lo]
    d_hi = E2M1_POS[hi] - a
    code = np.where((d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0)), lo, hi)
    code = np.where(a >= 6.0, 7, code)
    return (code | np.where(x < 0, 8, 0)).astype(np.uint8)


def encode_nvfp4(x, pow2_head_scale: bool = False):
    """A float32 cache [B, Hkv, cap, D] (D a multiple of 16) -> (codes [B,Hkv,cap,D/2] with the even element in
    the low nibble, E4M3 block scales [B,Hkv,cap,D/16], fp32 head scales [Hkv]).  Head scale
    amax / (6 * 448) (or the next power of two above it), block scale = E4M3(block amax / 6 / head scale), codes =
    E2M1(x / (block * head)).  Data encoding only."""
    x = np.asarray(x, np.float32)
    B, H, cap, D = x.shape
    amax = np.maximum(np.abs(x).max(axis=(0, 2, 3)).astype(np.float64), 1e-30)
    hs = amax / (6.0 * 448.0)
    if pow2_head_scale:
        hs = 2.0 ** np.ceil(np.log2(hs))
    hs = hs.astype(np.float32)
    blocks = x.reshape(B, H, cap, D // 16, 16).astype(np.float64)
    bamax = np.abs(blocks).max(axis=-1)
    bcode = f32_to_e4m3(bamax / 6.0 / hs[None, :, None, None].astype(np.float64))
    bval = _E4M3_POS[np.minimum(bcode & 0x7F, 126)]
    denom = bval[..., None] * hs[None, :, None, None, None].astype(np.float64)
    q = np.where(denom > 0, blocks / np.where(denom > 0, denom, 1.0), 0.0)
    codes = f32_to_e2m1_codes(q).reshape(B, H, cap, D)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, bcode.astype(np.uint8), hs


def encode(x, dt: str) -> np.ndarray:
    if dt == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dt == "bf16":
        return f32_to_bf16(x)
    raise ValueError(dt)


def decode_f32(a, dt: str) -> np.ndarray:
    """Decode an f32/bf16 encoded array to float32 (used by the generator to place forced maxima)."""
    return np.asarray(a, np.float32) if dt == "f32" else bf16_to_f32(a)


# ----------------------------------------------------------------------------------------------------
# trees
# ----------------------------------------------------------------------------------------------------
def level_sizes(T: int, branching) -> list[int]:
    depth = len(branching)
    rem = T - 1
    sizes = [1]
    for d in range(1, depth + 1):
        n = min(sizes[-1] * branching[d - 1], rem - (depth - d))
        if n < 1:
            raise ValueError(f"tree T={T} branching={branching} cannot reach depth {depth}")
        sizes.append(n)
        rem -= n
    if rem != 0:
        raise ValueError(f"tree T={T} branching={branching} leaves {rem} nodes unplaced")
    return sizes


def make_tree(rng: np.random.Generator, T: int, branching) -> np.ndarray:
    """Topological parent array (int32 [T], parent[0] = -1), BFS-numbered by (parent, rank)."""
    sizes = level_sizes(T, branching)
    parent = [-1]
    prev = [0]
    for d in range(1, len(sizes)):
        k = branching[d - 1]
        cand = [(p, r) for p in prev for r in range(k)]
        pick = np.sort(rng.choice(len(cand), size=sizes[d], replace=False))
        prev = []
        for i in pick:
            parent.append(cand[i][0])
            prev.append(len(parent) - 1)
    return np.asarray(parent, np.int32)


def chain_tree(T: int) -> np.ndarray:
    return np.arange(-1, T - 1, dtype=np.int32)


def star_tree(T: int) -> np.ndarray:
    p = np.zeros(T, np.int32)
    p[0] = -1
    return p


def children_of(parent: np.ndarray) -> list[list[int]]:
    ch = [[] for _ in range(len(parent))]
    for i in range(1, len(parent)):
        ch[int(parent[i])].append(i)
    return ch


# ----------------------------------------------------------------------------------------------------
# verify workloads (attention + acceptance)
# ----------------------------------------------------------------------------------------------------
@dataclass
class Verify:
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    kv_cap: int
    V: int
    q_dt: str
    kv_dt: str
    logit_dt: str
    q: np.ndarray                 # [B,T,Hq,D]
    k: np.ndarray                 # [B,Hkv,kv_cap,D]
    v: np.ndarray                 # [B,Hkv,kv_cap,D]
    k_scale: np.ndarray | None    # [Hkv] float32 (e4m3 only)
    v_scale: np.ndarray | None
    kv_len: np.ndarray            # [B] int32 prefix length L_b; tree K/V at L_b .. L_b+T-1
    parent: np.ndarray            # [B,T] int32
    tokens: np.ndarray            # [B,T] int32, tokens[b,0] = root token
    target_logits: np.ndarray     # [B,T,V]
    draft_logits: np.ndarray | None
    uniforms: np.ndarray | None   # [B,T] uint32
    temperature: float
    name: str = ""
    meta: dict = field(default_factory=dict)


def _encode_kv(x, dt, kv_len, T, junk):
    """Encode a [B,Hkv,cap,D] float32 cache; positions >= kv_len+T hold junk (random, or NaN patterns)."""
    B, Hkv, cap, D = x.shape
    valid = (np.arange(cap)[None, :] < (kv_len[:, None] + T))  # [B,cap]
    scale = None
    if dt == "e4m3":
        amax = np.max(np.abs(np.where(valid[:, None, :, None], x, 0.0)), axis=(0, 2, 3))
        scale = (np.maximum(amax, 1e-30) / 448.0).astype(np.float32)
        enc = f32_to_e4m3(x / scale[None, :, None, None])
        if junk == "nan":
            enc = np.where(valid[:, None, :, None], enc, np.uint8(0x7F))
        return enc, scale
    enc = encode(x, dt)
    if junk == "nan":
        nan = np.float32(np.nan) if dt == "f32" else np.uint16(0x7FC0)
        enc = np.where(valid[:, None, :, None], enc, nan).astype(enc.dtype)
    return enc, scale


def _force_max(row_f32: np.ndarray, tok: int) -> float:
    """Value that makes `tok` the unique maximum of the row after encoding (max + 1)."""
    return float(np.max(row_f32)) + 1.0


def _draft_tokens(parents: np.ndarray, tokens: np.ndarray, V: int, force_p: float, s_tok, s_force):
    """Greedy / one-hot draft tokens, written into tokens[:, 1:]: the children of every internal node get
    distinct random tokens; with probability force_p one uniformly chosen child's token is the one the
    target row of the parent is made to peak at, otherwise a token outside the children is.  Returns the
    (request, parent node, peak token) triples, in the order the streams were drawn."""
    B, T = parents.shape
    peaks = []
    for b in range(B):
        ch = children_of(parents[b])
        for p in range(T):
            if not ch[p]:
                continue
            toks = s_tok.choice(V, size=len(ch[p]) + 1, replace=False)
            for c, x in zip(ch[p], toks[:-1]):
                tokens[b, c] = x
            if s_force.random() < force_p:
                star = int(tokens[b, ch[p][s_force.integers(0, len(ch[p]))]])
            else:
                star = int(toks[-1])
            peaks.append((b, p, star))
    return peaks


def make_verify(seed: int, *, B: int, T: int, Hq: int, Hkv: int, D: int, L: tuple[int, int], V: int,
                q_dt: str = "bf16", kv_dt: str = "bf16", logit_dt: str = "bf16", tree="chain",
                mode: str = "greedy", temperature: float = 0.0, force_p: float = 0.7, sigma: float = 3.0,
                rho: float = 0.8, kv_cap: int | None = None, junk: str = "randn", name: str = "",
                with_attn: bool = True) -> Verify:
    """Draw one verify batch.

    mode 'greedy' / 'onehot': at every internal node, with probability force_p one uniformly chosen child
    carries the token that is made the row's unique maximum (its logit is set to the row max + 1); otherwise
    a token outside the children is made the maximum.  Children's tokens are distinct.
    mode 'prob': draft logits z_q = sigma*e1 and target logits z_p = sigma*(rho*e1 + sqrt(1-rho^2)*e2);
    each child's token is drawn from softmax(z_q(parent)/temperature) by the Gumbel-max trick.
    """
    (s_tree, s_len, s_q, s_k, s_v, s_lp, s_lq, s_tok, s_u, s_force, s_junk) = rng_streams(seed, 11)
    if tree == "chain":
        parents = np.stack([chain_tree(T) for _ in range(B)])
    elif tree == "star":
        parents = np.stack([star_tree(T) for _ in range(B)])
    else:
        parents = np.stack([make_tree(s_tree, T, tree) for _ in range(B)])
    lo, hi = L
    kv_len = s_len.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    cap = int(kv_cap if kv_cap is not None else hi + T)
    if with_attn:
        q = encode(s_q.standard_normal(size=(B, T, Hq, D), dtype=np.float32), q_dt)
        kx = s_k.standard_normal(size=(B, Hkv, cap, D), dtype=np.float32)
        vx = s_v.standard_normal(size=(B, Hkv, cap, D), dtype=np.float32)
        k, k_scale = _encode_kv(kx, kv_dt, kv_len, T, junk)
        v, v_scale = _encode_kv(vx, kv_dt, kv_len, T, junk)
        del kx, vx
    else:
        q = k = v = None
        k_scale = v_scale = None

    tokens = np.zeros((B, T), np.int32)
    tokens[:, 0] = s_tok.integers(0, V, size=B)
    draft = None
    uniforms = None
    if mode == "prob":
        e1 = s_lq.standard_normal(size=(B, T, V), dtype=np.float32)
        e2 = s_lp.standard_normal(size=(B, T, V), dtype=np.float32)
        zq = encode(sigma * e1, logit_dt)
        zp = encode(sigma * (rho * e1 + math.sqrt(1.0 - rho * rho) * e2), logit_dt)
        del e1, e2
        zq_f = decode_f32(zq, logit_dt)
        tinv = 1.0 / temperature
        for b in range(B):
            ch = children_of(parents[b])
            for p in range(T):
                if not ch[p]:
                    continue
                g = s_tok.gumbel(size=(len(ch[p]), V))
                picks = np.argmax(zq_f[b, p][None, :].astype(np.float64) * tinv + g, axis=1)
                for c, x in zip(ch[p], picks):
                    tokens[b, c] = x
        target, draft = zp, zq
    else:
        zf = (sigma * s_lp.standard_normal(size=(B, T, V), dtype=np.float32))
        target = encode(zf, logit_dt)
        tf = decode_f32(target, logit_dt).copy()
        for b, p, star in _draft_tokens(parents, tokens, V, force_p, s_tok, s_force):
            tf[b, p, star] = _force_max(tf[b, p], star)
        target = encode(tf, logit_dt)
        del tf, zf
    if mode in ("prob", "onehot"):
        uniforms = s_u.integers(0, 2 ** 32, size=(B, T), dtype=np.uint32)
    return Verify(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, kv_cap=cap, V=V, q_dt=q_dt, kv_dt=kv_dt,
                  logit_dt=logit_dt, q=q, k=k, v=v, k_scale=k_scale, v_scale=v_scale, kv_len=kv_len,
                  parent=parents, tokens=tokens, target_logits=target, draft_logits=draft,
                  uniforms=uniforms, temperature=float(temperature if mode != "greedy" else 0.0),
                  name=name, meta=dict(mode=mode, tree=tree, L=L, seed=seed))


# ----------------------------------------------------------------------------------------------------
# verify workloads drawn on the GPU (full-size batches whose caches and logits are too large to draw
# on the host in reasonable time)
# ----------------------------------------------------------------------------------------------------
def _torch_gen(seq: np.random.SeedSequence, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seq.generate_state(1, np.uint64)[0] & 0x7FFFFFFFFFFFFFFF))
    return g


def make_verify_device(seed: int, *, B: int, T: int, Hq: int, Hkv: int, D: int, L: tuple[int, int], V: int,
                       q_dt: str = "bf16", kv_dt: str = "e4m3", logit_dt: str = "bf16", tree="chain",
                       mode: str = "greedy", temperature: float = 0.0, force_p: float = 0.7, sigma: float = 3.0,
                       kv_cap: int | None = None, name: str = "", with_attn: bool = True, device="cuda",
                       **_ignored) -> Verify:
    """The greedy / one-hot recipe of make_verify with the large tensors drawn on the GPU.

    The tree, the prefix lengths, the draft tokens, the forced peaks and the uniforms come from the same
    numpy streams as make_verify (so they are identical to the host recipe's).  Q, the caches and the target
    logits are drawn with torch's CUDA generator from their own child seeds:
      * Q ~ N(0,1) rounded to bf16;
      * K, V ~ N(0,1); e4m3 caches use the per-kv-head amax scale over the valid positions (< kv_len + T),
        codes by torch's float8_e4m3fn conversion of x / scale clamped to +-448; bf16 caches round x;
      * target logits sigma * N(0,1) rounded to bf16; at each internal node the peak token's logit is set
        to the row's maximum + 1 (in float32, then rounded to bf16), as in the host recipe.
    The returned Verify holds torch CUDA tensors in q, k, v, k_scale, v_scale and target_logits (bf16 bits
    as int16, e4m3 codes as uint8) and numpy arrays in kv_len, parent, tokens and uniforms.  Use
    host_requests() to copy a few requests to numpy for the oracle."""
    import torch
    if mode not in ("greedy", "onehot") or q_dt != "bf16" or logit_dt != "bf16" or kv_dt not in ("bf16", "e4m3"):
        raise ValueError("the device recipe covers greedy / one-hot batches with bf16 Q and logits")
    (s_tree, s_len, s_q, s_k, s_v, s_lp, s_lq, s_tok, s_u, s_force, s_junk) = rng_streams(seed, 11)
    seqs = np.random.SeedSequence(seed).spawn(11)
    if tree == "chain":
        parents = np.stack([chain_tree(T) for _ in range(B)])
    elif tree == "star":
        parents = np.stack([star_tree(T) for _ in range(B)])
    else:
        parents = np.stack([make_tree(s_tree, T, tree) for _ in range(B)])
    lo, hi = L
    kv_len = s_len.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    cap = int(kv_cap if kv_cap is not None else hi + T)
    q = k = v = k_scale = v_scale = None
    if with_attn:
        gq = _torch_gen(seqs[2], device)
        q = torch.randn((B, T, Hq, D), generator=gq, device=device).to(torch.bfloat16).view(torch.int16)
        valid = (torch.arange(cap, device=device)[None, :] < torch.as_tensor(kv_len, device=device)[:, None] + T)
        caches, scales = [], []
        for seq in (seqs[3], seqs[4]):
            g = _torch_gen(seq, device)
            c = torch.empty((B, Hkv, cap, D), dtype=torch.uint8 if kv_dt == "e4m3" else torch.int16, device=device)
            sc = torch.ones(Hkv, dtype=torch.float32, device=device)
            for h in range(Hkv):          # one kv head at a time bounds the float32 temporary
                x = torch.randn((B, cap, D), generator=g, device=device)
                if kv_dt == "e4m3":
                    amax = torch.where(valid[:, :, None], x.abs(), torch.zeros((), device=device)).amax()
                    sc[h] = torch.clamp(amax, min=1e-30) / 448.0
                    c[:, h] = (x / sc[h]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
                else:
                    c[:, h] = x.to(torch.bfloat16).view(torch.int16)
                del x
            caches.append(c)
            scales.append(sc if kv_dt == "e4m3" else None)
        k, v = caches
        k_scale, v_scale = scales
    tokens = np.zeros((B, T), np.int32)
    tokens[:, 0] = s_tok.integers(0, V, size=B)
    peaks = _draft_tokens(parents, tokens, V, force_p, s_tok, s_force)
    gz = _torch_gen(seqs[5], device)
    target = (sigma * torch.randn((B, T, V), generator=gz, device=device)).to(torch.bfloat16)
    if peaks:
        bi, pi, ti = (torch.as_tensor(np.array(x, np.int64), device=device) for x in zip(*peaks))
        rmax = target[bi, pi].float().amax(dim=-1)
        target[bi, pi, ti] = (rmax + 1.0).to(torch.bfloat16)
    target = target.view(torch.int16)
    uniforms = s_u.integers(0, 2 ** 32, size=(B, T), dtype=np.uint32) if mode == "onehot" else None
    return Verify(B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, kv_cap=cap, V=V, q_dt=q_dt, kv_dt=kv_dt, logit_dt=logit_dt,
                  q=q, k=k, v=v, k_scale=k_scale, v_scale=v_scale, kv_len=kv_len, parent=parents, tokens=tokens,
                  target_logits=target, draft_logits=None, uniforms=uniforms,
                  temperature=float(temperature if mode != "greedy" else 0.0), name=name,
                  meta=dict(mode=mode, tree=tree, L=L, seed=seed, device_recipe=True))


def host_requests(w: Verify, reqs, with_logits: bool = True) -> Verify:
    """The requests `reqs` of a batch drawn by make_verify_device, copied to numpy in the host encodings
    (bf16 as uint16 bits, e4m3 as uint8 codes), as a Verify of len(reqs) requests."""
    import torch
    idx = torch.as_tensor(np.asarray(reqs, np.int64), device=w.target_logits.device)

    def take(t, view=None):
        if t is None:
            return None
        a = t.index_select(0, idx).cpu().numpy()
        return a.view(np.uint16) if a.dtype == np.int16 else a

    r = np.asarray(reqs, np.int64)
    return Verify(B=len(r), T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, kv_cap=w.kv_cap, V=w.V, q_dt=w.q_dt, kv_dt=w.kv_dt,
                  logit_dt=w.logit_dt, q=take(w.q), k=take(w.k), v=take(w.v),
                  k_scale=None if w.k_scale is None else w.k_scale.cpu().numpy(),
                  v_scale=None if w.v_scale is None else w.v_scale.cpu().numpy(),
                  kv_len=w.kv_len[r], parent=w.parent[r], tokens=w.tokens[r],
                  target_logits=take(w.target_logits) if with_logits else None, draft_logits=None,
                  uniforms=None if w.uniforms is None else w.uniforms[r], temperature=w.temperature,
                  name=w.name, meta=dict(w.meta, requests=[int(x) for x in r]))


# ----------------------------------------------------------------------------------------------------
# loss workloads
# ----------------------------------------------------------------------------------------------------
@dataclass
class LossBatch:
    N: int
    T: int
    V: int
    logits: np.ndarray    # [N*T, V] bf16 bits
    tokens: np.ndarray    # [N,T] int32
    parent: np.ndarray    # [N,T] int32
    labels: np.ndarray    # [N,T] int32 (target argmax after each node)
    name: str = ""
    meta: dict = field(default_factory=dict)


def make_loss(seed: int, *, N: int, T: int, V: int, tree=(4, 3, 2, 1, 1), sigma: float = 3.0,
              accept_frac: float = 0.45, name: str = "") -> LossBatch:
    """Logged traces: at each internal node, with probability pi = min(1, accept_frac*(T-1)/n_internal)
    one uniformly chosen child carries the parent's label; the other children carry distinct tokens that
    differ from the label."""
    (s_tree, s_z, s_lab, s_tok, s_pi) = rng_streams(seed, 5)
    if tree == "chain":
        parents = np.stack([chain_tree(T) for _ in range(N)])
    else:
        parents = np.stack([make_tree(s_tree, T, tree) for _ in range(N)])
    logits = f32_to_bf16(sigma * s_z.standard_normal(size=(N * T, V), dtype=np.float32))
    labels = s_lab.integers(0, V, size=(N, T)).astype(np.int32)
    tokens = np.zeros((N, T), np.int32)
    tokens[:, 0] = s_tok.integers(0, V, size=N)
    for n in range(N):
        ch = children_of(parents[n])
        n_int = sum(1 for c in ch if c)
        pi = min(1.0, accept_frac * (T - 1) / max(n_int, 1))
        for p in range(T):
            if not ch[p]:
                continue
            lab = int(labels[n, p])
            pool = s_tok.choice(V - 1, size=len(ch[p]), replace=False)
            others = [int(x) + (1 if x >= lab else 0) for x in pool]   # distinct, never the label
            for c, x in zip(ch[p], others):
                tokens[n, c] = x
            if s_pi.random() < pi:
                tokens[n, ch[p][s_pi.integers(0, len(ch[p]))]] = lab
    return LossBatch(N=N, T=T, V=V, logits=logits, tokens=tokens, parent=parents, labels=labels,
                     name=name, meta=dict(tree=tree, seed=seed))


# ----------------------------------------------------------------------------------------------------
# paged KV caches
# ----------------------------------------------------------------------------------------------------
def to_pages(seed: int, cache: np.ndarray, kv_len: np.ndarray, T: int, page_size: int, extra_pages: int = 3,
             junk=None):
    """Scatter a contiguous cache [B, Hkv, kv_cap, D] into a page pool [num_pages, Hkv, page_size, D] with a
    random page table [B, max_pages] (max_pages = ceil(kv_cap / page_size)).  Every page a request uses
    (those covering positions < kv_len + T) gets a distinct pool page in random order; unused table entries
    are -1; the pool holds `extra_pages` pages nobody uses, filled with `junk` (or zeros).  Data layout only."""
    (s_perm,) = rng_streams(seed, 1)
    B, Hkv, cap, D = cache.shape
    max_pages = -(-cap // page_size)
    used = [-(-(int(kv_len[b]) + T) // page_size) for b in range(B)]
    num_pages = sum(used) + extra_pages
    perm = s_perm.permutation(num_pages)
    pool = np.zeros((num_pages, Hkv, page_size, D), dtype=cache.dtype)
    if junk is not None:
        pool[...] = junk
    table = np.full((B, max_pages), -1, np.int32)
    k = 0
    for b in range(B):
        for pg in range(used[b]):
            dst = int(perm[k])
            k += 1
            table[b, pg] = dst
            lo = pg * page_size
            n = min(page_size, cap - lo)
            pool[dst, :, :n] = cache[b, :, lo:lo + n]
    return pool, table


# ----------------------------------------------------------------------------------------------------
# KV compaction inputs: accepted root paths
# ----------------------------------------------------------------------------------------------------
def random_root_paths(seed: int, parent: np.ndarray, stop_p: float = 0.3, full_p: float = 0.2):
    """For every request a root path drawn by a random walk: from the current node, stop with probability
    stop_p, else step to a uniformly chosen child; with probability full_p the walk never stops early
    (it runs to a leaf).  Returns accept_len [B] int32 and path [B,T] int32 (-1 padded)."""
    s_walk, s_full = rng_streams(seed, 2)
    B, T = parent.shape
    accept_len = np.zeros(B, np.int32)
    path = np.full((B, T), -1, np.int32)
    for b in range(B):
        ch = children_of(parent[b])
        full = s_full.random() < full_p
        cur, n = 0, 0
        while ch[cur] and (full or s_walk.random() >= stop_p):
            cur = ch[cur][int(s_walk.integers(0, len(ch[cur])))]
            path[b, n] = cur
            n += 1
        accept_len[b] = n
    return accept_len, path


# ----------------------------------------------------------------------------------------------------
# draft tree expansion inputs: one level's frontier logits and path scores
# ----------------------------------------------------------------------------------------------------
@dataclass
class Expand:
    B: int
    n_front: int
    V: int
    k: int
    n_keep: int
    logit_dt: str
    logits: np.ndarray        # [B, n_front, V] draft logits of the frontier nodes
    front_score: np.ndarray   # [B, n_front] float32 path scores (sums of log-probabilities, <= 0)
    name: str = ""
    meta: dict = field(default_factory=dict)


def make_expand(seed: int, *, B: int, n_front: int, V: int, k: int, n_keep: int, logit_dt: str = "bf16",
                sigma: float = 3.0, score_range: float = 6.0, ties: int = 0, name: str = "") -> Expand:
    """Frontier logits ~ N(0, sigma^2) and path scores uniform in [-score_range, 0] (the root's is 0 when
    n_front == 1).  ties > 0 plants, in every row, `ties` extra copies of the row maximum at random
    positions so that the lower-token-first rule decides the order."""
    s_z, s_score, s_tie = rng_streams(seed, 3)
    zf = sigma * s_z.standard_normal(size=(B, n_front, V), dtype=np.float32)
    if ties:
        enc = decode_f32(encode(zf, logit_dt), logit_dt)
        for b in range(B):
            for s in range(n_front):
                pos = s_tie.choice(V, size=min(ties, V), replace=False)
                zf[b, s, pos] = enc[b, s].max()
        del enc
    logits = encode(zf, logit_dt)
    if n_front == 1:
        front = np.zeros((B, 1), np.float32)
    else:
        front = (-score_range * s_score.random(size=(B, n_front))).astype(np.float32)
    return Expand(B=B, n_front=n_front, V=V, k=k, n_keep=n_keep, logit_dt=logit_dt, logits=logits,
                  front_score=front, name=name, meta=dict(seed=seed, sigma=sigma))


def expansion_levels(T: int, branching) -> list[tuple[int, int, int]]:
    """(n_front, k, n_keep) of every level of a budgeted tree with the given node count and branching:
    the level sizes of the tree generator above, expanded level by level."""
    sizes = level_sizes(T, branching)
    return [(sizes[d - 1], branching[d - 1], sizes[d]) for d in range(1, len(sizes))]


# ----------------------------------------------------------------------------------------------------
# named workloads (the shapes of the pages' serving setups, with the recipe of the generators above)
# ----------------------------------------------------------------------------------------------------
WORKLOADS = {
    # B=1, chain of 5 drafts, 4/1 heads, D=64, fp32 QKV, L=128, fp32 logits V=1024, greedy
    "tiny_chain": dict(kind="verify", B=1, T=6, Hq=4, Hkv=1, D=64, L=(128, 128), V=1024, q_dt="f32",
                       kv_dt="f32", logit_dt="f32", tree="chain", mode="greedy", force_p=0.7, sigma=3.0),
    # Llama3-8B-shaped EAGLE tree: B=8, 60 nodes depth 6 (4/3/2/2/1/1), 32/8 heads, D=128, L in [2048,8192]
    "llama3_8b_tree": dict(kind="verify", B=8, T=60, Hq=32, Hkv=8, D=128, L=(2048, 8192), V=128256,
                           q_dt="bf16", kv_dt="bf16", logit_dt="bf16", tree=(4, 3, 2, 2, 1, 1),
                           mode="greedy", force_p=0.65, sigma=3.0),
    # Qwen3-8B-shaped stochastic chain: B=32, lookahead 5, L in [512,4096], V=151936, T=1.0
    "qwen3_8b_stochastic": dict(kind="verify", B=32, T=6, Hq=32, Hkv=8, D=128, L=(512, 4096), V=151936,
                                q_dt="bf16", kv_dt="bf16", logit_dt="bf16", tree="chain", mode="prob",
                                temperature=1.0, sigma=2.5, rho=0.8),
    # online-training loss: 64 traces x 32 nodes, depth 5 (4/3/2/1/1), V=128256
    "loss_batch": dict(kind="loss", N=64, T=32, V=128256, tree=(4, 3, 2, 1, 1), sigma=3.0,
                       accept_frac=0.45),
    # FP8 long context: B=128, 64 nodes depth 7 (4/3/2/2/1/1/1), 64/8 heads, e4m3 KV, L in [8192,32768]
    "fp8_long_context": dict(kind="verify", B=128, T=64, Hq=64, Hkv=8, D=128, L=(8192, 32768), V=151936,
                             q_dt="bf16", kv_dt="e4m3", logit_dt="bf16", tree=(4, 3, 2, 2, 1, 1, 1),
                             mode="greedy", force_p=0.7, sigma=3.0),
}


def make_workload(name: str, seed: int = 0, device=None, **overrides):
    """A named workload; device="cuda" draws a verify batch with make_verify_device (greedy / one-hot)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    kind = cfg.pop("kind")
    if kind == "loss":
        return make_loss(seed, name=name, **cfg)
    if device is not None:
        return make_verify_device(seed, name=name, device=device, **cfg)
    return make_verify(seed, name=name, **cfg)
