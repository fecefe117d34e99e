"""CPU oracle for speculative tree verification (ctypes binding over oracle.c).

TEST INFRASTRUCTURE ONLY.  Imported by tests/, by ``__graft_entry__.smoke()`` (as the checker) and by
bench.py's CPU-baseline / reference leg.  The library under speculative_decoding_tree_verify_gb300 never
imports it, and it never imports the library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
BUILD = HERE / "_build"
LIB = BUILD / "liboracle.so"

DT = {"f32": 0, "bf16": 1, "e4m3": 2}


def build(force: bool = False) -> Path:
    """Compile oracle.c with gcc (OpenMP when available).  fp contraction is off: the acceptance
    contract is defined op by op in IEEE float32."""
    src = HERE / "oracle.c"
    if LIB.exists() and not force and LIB.stat().st_mtime >= max(src.stat().st_mtime,
                                                                   (HERE / "oracle.h").stat().st_mtime):
        return LIB
    BUILD.mkdir(exist_ok=True)
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            str(src), "-o", str(LIB) + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(str(LIB) + ".tmp", LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(LIB)
    return _lib


def use(path):
    """Point the binding at another build of oracle.c (the mutation tests build planted-mistake copies)."""
    global _lib
    prev = _lib
    _lib = load(path)
    return prev


def restore(prev):
    global _lib
    _lib = prev


def load(path):
    L = C.CDLL(str(path))
    P = C.c_void_p
    i = C.c_int
    L.or_tree_check.argtypes = [i, P]
    L.or_tree_depth.argtypes = [i, P, P]
    L.or_tree_attn.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, P, P, C.c_double, P, i, P, P, P]
    L.or_fx_weight.argtypes = [C.c_float, C.c_float]
    L.or_fx_weight.restype = C.c_uint32
    L.or_fx_exp2.argtypes = [C.c_float]
    L.or_fx_exp2.restype = C.c_float
    L.or_fx_exp2_batch.argtypes = [P, P, C.c_long]
    L.or_fx_weight_batch.argtypes = [P, C.c_float, P, C.c_long]
    L.or_accept.argtypes = [i, i, i, i, P, P, P, P, C.c_float, P, P, P, P, P, P, P]
    L.or_loss_f64.argtypes = [i, i, i, P] + [P] * 9
    L.or_loss.argtypes = [i, i, i, P] + [P] * 9
    L.or_kv_compact.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P]
    L.or_tree_expand.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P]
    L.or_tree_attn_bwd.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, C.c_double, P, P, P, P, P]
    L.or_tree_attn_e2m1.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, C.c_double, P, i, P, P, P]
    L.or_set_num_threads.argtypes = [i]
    L.or_set_num_threads.restype = None
    return L


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def num_threads() -> int:
    return int(lib().or_num_threads())


def set_num_threads(n: int) -> None:
    """Thread count of later oracle calls (OpenMP)."""
    lib().or_set_num_threads(int(n))


# ------------------------------------------------------------------------------------------------ tree
def tree_check(parent) -> int:
    parent = np.ascontiguousarray(parent, np.int32)
    return int(lib().or_tree_check(len(parent), _p(parent)))


def tree_depth(parent):
    parent = np.ascontiguousarray(parent, np.int32)
    d = np.zeros(len(parent), np.int32)
    st = lib().or_tree_depth(len(parent), _p(parent), _p(d))
    return st, d


# ------------------------------------------------------------------------------------------------ attention
def tree_attn(q, k, v, kv_len, parent, *, Hq, Hkv, q_dt, kv_dt, k_scale=None, v_scale=None,
              sm_scale=0.0, rows=None):
    """float64 tree-masked attention.  Returns (out [B,T,Hq,D] f64, lse [B,T,Hq] f64, status [B], rc).
    rows: optional int array [n,3] of (b, i, h) to compute; other entries stay NaN."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    B, T = parent.shape
    D = q.shape[-1]
    kv_cap = k.shape[2]
    kv_len = np.ascontiguousarray(kv_len, np.int32)
    parent = np.ascontiguousarray(parent, np.int32)
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, np.float32)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, np.float32)
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    status = np.zeros(B, np.int32)
    r = None if rows is None else np.unique(np.asarray(rows, np.int32).reshape(-1, 3), axis=0)
    r = None if r is None else np.ascontiguousarray(r, np.int32)
    rc = lib().or_tree_attn(B, T, Hq, Hkv, D, kv_cap, DT[q_dt], DT[kv_dt], _p(q), _p(k), _p(v), _p(ks),
                            _p(vs), _p(kv_len), _p(parent), float(sm_scale), _p(r),
                            0 if r is None else len(r), _p(out), _p(lse), _p(status))
    return out, lse, status, rc


def tree_attn_w(w, rows=None, sm_scale=0.0):
    """tree_attn on a workloads.Verify batch."""
    return tree_attn(w.q, w.k, w.v, w.kv_len, w.parent, Hq=w.Hq, Hkv=w.Hkv, q_dt=w.q_dt, kv_dt=w.kv_dt,
                     k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=sm_scale, rows=rows)


def tree_attn_e2m1(q, k_codes, v_codes, k_block, v_block, k_scale, v_scale, kv_len, parent, *, Hq, q_dt,
                   sm_scale=0.0, rows=None):
    """Tree attention over FP4 (E2M1) caches with E4M3 block scales (16 elements) and fp32 head scales.
    k_codes / v_codes [B, Hkv, kv_cap, D/2] uint8 (even element in the low nibble).  Returns (out, lse,
    status, rc) like tree_attn; rows: optional (b, i, h) triples to compute, other entries stay NaN."""
    q = np.ascontiguousarray(q)
    B, T = parent.shape
    D = q.shape[-1]
    Hkv, kv_cap = k_codes.shape[1], k_codes.shape[2]
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    status = np.zeros(B, np.int32)
    args = [np.ascontiguousarray(x, np.uint8) for x in (k_codes, v_codes, k_block, v_block)]
    ks = np.ascontiguousarray(k_scale, np.float32)
    vs = np.ascontiguousarray(v_scale, np.float32)
    r = None if rows is None else np.ascontiguousarray(np.unique(np.asarray(rows, np.int32).reshape(-1, 3), axis=0))
    rc = lib().or_tree_attn_e2m1(B, T, Hq, Hkv, D, kv_cap, DT[q_dt], _p(q), *[_p(x) for x in args], _p(ks), _p(vs),
                                 _p(np.ascontiguousarray(kv_len, np.int32)), _p(np.ascontiguousarray(parent, np.int32)),
                                 float(sm_scale), _p(r), 0 if r is None else len(r), _p(out), _p(lse), _p(status))
    return out, lse, status, rc


def tree_attn_paged(q, k_pool, v_pool, page_table, kv_len, parent, *, Hq, Hkv, q_dt, kv_dt, k_scale=None,
                    v_scale=None, sm_scale=0.0):
    """Tree attention over paged caches: each request's logical cache is read through its page table (pool
    page page_table[b, j // P] holds positions j), then the plain definition above runs on it.  A request
    whose kv_len + T exceeds the table's capacity or that names a page outside the pool gets status 1."""
    num_pages, _, P, D = k_pool.shape
    B, max_pages = page_table.shape
    T = parent.shape[1]
    cap = max_pages * P
    junk = np.zeros((), dtype=k_pool.dtype)
    k = np.full((B, Hkv, cap, D), junk, dtype=k_pool.dtype)
    v = np.full((B, Hkv, cap, D), junk, dtype=v_pool.dtype)
    bad = np.zeros(B, bool)
    for b in range(B):
        n = int(kv_len[b]) + T
        if n > cap or int(kv_len[b]) < 0:
            bad[b] = True
            continue
        for pg in range(-(-n // P)):
            src = int(page_table[b, pg])
            if not 0 <= src < num_pages:
                bad[b] = True
                break
            k[b, :, pg * P:(pg + 1) * P] = k_pool[src]
            v[b, :, pg * P:(pg + 1) * P] = v_pool[src]
    out, lse, status, rc = tree_attn(q, k, v, kv_len, parent, Hq=Hq, Hkv=Hkv, q_dt=q_dt, kv_dt=kv_dt,
                                     k_scale=k_scale, v_scale=v_scale, sm_scale=sm_scale)
    status = np.where(bad & (status == 0), 1, status).astype(np.int32)
    out[bad] = 0.0
    lse[bad] = 0.0
    return out, lse, status, rc


def tree_attn_bwd(q, k, v, kv_len, parent, dout, *, Hq, Hkv, q_dt, kv_dt, sm_scale=0.0):
    """float64 backward of the tree-masked attention for the upstream gradient dout (q's layout and dtype).
    Returns (dq [B,T,Hq,D], dk [B,Hkv,kv_cap,D], dv [B,Hkv,kv_cap,D], status [B], rc)."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    dout = np.ascontiguousarray(dout)
    B, T = parent.shape
    D = q.shape[-1]
    kv_cap = k.shape[2]
    dq = np.zeros((B, T, Hq, D))
    dk = np.zeros((B, Hkv, kv_cap, D))
    dv = np.zeros((B, Hkv, kv_cap, D))
    status = np.zeros(B, np.int32)
    rc = lib().or_tree_attn_bwd(B, T, Hq, Hkv, D, kv_cap, DT[q_dt], DT[kv_dt], _p(q), _p(k), _p(v),
                                _p(np.ascontiguousarray(kv_len, np.int32)), _p(np.ascontiguousarray(parent, np.int32)),
                                float(sm_scale), _p(dout), _p(dq), _p(dk), _p(dv), _p(status))
    return dq, dk, dv, status, rc


# ------------------------------------------------------------------------------------------------ acceptance
def fx_exp2(f):
    f = np.ascontiguousarray(f, np.float32)
    out = np.empty_like(f)
    lib().or_fx_exp2_batch(_p(f), _p(out), f.size)
    return out


def fx_weight(y, m: float):
    y = np.ascontiguousarray(y, np.float32)
    out = np.empty(y.shape, np.uint32)
    lib().or_fx_weight_batch(_p(y), C.c_float(m), _p(out), y.size)
    return out


def accept(target, tokens, parent, *, V, logit_dt, temperature=0.0, draft=None, uniforms=None,
           want_argmax=True):
    target = np.ascontiguousarray(target)
    draft = None if draft is None else np.ascontiguousarray(draft)
    tokens = np.ascontiguousarray(tokens, np.int32)
    parent = np.ascontiguousarray(parent, np.int32)
    B, T = parent.shape
    u = None if uniforms is None else np.ascontiguousarray(uniforms, np.uint32)
    res = dict(accept_len=np.zeros(B, np.int32), path=np.zeros((B, T), np.int32),
               out_tokens=np.zeros((B, T), np.int32), bonus=np.zeros(B, np.int32),
               argmax=np.zeros((B, T), np.int32) if want_argmax else None, status=np.zeros(B, np.int32))
    rc = lib().or_accept(B, T, V, DT[logit_dt], _p(target), _p(draft), _p(tokens), _p(parent),
                         C.c_float(temperature), _p(u), _p(res["accept_len"]), _p(res["path"]),
                         _p(res["out_tokens"]), _p(res["bonus"]), _p(res["argmax"]), _p(res["status"]))
    res["rc"] = rc
    return res


def accept_w(w, temperature=None, draft="auto"):
    """accept on a workloads.Verify batch."""
    t = w.temperature if temperature is None else temperature
    d = w.draft_logits if draft == "auto" else draft
    return accept(w.target_logits, w.tokens, w.parent, V=w.V, logit_dt=w.logit_dt, temperature=t,
                  draft=d if t > 0 else None, uniforms=w.uniforms)


# ------------------------------------------------------------------------------------------------ loss
def _loss(fn, N, T, V, logits, tokens, parent, labels, want_grad):
    tokens = np.ascontiguousarray(tokens, np.int32)
    parent = np.ascontiguousarray(parent, np.int32)
    labels = np.ascontiguousarray(labels, np.int32)
    res = dict(row_loss=np.zeros(N * T), row_acc=np.zeros(N * T), row_rej=np.zeros(N * T), sums=np.zeros(3),
               grad=np.zeros((N * T, V)) if want_grad else None, status=np.zeros(N, np.int32))
    res["rc"] = fn(N, T, V, _p(logits), _p(tokens), _p(parent), _p(labels), _p(res["row_loss"]),
                   _p(res["row_acc"]), _p(res["row_rej"]), _p(res["sums"]), _p(res["grad"]),
                   _p(res["status"]))
    res["loss"] = (res["sums"][0] + res["sums"][1]) / res["sums"][2] if res["sums"][2] else 0.0
    return res


def loss(logits_bf16, tokens, parent, labels, *, V, want_grad=True):
    N, T = parent.shape
    lg = np.ascontiguousarray(logits_bf16, np.uint16)
    return _loss(lib().or_loss, N, T, V, lg, tokens, parent, labels, want_grad)


def loss_f64(logits, tokens, parent, labels, *, V, want_grad=True):
    N, T = parent.shape
    lg = np.ascontiguousarray(logits, np.float64)
    return _loss(lib().or_loss_f64, N, T, V, lg, tokens, parent, labels, want_grad)


def loss_w(lb, want_grad=True):
    return loss(lb.logits, lb.tokens, lb.parent, lb.labels, V=lb.V, want_grad=want_grad)


# ------------------------------------------------------------------------------------------------ KV compaction
def kv_compact(k, v, kv_len, parent, accept_len, path, *, kv_dt):
    """Compaction of the accepted path's K/V.  Returns (k', v', new_kv_len, status, rc) on copies."""
    k = np.array(k, copy=True, order="C")
    v = np.array(v, copy=True, order="C")
    B, Hkv, kv_cap, D = k.shape
    T = parent.shape[1]
    parent = np.ascontiguousarray(parent, np.int32)
    kv_len = np.ascontiguousarray(kv_len, np.int32)
    accept_len = np.ascontiguousarray(accept_len, np.int32)
    path = np.ascontiguousarray(path, np.int32)
    new_len = np.zeros(B, np.int32)
    status = np.zeros(B, np.int32)
    rc = lib().or_kv_compact(B, T, Hkv, D, kv_cap, DT[kv_dt], _p(k), _p(v), _p(kv_len), _p(parent),
                             _p(accept_len), _p(path), _p(new_len), _p(status))
    return k, v, new_len, status, rc


# ------------------------------------------------------------------------------------------------ tree expansion
def tree_expand(logits, front_score, *, V, k, n_keep, logit_dt):
    """One level of draft tree expansion.  logits [B, n_front, V]; front_score [B, n_front] float32."""
    logits = np.ascontiguousarray(logits)
    fs = np.ascontiguousarray(front_score, np.float32)
    B, n_front = fs.shape
    res = dict(topk_token=np.zeros((B, n_front, k), np.int32), topk_logprob=np.zeros((B, n_front, k)),
               child_parent=np.zeros((B, n_keep), np.int32), child_token=np.zeros((B, n_keep), np.int32),
               child_score=np.zeros((B, n_keep)), status=np.zeros(B, np.int32))
    res["rc"] = lib().or_tree_expand(B, n_front, V, k, n_keep, DT[logit_dt], _p(logits), _p(fs),
                                     _p(res["topk_token"]), _p(res["topk_logprob"]), _p(res["child_parent"]),
                                     _p(res["child_token"]), _p(res["child_score"]), _p(res["status"]))
    return res
