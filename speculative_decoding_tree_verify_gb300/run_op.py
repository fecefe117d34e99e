"""Run one library call repeatedly on a named synthetic workload (for profilers such as ncu).

python -m speculative_decoding_tree_verify_gb300.run_op --op OP --workload NAME [--reps N]
                                                        [--batch B] [--mode greedy|onehot|prob] [--device-recipe]
OP: attn, accept, loss, attn_bwd (forward once, then the backward), attn_paged (caches in 128-row pages),
compact (random accepted root paths), expand (the widest level of the workload's tree).
Inputs are generated once and stay on the device; the call is repeated --reps times.  --device-recipe draws
a greedy / one-hot verify batch on the GPU (the generator's device recipe), for full-size batches.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import sv
from . import workloads as W


def _dev(a):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.cuda()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["attn", "accept", "loss", "attn_bwd", "attn_paged", "compact", "expand"],
                    required=True)
    ap.add_argument("--workload", required=True)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--batch", type=int, default=None, help="override the batch size")
    ap.add_argument("--mode", default=None, help="override the acceptance mode")
    ap.add_argument("--temperature", type=float, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--device-recipe", action="store_true", help="draw the verify batch on the GPU")
    args = ap.parse_args()
    over = {}
    if args.batch is not None:
        over["N" if args.op == "loss" else "B"] = args.batch
    if args.mode is not None:
        over["mode"] = args.mode
    if args.temperature is not None:
        over["temperature"] = args.temperature
    if args.op in ("accept", "expand"):
        over["with_attn"] = False
    if args.device_recipe:
        over.pop("with_attn", None)
        over["device"] = "cuda"
    w = W.make_workload(args.workload, seed=args.seed, **over)
    i32 = dict(dtype=torch.int32, device="cuda")
    if args.op == "attn":
        q, k, v = _dev(w.q), _dev(w.k), _dev(w.v)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        n = sv.workspace_size(sv.OP_TREE_ATTN, w.B, w.T, w.Hq, w.Hkv, w.D, w.kv_cap, 0)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
        kl, par, ks, vs = _dev(w.kv_len), _dev(w.parent), _dev(w.k_scale), _dev(w.v_scale)
        for _ in range(args.reps):
            sv.tree_attn(q, k, v, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st, workspace=ws)
    elif args.op == "accept":
        B, T, V = w.B, w.T, w.V
        tgt = _dev(w.target_logits)
        dr = _dev(w.draft_logits) if w.temperature > 0 else None
        tok, par, u = _dev(w.tokens), _dev(w.parent), _dev(w.uniforms)
        outs = [torch.empty((B,), **i32), torch.empty((B, T), **i32), torch.empty((B, T), **i32),
                torch.empty((B,), **i32)]
        st = torch.empty((B,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_ACCEPT, B, T, V=V), 256), dtype=torch.uint8, device="cuda")
        for _ in range(args.reps):
            sv.accept(tgt, tok, par, *outs, draft_logits=dr, temperature=w.temperature, uniforms=u, status=st,
                      workspace=ws)
    elif args.op in ("attn_bwd", "attn_paged"):
        q, kl, par = _dev(w.q), _dev(w.kv_len), _dev(w.parent)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        if args.op == "attn_paged":
            kp, table = W.to_pages(args.seed, w.k, w.kv_len, w.T, 128)
            vp, _ = W.to_pages(args.seed, w.v, w.kv_len, w.T, 128)
            kpd, vpd, tbl, ks, vs = _dev(kp), _dev(vp), _dev(table), _dev(w.k_scale), _dev(w.v_scale)
            for _ in range(args.reps):
                sv.tree_attn_paged(q, kpd, vpd, tbl, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st)
        else:
            k, v = _dev(w.k), _dev(w.v)
            sv.tree_attn(q, k, v, kl, par, out, lse=lse, status=st)
            dout = torch.randn(q.shape, device="cuda").to(torch.bfloat16).view(torch.int16) \
                if w.q_dt == "bf16" else torch.randn(q.shape, device="cuda")
            dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
            dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
            dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
            ws = torch.empty(max(sv.workspace_size(sv.OP_TREE_ATTN_BWD, w.B, w.T, w.Hq), 256), dtype=torch.uint8,
                             device="cuda")
            for _ in range(args.reps):
                sv.tree_attn_bwd(q, k, v, kl, par, out, lse, dout, dq, dk, dv, status=st, workspace=ws)
    elif args.op == "compact":
        k, v = _dev(w.k), _dev(w.v)
        acc, path = W.random_root_paths(args.seed, w.parent)
        nl = torch.empty((w.B,), **i32)
        st = torch.empty((w.B,), **i32)
        al, pth, kl, par = _dev(acc), _dev(path), _dev(w.kv_len), _dev(w.parent)
        for _ in range(args.reps):
            sv.kv_compact(k, v, kl, par, al, pth, nl, status=st)
    elif args.op == "expand":
        tree = w.meta["tree"]
        levels = W.expansion_levels(w.T, tree) if tree not in ("chain", "star") else [(1, 1, 1)]
        nf, kk, nk = max(levels, key=lambda x: x[0])
        e = W.make_expand(args.seed, B=w.B, n_front=nf, V=w.V, k=kk, n_keep=nk, logit_dt="bf16")
        z, fs = _dev(e.logits).view(w.B, nf, w.V), _dev(e.front_score)
        tt = torch.empty((w.B, nf, kk), **i32)
        tl = torch.empty((w.B, nf, kk), dtype=torch.float32, device="cuda")
        cp, ct = torch.empty((w.B, max(nk, 1)), **i32), torch.empty((w.B, max(nk, 1)), **i32)
        cs = torch.empty((w.B, max(nk, 1)), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        for _ in range(args.reps):
            sv.tree_expand(z, fs, kk, nk, tt, tl, cp, ct, cs, status=st)
    else:
        z, tok, par, lab = _dev(w.logits), _dev(w.tokens), _dev(w.parent), _dev(w.labels)
        rl = torch.empty((w.N * w.T,), dtype=torch.float32, device="cuda")
        sums = torch.empty((3,), dtype=torch.float32, device="cuda")
        grad = torch.empty_like(z)
        st = torch.empty((w.N,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_LOSS, w.N, w.T, V=w.V), 256), dtype=torch.uint8, device="cuda")
        for _ in range(args.reps):
            sv.loss(z, tok, par, lab, rl, sums, grad=grad, status=st, workspace=ws)
    torch.cuda.synchronize()
    print(f"{args.op} x{args.reps} on {args.workload}: ok")


if __name__ == "__main__":
    main()
