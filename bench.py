"""Benchmark: verified tree nodes per second of one verification step (tree attention + acceptance).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl sv|reference] [--workload NAME]

A step is one pass of the verify path over one batch: sv_tree_attn over every node of every request,
then sv_accept (walk + bonus).  The default workload is the Llama3-8B-shaped EAGLE tree batch
(B=8, 60-node trees, 32/8 heads, D=128, bf16, KV prefixes of 2048..8192, vocabulary 128256, greedy).
value = B*T*world / device time per step (CUDA events on the launching stream, L2 flushed between steps
by a 256 MB write outside the timed events; each call replayed from a CUDA graph captured after the
warm-up).  e2e = the same metric through the C ABI with the step's
inputs copied from pinned host memory and its outputs copied back inside the timed region.  Under
torchrun every rank verifies its own batch (weak scaling, no collective on the data path).
--impl reference times the CPU oracle on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
METRIC = "verified tree nodes/s on 1 GB300 (attn+accept); % of HBM roofline achieved"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["sv", "reference"], default="sv")
    ap.add_argument("--workload", default="llama3_8b_tree")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--ops", nargs="*", default=None,
                    help="instead of the step: time every library call on the named workloads (all if none given), "
                         "one JSON line per call")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------ ranks
def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the slowest rank's step time); x itself on one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def nodes_per_second(B: int, T: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank verifies its own batch of B requests x T nodes per step (weak scaling)."""
    return B * T * world / (ms * 1e-3)


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch from its own seed."""
    return seed + rank


# ------------------------------------------------------------------------------------------ algorithmic bytes
ES = {"f32": 4, "bf16": 2, "e4m3": 1}


def attn_bytes(w):
    """Bytes the method must move: K and V of every allowed position (prefix + tree block) once per kv head,
    Q in, O out, lse out, plus the small int arrays."""
    kv = int(np.sum(w.kv_len.astype(np.int64) + w.T)) * w.Hkv * w.D * 2 * ES[w.kv_dt]
    qo = 2 * w.B * w.T * w.Hq * w.D * ES[w.q_dt]
    return kv + qo + w.B * w.T * w.Hq * 4 + w.B * (w.T + 1) * 4


def accept_bytes(w):
    rows = w.B * w.T * (2 if (w.temperature > 0 and w.draft_logits is not None) else 1)
    return rows * w.V * ES[w.logit_dt] + w.B * w.T * 4 * 6


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------ CPU oracle timing
def cpu_oracle_sample(w, budget_s: float):
    """Time the oracle (as it stands) on whole requests of the workload until the budget is spent.
    Returns (nodes per second, threads, description)."""
    import oracle
    from speculative_decoding_tree_verify_gb300 import workloads as W
    done, t_total = 0, 0.0
    for b in range(w.B):
        sub = W.Verify(B=1, T=w.T, Hq=w.Hq, Hkv=w.Hkv, D=w.D, kv_cap=w.kv_cap, V=w.V, q_dt=w.q_dt, kv_dt=w.kv_dt,
                       logit_dt=w.logit_dt, q=w.q[b:b + 1], k=w.k[b:b + 1], v=w.v[b:b + 1], k_scale=w.k_scale,
                       v_scale=w.v_scale, kv_len=w.kv_len[b:b + 1], parent=w.parent[b:b + 1],
                       tokens=w.tokens[b:b + 1], target_logits=w.target_logits[b:b + 1],
                       draft_logits=None if w.draft_logits is None else w.draft_logits[b:b + 1],
                       uniforms=None if w.uniforms is None else w.uniforms[b:b + 1], temperature=w.temperature)
        t0 = time.perf_counter()
        oracle.tree_attn_w(sub)
        oracle.accept_w(sub)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    return done * w.T / t_total, oracle.num_threads(), f"{done} of {w.B} requests (all {w.T} nodes, all heads)"


# ------------------------------------------------------------------------------------------ profiles
def traffic_from_profile(kernel_src: Path, workload: str):
    """DRAM traffic per launch from a committed ncu summary, valid only while the kernel source is unchanged."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text()).get(workload)
    if not d:
        return None
    h = hashlib.sha256(kernel_src.read_bytes()).hexdigest()[:16]
    return d["traffic_bytes_per_launch"] if d.get("source_sha") == h else None


# ------------------------------------------------------------------------------------------ per-call timings
def run_ops(args):
    """One JSON line per (workload, call): median of 10 CUDA-graph replays, each after a 256 MB L2 flush,
    with the call's algorithmic bytes and the fraction of the HBM peak they represent."""
    import torch

    from speculative_decoding_tree_verify_gb300 import sv
    from speculative_decoding_tree_verify_gb300 import workloads as W

    peak, peak_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(args.seed)

    def dev(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        elif a.dtype == np.uint32:
            a = a.view(np.int32)
        return torch.from_numpy(a).cuda()

    def timed(fn, reps=10):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            fn()
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return float(np.median(ts))

    def report(name, op, us, nbytes, note=""):
        gbs = nbytes / (us * 1e-6) / 1e9
        print(json.dumps({"workload": name, "op": op, "us": round(us, 1), "alg_MB": round(nbytes / 1e6, 3),
                          "GB_s": round(gbs, 1), "frac": round(gbs / peak, 3), "peak_kind": peak_kind,
                          "note": note}), flush=True)

    i32 = dict(dtype=torch.int32, device="cuda")

    def attn_case(name, w, device_kv=False):
        q = dev(w.q)
        if device_kv:   # timing only: seeded random cache codes of the right dtype, drawn on the device
            shape = (w.B, w.Hkv, w.kv_cap, w.D)
            if w.kv_dt == "e4m3":
                k = torch.randint(0, 0x7E, shape, dtype=torch.uint8, device="cuda", generator=gen)
                v = torch.randint(0, 0x7E, shape, dtype=torch.uint8, device="cuda", generator=gen)
            else:
                k = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16).view(torch.int16)
                v = torch.randn(shape, device="cuda", generator=gen).to(torch.bfloat16).view(torch.int16)
            ks = torch.full((w.Hkv,), 0.01, device="cuda")
            vs = ks.clone()
        else:
            k, v, ks, vs = dev(w.k), dev(w.v), dev(w.k_scale), dev(w.v_scale)
        if q is None:
            q = torch.randn((w.B, w.T, w.Hq, w.D), device="cuda", generator=gen).to(torch.bfloat16).view(torch.int16)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        n = sv.workspace_size(sv.OP_TREE_ATTN, w.B, w.T, w.Hq, w.Hkv, w.D, w.kv_cap, 0)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
        kl, par = dev(w.kv_len), dev(w.parent)
        fn = lambda: sv.tree_attn(q, k, v, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st, workspace=ws)
        us = timed(fn, reps=5 if w.kv_dt == "e4m3" else 10)
        tc = w.q_dt == "bf16" and w.kv_dt in ("bf16", "e4m3") and w.D == 128
        report(name, "tree_attn", us, attn_bytes(w), "tensor cores" if tc else "CUDA cores")

    def accept_case(name, w, temperature, draft):
        B, T, V = w.B, w.T, w.V
        tgt = dev(w.target_logits).view(B, T, V)
        dr = dev(draft).view(B, T, V) if draft is not None else None
        tok, par, u = dev(w.tokens), dev(w.parent), dev(w.uniforms)
        outs = [torch.empty((B,), **i32), torch.empty((B, T), **i32), torch.empty((B, T), **i32),
                torch.empty((B,), **i32)]
        st = torch.empty((B,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_ACCEPT, B, T, V=V), 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sv.accept(tgt, tok, par, *outs, draft_logits=dr, temperature=temperature, uniforms=u, status=st,
                               workspace=ws)
        us = timed(fn)
        rows = B * T * (2 if dr is not None else 1)
        mode = "greedy" if temperature == 0 else ("prob" if dr is not None else "onehot")
        report(name, f"accept_{mode}", us, rows * V * ES[w.logit_dt] + B * T * 24)

    def loss_case(name, lb):
        N, T, V = lb.N, lb.T, lb.V
        z, tok, par, lab = dev(lb.logits), dev(lb.tokens), dev(lb.parent), dev(lb.labels)
        rl = torch.empty((N * T,), dtype=torch.float32, device="cuda")
        sums = torch.empty((3,), dtype=torch.float32, device="cuda")
        grad = torch.empty_like(z)
        st = torch.empty((N,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_LOSS, N, T, V=V), 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sv.loss(z, tok, par, lab, rl, sums, grad=grad, status=st, workspace=ws)
        report(name, "loss+grad", timed(fn), 2 * N * T * V * 2 + N * T * 16)

    def bwd_case(name, w):
        """Tree-attention backward (CUDA cores): FLOPs = 10 * D per (query row, allowed position) -- the five
        products s, dp, dq, dk, dv -- against the FP32 CUDA-core peak (152 SMs x 128 FMA lanes x 2 x 2.07 GHz)."""
        q, k, v = dev(w.q), dev(w.k), dev(w.v)
        kl, par = dev(w.kv_len), dev(w.parent)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        sv.tree_attn(q, k, v, kl, par, out, lse=lse)
        dout = torch.randn(q.shape, device="cuda", generator=gen).to(torch.bfloat16).view(torch.int16)
        dq = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        dk = torch.empty(k.shape, dtype=torch.float32, device="cuda")
        dv = torch.empty(v.shape, dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_TREE_ATTN_BWD, w.B, w.T, w.Hq), 256), dtype=torch.uint8,
                         device="cuda")
        fn = lambda: sv.tree_attn_bwd(q, k, v, kl, par, out, lse, dout, dq, dk, dv, status=st, workspace=ws)
        us = timed(fn, reps=5)
        def n_ancestors(par, i):          # tree slots node i attends to: itself and its ancestors
            n = 0
            while i >= 0:
                n, i = n + 1, int(par[i])
            return n

        depth = np.array([[n_ancestors(w.parent[b], i) for i in range(w.T)] for b in range(w.B)])
        pairs = int(sum(int(w.kv_len[b]) * w.T + int(depth[b].sum()) for b in range(w.B))) * w.Hq
        flops = 10.0 * w.D * pairs
        peak_alu = 152 * 128 * 2 * 2.07e9 / 1e12   # TFLOP/s
        tf = flops / (us * 1e-6) / 1e12
        print(json.dumps({"workload": name, "op": "tree_attn_bwd", "us": round(us, 1), "TFLOP_s": round(tf, 2),
                          "frac": round(tf / peak_alu, 3), "bound": "alu", "peak_TFLOP_s": round(peak_alu, 1),
                          "note": "CUDA cores, fp32; FLOPs = 10*D per (query row, allowed position)"}), flush=True)

    def paged_case(name, w, page_size=128):
        """Tree attention over the same caches scattered into a page pool (CUDA-core kernel); bytes as for
        the contiguous call."""
        kp, table = W.to_pages(args.seed, w.k, w.kv_len, w.T, page_size)
        vp, _ = W.to_pages(args.seed, w.v, w.kv_len, w.T, page_size)
        q, kpd, vpd, tbl = dev(w.q), dev(kp), dev(vp), dev(table)
        kl, par, ks, vs = dev(w.kv_len), dev(w.parent), dev(w.k_scale), dev(w.v_scale)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        fn = lambda: sv.tree_attn_paged(q, kpd, vpd, tbl, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st)
        report(name, "tree_attn_paged", timed(fn, reps=5), attn_bytes(w), f"CUDA cores, {page_size}-row pages")

    def compact_case(name, B, T, Hkv, D, kv_cap, kv_dt, kv_len, parent, seed):
        """KV compaction of random accepted root paths; bytes = the moved rows read once and written once."""
        shape = (B, Hkv, kv_cap, D)
        dt = {"e4m3": torch.uint8, "bf16": torch.int16, "f32": torch.float32}[kv_dt]
        k = torch.zeros(shape, dtype=dt, device="cuda")
        v = torch.zeros_like(k)
        acc, path = W.random_root_paths(seed, parent)
        kl, par, al, pth = dev(kv_len), dev(parent), dev(acc), dev(path)
        nl = torch.empty((B,), **i32)
        st = torch.empty((B,), **i32)
        fn = lambda: sv.kv_compact(k, v, kl, par, al, pth, nl, status=st)
        moved = sum(int(np.sum(path[b, :acc[b]] != np.arange(1, acc[b] + 1))) for b in range(B))
        report(name, "kv_compact", timed(fn), moved * Hkv * D * ES[kv_dt] * 2 * 2,
               f"mean accept_len {float(np.mean(acc)):.2f}, launch-bound")

    def expand_case(name, B, V, levels, sigma, seed):
        """Every level of the tree, one call each; bytes = the frontier logit rows read once."""
        tot_us, tot_b = 0.0, 0
        for d, (nf, kk, nk) in enumerate(levels):
            e = W.make_expand(seed + d, B=B, n_front=nf, V=V, k=kk, n_keep=nk, logit_dt="bf16", sigma=sigma)
            z, fs = dev(e.logits).view(B, nf, V), dev(e.front_score)
            tt = torch.empty((B, nf, kk), **i32)
            tl = torch.empty((B, nf, kk), dtype=torch.float32, device="cuda")
            cp, ct = torch.empty((B, max(nk, 1)), **i32), torch.empty((B, max(nk, 1)), **i32)
            cs = torch.empty((B, max(nk, 1)), dtype=torch.float32, device="cuda")
            st = torch.empty((B,), **i32)
            fn = lambda: sv.tree_expand(z, fs, kk, nk, tt, tl, cp, ct, cs, status=st)
            us = timed(fn)
            nb = B * nf * V * 2
            tot_us += us
            tot_b += nb
            report(name, f"tree_expand_level{d + 1}", us, nb, f"{nf} x top-{kk} -> {nk}")
        report(name, "tree_expand_all_levels", tot_us, tot_b, f"{len(levels)} calls")

    which = args.ops or ["tiny_chain", "llama3_8b_tree", "qwen3_8b_stochastic", "loss_batch", "fp8_long_context"]
    for name in which:
        if name == "loss_batch":
            loss_case(name, W.make_workload(name, seed=args.seed))
            continue
        if name == "fp8_long_context":
            w = W.make_workload(name, seed=args.seed, with_attn=False)
            accept_case(name, w, 0.0, None)
            w2 = W.make_workload(name, seed=args.seed, with_attn=False, mode="onehot", temperature=0.7)
            accept_case(name, w2, 0.7, None)
            del w2
            attn_case(name, w, device_kv=True)
            compact_case(name, w.B, w.T, w.Hkv, w.D, w.kv_cap, w.kv_dt, w.kv_len, w.parent, args.seed)
            expand_case(name, w.B, w.V, W.expansion_levels(64, (4, 3, 2, 2, 1, 1, 1)), 3.0, 500 + args.seed)
            continue
        w = W.make_workload(name, seed=args.seed)
        attn_case(name, w)
        accept_case(name, w, w.temperature, w.draft_logits if w.temperature > 0 else None)
        if name in ("llama3_8b_tree", "qwen3_8b_stochastic"):
            bwd_case(name, w)
            paged_case(name, w)
        compact_case(name, w.B, w.T, w.Hkv, w.D, w.kv_cap, w.kv_dt, w.kv_len, w.parent, args.seed)
        if name == "llama3_8b_tree":
            expand_case(name, w.B, w.V, W.expansion_levels(60, (4, 3, 2, 2, 1, 1)), 3.0, 200 + args.seed)
        elif name == "qwen3_8b_stochastic":
            expand_case(name, w.B, w.V, [(1, 1, 1)] * 5, 2.5, 300 + args.seed)


# ------------------------------------------------------------------------------------------ main arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    from speculative_decoding_tree_verify_gb300 import workloads as W
    w = W.make_workload(args.workload, seed=args.seed)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        v, cores, desc = cpu_oracle_sample(w, per_step)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w.B * w.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "V": w.V, "kv_dt": w.kv_dt, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_sv(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from speculative_decoding_tree_verify_gb300 import sv
    from speculative_decoding_tree_verify_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = W.make_workload(args.workload, seed=rank_seed(args.seed, rank))

    def to_dev(a, pin=False):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        elif a.dtype == np.uint32:
            a = a.view(np.int32)
        t = torch.from_numpy(a)
        return t.pin_memory() if pin else t.to(dev)

    names = ("q", "k", "v", "k_scale", "v_scale", "kv_len", "parent", "tokens", "target_logits", "draft_logits",
             "uniforms")
    host = {k: to_dev(getattr(w, k), pin=True) for k in names if getattr(w, k) is not None}
    d = {k: t.to(dev) for k, t in host.items()}
    for k in names:
        d.setdefault(k, None)
    B, T, V = w.B, w.T, w.V
    i32 = dict(dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, T, w.Hq), dtype=torch.float32, device=dev)
    st_a = torch.empty((B,), **i32)
    acc = dict(accept_len=torch.empty((B,), **i32), path=torch.empty((B, T), **i32),
               out_tokens=torch.empty((B, T), **i32), bonus=torch.empty((B,), **i32),
               status=torch.empty((B,), **i32))
    ws_attn_n = sv.workspace_size(sv.OP_TREE_ATTN, B, T, w.Hq, w.Hkv, w.D, w.kv_cap, 0)
    ws_attn = torch.empty(max(ws_attn_n, 256), dtype=torch.uint8, device=dev)
    ws_acc = torch.empty(max(sv.workspace_size(sv.OP_ACCEPT, B, T, V=V), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    logits = d["target_logits"]

    def attn_call():
        sv.tree_attn(d["q"], d["k"], d["v"], d["kv_len"], d["parent"], out, k_scale=d.get("k_scale"),
                     v_scale=d.get("v_scale"), lse=lse, status=st_a, workspace=ws_attn)

    def accept_call():
        sv.accept(logits, d["tokens"], d["parent"], acc["accept_len"], acc["path"], acc["out_tokens"],
                  acc["bonus"], draft_logits=d["draft_logits"], temperature=w.temperature, uniforms=d["uniforms"],
                  status=acc["status"], workspace=ws_acc)

    def step():
        attn_call()
        ev_mid = torch.cuda.Event(enable_timing=True)
        ev_mid.record(stream)
        accept_call()
        return ev_mid

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert (st_a == 0).all() and (acc["status"] == 0).all(), "verify step reported a per-request error"

    # The timed steps replay the two calls as CUDA graphs captured after the warm-up (one graph per call, so
    # an event still separates attention from acceptance): the device runs the same kernels, without the
    # host-side launch work of each call in front of them.
    g_attn, g_acc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_attn, stream=side):
            attn_call()
        with torch.cuda.graph(g_acc, stream=side):
            accept_call()
    stream.wait_stream(side)
    torch.cuda.synchronize()

    def graph_step():
        g_attn.replay()
        ev_mid = torch.cuda.Event(enable_timing=True)
        ev_mid.record(stream)
        g_acc.replay()
        return ev_mid

    for _ in range(2):
        flush.zero_()
        graph_step()
    torch.cuda.synchronize()
    assert (st_a == 0).all() and (acc["status"] == 0).all(), "graph-replayed step reported a per-request error"

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = []
    with ClockSampler(local_rank) as clk:
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e1 = graph_step()
            e2.record(stream)
            evs.append((e0, e1, e2))
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_attn = sum(e0.elapsed_time(e1) for e0, e1, _ in evs) / args.steps
    t_acc = sum(e1.elapsed_time(e2) for _, e1, e2 in evs) / args.steps
    ms = max_over_ranks(t_attn + t_acc, world, dev)
    value = nodes_per_second(B, T, world, ms)

    # end to end through the C ABI: inputs from pinned host memory, outputs back, inside the timed region
    e2e = None
    if not args.no_e2e:
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        res_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in acc.items() if k != "status"}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size() + sum(t.numel() * t.element_size() for t in res_h.values())

        def e2e_step():
            for k, t in host.items():
                d[k].copy_(t, non_blocking=True)
            step()
            out_h.copy_(out, non_blocking=True)
            for k, t in res_h.items():
                t.copy_(acc[k], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, args.steps // 2)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        t1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(t0.elapsed_time(t1) / n_e2e, world, dev)
        e2e = {"value": nodes_per_second(B, T, world, ms_e2e), "unit": "nodes/s", "h2d_bytes_per_step": int(h2d) * world,
               "d2h_bytes_per_step": int(d2h) * world, "ms_per_step": ms_e2e}

    if rank != 0:
        return
    peak, peak_kind = peaks()
    ab, cb = attn_bytes(w), accept_bytes(w)
    # the dominant kernel is the one with the larger share of the step
    tc = w.q_dt == "bf16" and w.kv_dt == "bf16" and w.D == 128
    if t_attn >= t_acc:
        dom, byt, t_dom = "tree_attn", ab, t_attn
        src = ROOT / "speculative_decoding_tree_verify_gb300/csrc" / ("attn_tc.cu" if tc else "attn_simt.cu")
    else:
        dom, byt, t_dom, src = "accept", cb, t_acc, ROOT / "speculative_decoding_tree_verify_gb300/csrc/accept.cu"
    achieved = byt / (t_dom * 1e-3) / 1e9
    label = {"tree_attn": "sv_tree_attn (attn_tc_kernel + attn_merge_kernel)" if tc else "sv_tree_attn (attn_simt_kernel)",
             "accept": "sv_accept (accept_rows_kernel + accept_walk_kernel)"}[dom]
    roofline = {"bound": "hbm", "kernel": label, "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": achieved / peak, "algorithmic_bytes_per_launch": byt,
                "traffic": traffic_from_profile(src, args.workload),
                "step_frac": (ab + cb) / (ms * 1e-3) / 1e9 / peak}
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc = cpu_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": v, "unit": "nodes/s", "cores": cores, "kind": "oracle", "sample": desc}
    launches_per_step = (2 if tc else 1) + 2     # attention [+ merge], accept rows + walk
    line = {"metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.q_dt, "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "T": T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "V": V,
                       "kv_dt": w.kv_dt, "logit_dt": w.logit_dt, "mode": w.meta["mode"],
                       "mean_kv_len": float(np.mean(w.kv_len)), "l2": "flushed by a 256 MB write between steps",
                       "launch": "each call replayed as a CUDA graph captured after the warm-up",
                       "parallelism": f"replicas{world}" if world > 1 else "single"},
            "components": {"attn_ms": t_attn, "accept_ms": t_acc, "attn_bytes": ab, "accept_bytes": cb},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clk.summary(),
            "mean_accept_len": float(acc["accept_len"].float().mean().item())}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.ops is not None:
        if rank == 0:
            run_ops(args)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_sv(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.path.insert(0, str(ROOT))
    main()
