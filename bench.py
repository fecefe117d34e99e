"""Benchmark: verified tree nodes per second of one verification step (tree attention + acceptance).

python bench.py [--steps K] [--warmup W] [--impl sv|reference] [--workload NAME] [--ops [NAME ...]]

A step is one pass of the verify path over one batch: sv_tree_attn over every node of every request, then
sv_accept (walk + bonus) in each acceptance mode the workload runs.  The default workload is the large-context
FP8 batch (B=128, 64-node trees of depth 7, 64/8 heads, D=128, e4m3 KV with per-head scales, prefixes of
8192..32768, vocabulary 151936, greedy AND temperature-0.7 one-hot rejection sampling, both on every step).
The other named workloads: tiny_chain, llama3_8b_tree, qwen3_8b_stochastic (verify steps) and loss_batch
(one sv_loss call with its bf16 gradient per step; throughput in trace nodes per second).

value = B*T / device time per step (CUDA events on the launching stream, L2 flushed between steps by a
256 MB write outside the timed events; each call replayed from a CUDA graph captured after the warm-up).
e2e = the same metric through the C ABI with the step's inputs copied from pinned host memory and its
outputs copied back inside the timed region.  The library is single-GPU: --gpus N > 1 (or a launch under
torchrun with WORLD_SIZE > 1) prints an "unavailable" line and exits.
--impl reference times the CPU oracle on a bounded sample of the same workload.
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
DEFAULT_WORKLOAD = "fp8_long_context"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ES = {"f32": 4, "bf16": 2, "e4m3": 1}
# sources the attention objects are built from: a recorded DRAM traffic figure is valid only while all of
# them are unchanged
ATTN_SOURCES = ("speculative_decoding_tree_verify_gb300/csrc/attn_tc.cu",
                "speculative_decoding_tree_verify_gb300/csrc/tc_ptx.cuh",
                "speculative_decoding_tree_verify_gb300/csrc/sv_internal.cuh",
                "include/sv.h")
ACCEPT_SOURCES = ("speculative_decoding_tree_verify_gb300/csrc/accept.cu",
                  "speculative_decoding_tree_verify_gb300/csrc/sv_internal.cuh",
                  "include/sv.h")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["sv", "reference"], default="sv")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of each CPU-baseline sample")
    ap.add_argument("--ops", nargs="*", default=None,
                    help="instead of the step: time every library call on the named workloads (all if none given), "
                         "one JSON line per call")
    ap.add_argument("--calls", default="attn,accept,loss,bwd,paged,compact,expand",
                    help="with --ops: the calls to time (comma-separated)")
    return ap.parse_args(argv)


def world_size() -> int:
    return int(os.environ.get("WORLD_SIZE", 1))


def rank() -> int:
    return int(os.environ.get("RANK", 0))


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    return dict(FALLBACK), "fallback"


def source_sha(paths) -> str:
    """Hash over the named source files (path and bytes, in order)."""
    h = hashlib.sha256()
    for rel in paths:
        h.update(rel.encode())
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def traffic_from_profile(workload: str, kernel: str, paths):
    """DRAM bytes per launch from profiles/traffic.json, valid only while every source the kernel is built from
    is unchanged (the record's key is source_sha over those files); otherwise None."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    rec = json.loads(p.read_text()).get(f"{kernel}/{workload}")
    if not rec or rec.get("source_sha") != source_sha(paths):
        return None
    return rec["traffic_bytes_per_launch"]


# ------------------------------------------------------------------------------------------ algorithmic work
def ancestors_count(parent_row) -> np.ndarray:
    """|anc(i)| (itself and the root included) for every node of one tree."""
    T = len(parent_row)
    d = np.zeros(T, np.int64)
    for i in range(T):
        d[i] = 1 if i == 0 else d[int(parent_row[i])] + 1
    return d


def attn_bytes(w) -> int:
    """Bytes the method must move: K and V of every allowed position (prefix + tree block) once per kv head,
    Q in, O out, lse out, plus the small int arrays."""
    kv = int(np.sum(w.kv_len.astype(np.int64) + w.T)) * w.Hkv * w.D * 2 * ES[w.kv_dt]
    qo = 2 * w.B * w.T * w.Hq * w.D * ES[w.q_dt]
    return kv + qo + w.B * w.T * w.Hq * 4 + w.B * (w.T + 1) * 4


def attn_flops(w) -> float:
    """FLOPs the method must do: 2*D for q.k and 2*D for p*v per (query row, allowed position)."""
    pairs = sum(int(w.kv_len[b]) * w.T + int(ancestors_count(w.parent[b]).sum()) for b in range(w.B)) * w.Hq
    return 4.0 * w.D * pairs


def workload_modes(name: str):
    """(label, temperature, uses draft logits) of every acceptance call of one step of a named workload."""
    from speculative_decoding_tree_verify_gb300 import workloads as W
    cfg = W.WORKLOADS[name]
    if name == "fp8_long_context":
        return [("greedy", 0.0, False), ("onehot", 0.7, False)]
    if cfg.get("mode") == "prob":
        return [("prob", float(cfg["temperature"]), True)]
    if cfg.get("mode") == "onehot":
        return [("onehot", float(cfg["temperature"]), False)]
    return [("greedy", 0.0, False)]


def accept_modes(w):
    return workload_modes(w.name)


def accept_bytes(w, with_draft: bool) -> int:
    rows = w.B * w.T * (2 if with_draft else 1)
    return rows * w.V * ES[w.logit_dt] + w.B * w.T * 4 * 6


def tensor_core_attn(w) -> bool:
    return w.q_dt == "bf16" and w.kv_dt in ("bf16", "e4m3") and w.D == 128


def workload_config(name: str, args) -> dict:
    """The config object of the JSON line, from the workload table alone (both arms print the same one)."""
    from speculative_decoding_tree_verify_gb300 import workloads as W
    c = W.WORKLOADS[name]
    common = {"seed": args.seed, "l2": "flushed by a 256 MB write between steps",
              "launch": "each call replayed as a CUDA graph captured after the warm-up", "parallelism": "single"}
    if c["kind"] == "loss":
        return dict({"workload": name, "traces": c["N"], "T": c["T"], "tree": str(c["tree"]), "V": c["V"],
                     "logit_dt": "bf16", "grad_dt": "bf16", "accepted_edge_frac": c["accept_frac"]}, **common)
    modes = workload_modes(name)
    return dict({"workload": name, "B": c["B"], "T": c["T"], "tree": str(c["tree"]), "Hq": c["Hq"], "Hkv": c["Hkv"],
                 "D": c["D"], "q_dt": c["q_dt"], "kv_dt": c["kv_dt"], "kv_len_range": list(c["L"]), "V": c["V"],
                 "logit_dt": c["logit_dt"], "accept": [m[0] for m in modes], "temperature": [m[1] for m in modes],
                 "draft_logits": any(m[2] for m in modes)}, **common)


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

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
        for ln in self.lines:
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
def cpu_sample_workload(name: str, seed: int):
    """The bounded sample the oracle is timed on: one request of the named verify workload (or 4 traces of the
    loss batch), drawn on the host by the same recipe."""
    from speculative_decoding_tree_verify_gb300 import workloads as W
    if W.WORKLOADS[name]["kind"] == "loss":
        return W.make_workload(name, seed=seed, N=4)
    over = dict(mode="onehot", temperature=0.7) if name == "fp8_long_context" else {}
    return W.make_workload(name, seed=seed, B=1, **over)


def cpu_oracle_sample(w, budget_s: float):
    """Time the oracle (as it stands, on the threads it is set to) on the sample until the budget is spent.
    Verify: acceptance of the whole request in every mode of the step, then the attention of the request's nodes
    (all heads each) a few at a time; value = nodes / (attention time + acceptance time per node * nodes).
    Loss: whole traces.  Returns (value, threads used, description)."""
    import oracle
    used = oracle.num_threads()
    if hasattr(w, "N"):      # loss batch
        t0 = time.perf_counter()
        n = 0
        while n == 0 or (time.perf_counter() - t0 < budget_s and n < 3):
            oracle.loss_w(w)
            n += 1
        dt = (time.perf_counter() - t0) / n
        return w.N * w.T / dt, used, f"{w.N} traces x {w.T} nodes (loss + fp64 gradient), {n} rep(s)"
    t_acc = 0.0
    for _label, temp, draft in accept_modes(w):
        t0 = time.perf_counter()
        oracle.accept_w(w, temperature=temp, draft=w.draft_logits if draft else None)
        t_acc += time.perf_counter() - t0
    per_node_acc = t_acc / w.T
    nodes, t_attn, step = 0, 0.0, 1
    while nodes < w.T and (nodes == 0 or t_attn + per_node_acc * nodes < budget_s):
        chunk = list(range(nodes, min(w.T, nodes + step)))
        rows = np.array([[0, i, h] for i in chunk for h in range(w.Hq)], np.int32)
        t0 = time.perf_counter()
        oracle.tree_attn_w(w, rows=rows)
        t_attn += time.perf_counter() - t0
        nodes += len(chunk)
        step = min(2 * step, 16)
    desc = (f"one request (L={int(w.kv_len[0])}): acceptance of all {w.T} rows in {len(accept_modes(w))} mode(s), "
            f"attention of {nodes} of {w.T} nodes x {w.Hq} heads")
    return nodes / (t_attn + per_node_acc * nodes), used, desc


def cpu_baselines(name: str, seed: int, budget_s: float):
    """The oracle timed on all host threads and on one thread, on the same sample."""
    import oracle
    w = cpu_sample_workload(name, seed)
    v_all, cores, desc = cpu_oracle_sample(w, budget_s)
    oracle.set_num_threads(1)
    try:
        v_one, one, _ = cpu_oracle_sample(w, budget_s)
    finally:
        oracle.set_num_threads(cores)
    unit = "trace nodes/s" if hasattr(w, "N") else "nodes/s"
    return {"value": v_all, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc,
            "affinity_cpus": len(os.sched_getaffinity(0)),
            "single_thread": {"value": v_one, "unit": unit, "cores": one}}


# ------------------------------------------------------------------------------------------ device helpers
def to_device(a, dev):
    """numpy array from the generator -> CUDA tensor with the same bytes (bf16 bits as int16, uint32 as int32);
    torch tensors are returned as they are."""
    import torch
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(dev)
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).to(dev)


def capture(fn, stream):
    """A CUDA graph of fn captured on a side stream (after the caller's warm-up)."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return g


def timed_graph_steps(graphs, steps, flush, stream, clock_index):
    """Replay the calls' graphs in order once per step, an event before and after each; returns the mean time of
    every call (ms) and the clock summary."""
    import torch
    evs = []
    with ClockSampler(clock_index) as clk:
        for _ in range(steps):
            flush.zero_()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
            e[0].record(stream)
            for i, g in enumerate(graphs):
                g.replay()
                e[i + 1].record(stream)
            evs.append(e)
        torch.cuda.synchronize()
    per_call = [sum(e[i].elapsed_time(e[i + 1]) for e in evs) / steps for i in range(len(graphs))]
    return per_call, clk.summary()


def prefix_rows(kv_len, T, Hkv, kv_cap):
    """The slices of a [B, Hkv, kv_cap, D] cache that a step reads: for every request b and kv head h the first
    kv_len[b] + T positions (the prefix and the tree's own K/V), each one contiguous run of memory."""
    out = []
    for b, L in enumerate(kv_len):
        n = min(int(L) + int(T), int(kv_cap))
        out.extend((b, h, n) for h in range(Hkv))
    return out


def e2e_time(host, dev_sets, call_sets, outs_dev, steps, stream, prefix=None):
    """Per-step time (ms) through the API with every input copied from pinned host memory and the outputs
    copied back, each step.  Two device copies of the inputs (`dev_sets`, with `call_sets` the calls bound to
    each) let the next step's host-to-device copies, on their own stream, run while the current step computes;
    a step's compute waits for its own copies, and a copy into a set waits until the step that last read it is
    done.  The timed region spans the first step's copies to the last step's outputs.  `prefix` maps a cache
    key to `prefix_rows(...)`: only those runs of the cache are copied (the rest is never read)."""
    import torch
    prefix = prefix or {}
    # (destination, source) pairs of each device set, views made once outside the timed region
    plans = []
    for ds in dev_sets:
        plan = []
        for k, t in host.items():
            if k in prefix:
                plan.extend((ds[k][r, h, :n], t[r, h, :n]) for (r, h, n) in prefix[k])
            else:
                plan.append((ds[k], t))
        plans.append(plan)
    outs_host = {k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in outs_dev.items()}
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    for e in done:
        e.record(stream)

    def h2d(b):
        copy_stream.wait_event(done[b])
        with torch.cuda.stream(copy_stream):
            for dst, src in plans[b]:
                dst.copy_(src, non_blocking=True)
            copied[b].record(copy_stream)

    def run(n):
        h2d(0)
        for s in range(n):
            b = s & 1
            if s + 1 < n:
                h2d(b ^ 1)
            stream.wait_event(copied[b])
            for c in call_sets[b]:
                c()
            for k, t in outs_host.items():
                t.copy_(outs_dev[k], non_blocking=True)
            done[b].record(stream)

    run(2)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    copy_stream.wait_stream(stream)
    run(steps)
    t1.record(stream)
    torch.cuda.synchronize()
    h2d_bytes = 0
    for k, t in host.items():
        if k in prefix:
            row = t[0, 0, 0].numel() * t.element_size()
            h2d_bytes += sum(n for (_, _, n) in prefix[k]) * row
        else:
            h2d_bytes += t.numel() * t.element_size()
    d2h_bytes = sum(t.numel() * t.element_size() for t in outs_host.values())
    return t0.elapsed_time(t1) / steps, h2d_bytes, d2h_bytes


# ------------------------------------------------------------------------------------------ the sv arm: verify
def run_sv_verify(args, w):
    import torch

    from speculative_decoding_tree_verify_gb300 import sv

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    names = ("q", "k", "v", "k_scale", "v_scale", "kv_len", "parent", "tokens", "target_logits", "draft_logits",
             "uniforms")
    d = {k: to_device(getattr(w, k), dev) for k in names}
    B, T, V = w.B, w.T, w.V
    i32 = dict(dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, T, w.Hq), dtype=torch.float32, device=dev)
    st_a = torch.empty((B,), **i32)
    ws_attn = torch.empty(max(sv.workspace_size(sv.OP_TREE_ATTN, B, T, w.Hq, w.Hkv, w.D, w.kv_cap, 0), 256),
                          dtype=torch.uint8, device=dev)
    ws_acc = torch.empty(max(sv.workspace_size(sv.OP_ACCEPT, B, T, V=V), 256), dtype=torch.uint8, device=dev)
    modes = accept_modes(w)
    acc = [dict(accept_len=torch.empty((B,), **i32), path=torch.empty((B, T), **i32),
                out_tokens=torch.empty((B, T), **i32), bonus=torch.empty((B,), **i32),
                status=torch.empty((B,), **i32)) for _ in modes]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def make_calls(dd):
        """The step's calls on the inputs in `dd` (outputs and workspaces shared)."""
        tg = dd["target_logits"].view(B, T, V)
        dl = None if dd["draft_logits"] is None else dd["draft_logits"].view(B, T, V)

        def attn_call():
            sv.tree_attn(dd["q"], dd["k"], dd["v"], dd["kv_len"], dd["parent"], out, k_scale=dd["k_scale"],
                         v_scale=dd["v_scale"], lse=lse, status=st_a, workspace=ws_attn)

        def accept_call(i):
            label, temp, with_draft = modes[i]
            a = acc[i]

            def call():
                sv.accept(tg, dd["tokens"], dd["parent"], a["accept_len"], a["path"], a["out_tokens"], a["bonus"],
                          draft_logits=dl if with_draft else None, temperature=temp,
                          uniforms=dd["uniforms"] if temp > 0 else None, status=a["status"], workspace=ws_acc)
            return call

        return [attn_call] + [accept_call(i) for i in range(len(modes))]

    calls = make_calls(d)

    def check(what):
        assert (st_a == 0).all(), f"{what}: attention reported a per-request error"
        for a in acc:
            assert (a["status"] == 0).all(), f"{what}: acceptance reported a per-request error"

    for _ in range(args.warmup):
        flush.zero_()
        for c in calls:
            c()
    torch.cuda.synchronize()
    check("warm-up")
    graphs = [capture(c, stream) for c in calls]
    for _ in range(2):
        flush.zero_()
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    check("graph replay")

    per_call, clocks = timed_graph_steps(graphs, args.steps, flush, stream, 0)
    check("timed steps")
    ms = sum(per_call)
    value = B * T / (ms * 1e-3)
    t_attn, t_acc = per_call[0], sum(per_call[1:])

    e2e = None
    if not args.no_e2e:
        host = {}
        for k in names:
            if d[k] is not None:
                h = torch.empty(d[k].shape, dtype=d[k].dtype).pin_memory()
                h.copy_(d[k])
                host[k] = h
        d2 = {k: (None if t is None else torch.empty_like(t)) for k, t in d.items()}
        outs = {"out": out, "lse": lse}
        for i, a in enumerate(acc):
            outs.update({f"{k}_{modes[i][0]}": t for k, t in a.items()})
        n_e2e = max(3, args.steps // 2)
        runs = prefix_rows(w.kv_len, T, w.Hkv, w.kv_cap)
        ms_e2e, h2d, d2h = e2e_time(host, [d, d2], [calls, make_calls(d2)], outs, n_e2e, stream,
                                    prefix={"k": runs, "v": runs})
        e2e = {"value": B * T / (ms_e2e * 1e-3), "unit": "nodes/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e, "steps": n_e2e,
               "copies": ("every input from pinned host memory each step (of the K/V caches, each request's "
                          "kv_len + T positions per kv head, the part a step reads), on a copy stream into one of "
                          "two device input sets while the previous step computes; outputs back each step")}
        check("end-to-end steps")
        del host, d2

    pk, pk_kind = peaks()
    ab = attn_bytes(w)
    acc_b = [accept_bytes(w, m[2]) for m in modes]
    tc = tensor_core_attn(w)
    if t_attn >= max(per_call[1:]):
        kernel = "sv_tree_attn (attn_tc_kernel + attn_merge_kernel)" if tc else "sv_tree_attn (attn_simt_kernel)"
        hbm_gbs = ab / (t_attn * 1e-3) / 1e9
        hbm = {"achieved": hbm_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": hbm_gbs / pk["hbm_gbs"],
               "algorithmic_bytes_per_launch": ab}
        traffic = traffic_from_profile(w.name, "attn", ATTN_SOURCES) if tc else None
        if w.kv_dt == "e4m3" and tc:
            # FP8 caches: f16 MMAs on exactly converted e4m3 (tensor-bound, as the survey's roofline says), judged
            # against the measured dense bf16 peak (f16 has the same nominal rate); the HBM fraction beside it
            fl = attn_flops(w)
            tf = fl / (t_attn * 1e-3) / 1e12
            roofline = {"bound": "tensor", "kernel": kernel, "achieved": tf, "peak": pk["bf16_tflops"],
                        "peak_kind": f"{pk_kind} bf16 dense burst (f16 MMAs; same nominal rate)", "unit": "TFLOP/s",
                        "frac": tf / pk["bf16_tflops"], "algorithmic_flops_per_launch": fl, "traffic": traffic,
                        "frac_of_sustained": tf / pk["bf16_tflops_sustained"], "hbm": hbm}
        else:
            roofline = dict({"bound": "hbm", "kernel": kernel, "peak_kind": pk_kind, "traffic": traffic}, **hbm)
    else:
        i = int(np.argmax(per_call[1:]))
        gbs = acc_b[i] / (per_call[1 + i] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": f"sv_accept {modes[i][0]} (accept rows + walk kernels)",
                    "achieved": gbs, "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s",
                    "frac": gbs / pk["hbm_gbs"], "algorithmic_bytes_per_launch": acc_b[i],
                    "traffic": traffic_from_profile(w.name, f"accept_{modes[i][0]}", ACCEPT_SOURCES)}
    roofline["step_hbm_frac"] = (ab + sum(acc_b)) / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]
    launches = (2 if tc else 1) + 2 * len(modes)
    dtype = {"f32": "f32", "bf16": "bf16", "e4m3": "f16"}[w.kv_dt]
    comps = {"attn_ms": t_attn, "attn_bytes": ab}
    for (label, _, _), t, b in zip(modes, per_call[1:], acc_b):
        comps[f"accept_{label}_ms"] = t
        comps[f"accept_{label}_bytes"] = b
        comps[f"accept_{label}_hbm_frac"] = b / (t * 1e-3) / 1e9 / pk["hbm_gbs"]
    comps["mean_accept_len"] = {m[0]: float(a["accept_len"].float().mean().item()) for m, a in zip(modes, acc)}
    return {"value": value, "unit": "nodes/s", "ms": ms, "dtype": dtype, "config": workload_config(w.name, args),
            "components": comps, "roofline": roofline, "e2e": e2e, "launches_per_step": launches, "clocks": clocks,
            "data": "synthetic" + (" (caches, Q and logits drawn on the GPU by the generator's device recipe)"
                                   if w.meta.get("device_recipe") else "")}


# ------------------------------------------------------------------------------------------ the sv arm: loss
def run_sv_loss(args, lb):
    import torch

    from speculative_decoding_tree_verify_gb300 import sv

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    N, T, V = lb.N, lb.T, lb.V
    d = {k: to_device(getattr(lb, k), dev) for k in ("logits", "tokens", "parent", "labels")}
    rl = torch.empty((N * T,), dtype=torch.float32, device=dev)
    sums = torch.empty((3,), dtype=torch.float32, device=dev)
    grad = torch.empty_like(d["logits"])
    st = torch.empty((N,), dtype=torch.int32, device=dev)
    ws = torch.empty(max(sv.workspace_size(sv.OP_LOSS, N, T, V=V), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        sv.loss(d["logits"], d["tokens"], d["parent"], d["labels"], rl, sums, grad=grad, status=st, workspace=ws)

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    assert (st == 0).all(), "loss reported a per-trace error"
    g = capture(call, stream)
    per_call, clocks = timed_graph_steps([g], args.steps, flush, stream, 0)
    ms = per_call[0]
    e2e = None
    if not args.no_e2e:
        host = {}
        for k, t in d.items():
            h = torch.empty(t.shape, dtype=t.dtype).pin_memory()
            h.copy_(t)
            host[k] = h
        d2 = {k: torch.empty_like(t) for k, t in d.items()}

        def call2():
            sv.loss(d2["logits"], d2["tokens"], d2["parent"], d2["labels"], rl, sums, grad=grad, status=st,
                    workspace=ws)
        ms_e2e, h2d, d2h = e2e_time(host, [d, d2], [[call], [call2]], {"row_loss": rl, "sums": sums, "grad": grad},
                                    max(3, args.steps // 2), stream)
        e2e = {"value": N * T / (ms_e2e * 1e-3), "unit": "trace nodes/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e}
    pk, pk_kind = peaks()
    nbytes = 2 * N * T * V * 2 + N * T * 16
    gbs = nbytes / (ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "sv_loss (loss_rows_kernel + loss_sums_kernel)", "achieved": gbs,
                "peak": pk["hbm_gbs"], "peak_kind": pk_kind, "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                "algorithmic_bytes_per_launch": nbytes,
                "traffic": traffic_from_profile(lb.name, "loss", ("speculative_decoding_tree_verify_gb300/csrc/loss.cu",
                                                                  "speculative_decoding_tree_verify_gb300/csrc/sv_internal.cuh",
                                                                  "include/sv.h"))}
    return {"value": N * T / (ms * 1e-3), "unit": "trace nodes/s", "ms": ms, "dtype": "bf16",
            "config": workload_config(lb.name, args), "components": {"loss_ms": ms, "loss_bytes": nbytes},
            "roofline": roofline, "e2e": e2e, "launches_per_step": 2, "clocks": clocks, "data": "synthetic"}


def load_workload(name: str, seed: int):
    from speculative_decoding_tree_verify_gb300 import workloads as W
    if name == "fp8_long_context":
        # the full batch (8.6 GB of e4m3 caches, 2.5 GB of logits) is drawn on the GPU; the one-hot mode's
        # uniforms come with it, and the greedy call ignores them
        return W.make_workload(name, seed=seed, device="cuda", mode="onehot", temperature=0.7)
    return W.make_workload(name, seed=seed)


def run_sv(args):
    import torch
    torch.cuda.set_device(0)
    w = load_workload(args.workload, args.seed)
    res = run_sv_loss(args, w) if hasattr(w, "N") else run_sv_verify(args, w)
    cpu = None if args.no_cpu_baseline else cpu_baselines(args.workload, args.seed, args.cpu_seconds)
    line = {"metric": METRIC, "value": res["value"], "unit": res["unit"], "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": res["dtype"], "data": res["data"], "config": res["config"],
            "components": res["components"], "roofline": res["roofline"], "cpu_baseline": cpu, "e2e": res["e2e"],
            "gpu_launches": res["launches_per_step"] * args.steps, "clocks": res["clocks"]}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------ the reference arm
def run_reference(args):
    """The CPU oracle (the pages have no code to install) on the host cores, one bounded sample per step; rank 0
    alone under a multi-process launch."""
    if rank() != 0:
        return
    from speculative_decoding_tree_verify_gb300 import workloads as W
    w = cpu_sample_workload(args.workload, args.seed)
    per_step = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        v, cores, desc = cpu_oracle_sample(w, per_step)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    unit = "trace nodes/s" if hasattr(w, "N") else "nodes/s"
    c = W.WORKLOADS[args.workload]
    nodes = c["N"] * c["T"] if c["kind"] == "loss" else c["B"] * c["T"]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * nodes / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, args),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------ per-call timings
def run_ops(args):
    """One JSON line per (workload, call): median of 10 CUDA-graph replays, each after a 256 MB L2 flush,
    with the call's algorithmic bytes and the fraction of the HBM peak they represent."""
    import torch

    from speculative_decoding_tree_verify_gb300 import sv
    from speculative_decoding_tree_verify_gb300 import workloads as W

    pk, peak_kind = peaks()
    peak = pk["hbm_gbs"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(args.seed)
    dev = lambda a: to_device(a, torch.device("cuda", 0))

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

    def report(name, op, us, nbytes, note="", flops=None):
        gbs = nbytes / (us * 1e-6) / 1e9
        line = {"workload": name, "op": op, "us": round(us, 1), "alg_MB": round(nbytes / 1e6, 3),
                "GB_s": round(gbs, 1), "frac": round(gbs / peak, 3), "peak_kind": peak_kind, "note": note}
        if flops is not None:
            tf = flops / (us * 1e-6) / 1e12
            line.update(TFLOP_s=round(tf, 1), tensor_frac=round(tf / pk["bf16_tflops"], 3))
        print(json.dumps(line), flush=True)

    i32 = dict(dtype=torch.int32, device="cuda")

    def attn_case(name, w):
        q, k, v, ks, vs = dev(w.q), dev(w.k), dev(w.v), dev(w.k_scale), dev(w.v_scale)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        n = sv.workspace_size(sv.OP_TREE_ATTN, w.B, w.T, w.Hq, w.Hkv, w.D, w.kv_cap, 0)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device="cuda")
        kl, par = dev(w.kv_len), dev(w.parent)
        fn = lambda: sv.tree_attn(q, k, v, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st, workspace=ws)
        us = timed(fn, reps=5 if w.kv_dt == "e4m3" else 10)
        assert (st == 0).all(), f"tree_attn statuses {st.cpu().tolist()}"
        report(name, "tree_attn", us, attn_bytes(w), "tensor cores" if tensor_core_attn(w) else "CUDA cores",
               flops=attn_flops(w))

    def accept_case(name, w, temperature, draft):
        B, T, V = w.B, w.T, w.V
        tgt = dev(w.target_logits).view(B, T, V)
        dr = dev(draft).view(B, T, V) if draft is not None else None
        tok, par, u = dev(w.tokens), dev(w.parent), dev(w.uniforms)
        outs = [torch.empty((B,), **i32), torch.empty((B, T), **i32), torch.empty((B, T), **i32),
                torch.empty((B,), **i32)]
        st = torch.empty((B,), **i32)
        ws = torch.empty(max(sv.workspace_size(sv.OP_ACCEPT, B, T, V=V), 256), dtype=torch.uint8, device="cuda")
        fn = lambda: sv.accept(tgt, tok, par, *outs, draft_logits=dr, temperature=temperature,
                               uniforms=u if temperature > 0 else None, status=st, workspace=ws)
        us = timed(fn)
        assert (st == 0).all()
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
        """Tree-attention backward: FLOPs = 10 * D per (query row, allowed position) -- the five products s, dp,
        dq, dk, dv."""
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
        flops = 2.5 * attn_flops(w)
        tf = flops / (us * 1e-6) / 1e12
        print(json.dumps({"workload": name, "op": "tree_attn_bwd", "us": round(us, 1), "TFLOP_s": round(tf, 2),
                          "tensor_frac": round(tf / pk["bf16_tflops"], 4),
                          "note": ("tensor cores" if (w.q_dt == "bf16" and w.kv_dt == "bf16" and w.D == 128) else "CUDA cores")
                                  + "; FLOPs = 10*D per (query row, allowed position)"}), flush=True)

    def paged_case(name, w, page_size=128):
        """Tree attention over the same caches scattered into a page pool; bytes as for the contiguous call."""
        kp, table = W.to_pages(args.seed, w.k, w.kv_len, w.T, page_size)
        vp, _ = W.to_pages(args.seed, w.v, w.kv_len, w.T, page_size)
        q, kpd, vpd, tbl = dev(w.q), dev(kp), dev(vp), dev(table)
        kl, par, ks, vs = dev(w.kv_len), dev(w.parent), dev(w.k_scale), dev(w.v_scale)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda")
        st = torch.empty((w.B,), **i32)
        fn = lambda: sv.tree_attn_paged(q, kpd, vpd, tbl, kl, par, out, k_scale=ks, v_scale=vs, lse=lse, status=st)
        report(name, "tree_attn_paged", timed(fn, reps=5), attn_bytes(w), f"{page_size}-row pages",
               flops=attn_flops(w))

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
        for dd, (nf, kk, nk) in enumerate(levels):
            e = W.make_expand(seed + dd, B=B, n_front=nf, V=V, k=kk, n_keep=nk, logit_dt="bf16", sigma=sigma)
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
            report(name, f"tree_expand_level{dd + 1}", us, nb, f"{nf} x top-{kk} -> {nk}")
        report(name, "tree_expand_all_levels", tot_us, tot_b, f"{len(levels)} calls")

    calls = set(args.calls.split(","))
    which = args.ops or ["tiny_chain", "llama3_8b_tree", "qwen3_8b_stochastic", "loss_batch", "fp8_long_context"]
    for name in which:
        if name == "loss_batch":
            if "loss" in calls:
                loss_case(name, W.make_workload(name, seed=args.seed))
            continue
        w = load_workload(name, args.seed)
        if "attn" in calls:
            attn_case(name, w)
        if "accept" in calls:
            for label, temp, with_draft in accept_modes(w):
                accept_case(name, w, temp, w.draft_logits if with_draft else None)
        if name in ("llama3_8b_tree", "qwen3_8b_stochastic"):
            if "bwd" in calls:
                bwd_case(name, w)
            if "paged" in calls:
                paged_case(name, w)
        if "compact" in calls:
            compact_case(name, w.B, w.T, w.Hkv, w.D, w.kv_cap, w.kv_dt, w.kv_len, w.parent, args.seed)
        if "expand" in calls:
            if name == "llama3_8b_tree":
                expand_case(name, w.B, w.V, W.expansion_levels(60, (4, 3, 2, 2, 1, 1)), 3.0, 200 + args.seed)
            elif name == "qwen3_8b_stochastic":
                expand_case(name, w.B, w.V, [(1, 1, 1)] * 5, 2.5, 300 + args.seed)
            elif name == "fp8_long_context":
                expand_case(name, w.B, w.V, W.expansion_levels(64, (4, 3, 2, 2, 1, 1, 1)), 3.0, 500 + args.seed)
        del w
        torch.cuda.empty_cache()


def unavailable_line(args, why: str) -> dict:
    return {"impl": args.impl, "metric": METRIC, "n_gpus": max(args.gpus, world_size()), "unavailable": why}


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        run_reference(args)
        return
    if args.gpus > 1 or world_size() > 1:
        # the library and its kernels are single-GPU; there is no multi-GPU path to run
        if rank() == 0:
            print(json.dumps(unavailable_line(args, "single-GPU library: the verify path runs on one GPU "
                                                    "(replicas only, no multi-GPU mode is built)")), flush=True)
        return
    if args.ops is not None:
        run_ops(args)
        return
    run_sv(args)


if __name__ == "__main__":
    sys.path.insert(0, str(ROOT))
    main()
