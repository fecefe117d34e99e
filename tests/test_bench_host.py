"""Host-side logic of bench.py (CPU only): the single-GPU refusal of multi-GPU launches, the reference arm's
rank-0 rule, identical config objects on both arms, the algorithmic work counts and the source hash that keys
recorded DRAM traffic."""
import json
import os
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
from speculative_decoding_tree_verify_gb300 import workloads as W  # noqa: E402


def test_multi_gpu_launch_prints_unavailable_and_exits_zero():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert "unavailable" in line and line["n_gpus"] == 2


def test_torchrun_style_launch_is_refused_on_every_rank(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--steps", "1", "--warmup", "3"])            # rank 1: nothing printed, nothing run
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.main(["--steps", "1", "--warmup", "3"])
    assert "unavailable" in json.loads(capsys.readouterr().out)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.parse(["--impl", "reference", "--workload", "tiny_chain"]))
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_both_arms_print_the_same_config(name):
    a = bench.parse(["--workload", name])
    cfg = bench.workload_config(name, a)
    assert cfg == bench.workload_config(name, bench.parse(["--impl", "reference", "--workload", name]))
    assert cfg["workload"] == name
    if W.WORKLOADS[name]["kind"] == "verify":
        assert cfg["kv_len_range"] == list(W.WORKLOADS[name]["L"]) and len(cfg["temperature"]) == len(cfg["accept"])


def test_attention_work_counts_match_a_brute_force_count():
    w = W.make_verify(3, B=3, T=13, Hq=4, Hkv=2, D=64, L=(5, 40), V=16, q_dt="bf16", kv_dt="bf16", tree=(3, 2, 2))
    pairs = 0
    for b in range(w.B):
        for i in range(w.T):
            anc, x = set(), i
            while x >= 0:
                anc.add(x)
                x = int(w.parent[b, x])
            pairs += int(w.kv_len[b]) + len(anc)
    assert bench.attn_flops(w) == 4.0 * w.D * w.Hq * pairs
    kv = sum(int(w.kv_len[b]) + w.T for b in range(w.B)) * w.Hkv * w.D * 2 * 2
    assert bench.attn_bytes(w) == kv + 2 * w.B * w.T * w.Hq * w.D * 2 + w.B * w.T * w.Hq * 4 + w.B * (w.T + 1) * 4


def test_end_to_end_cache_copies_cover_exactly_what_attention_reads():
    """The end-to-end leg copies, per request and kv head, the first kv_len + T cache positions: one contiguous
    run each in the [B, Hkv, kv_cap, D] layout, together the cache bytes of the attention's algorithmic count."""
    w = W.make_verify(5, B=4, T=7, Hq=4, Hkv=2, D=16, L=(3, 30), V=16, q_dt="bf16", kv_dt="bf16", tree="chain")
    runs = bench.prefix_rows(w.kv_len, w.T, w.Hkv, w.kv_cap)
    assert sorted((b, h) for b, h, _ in runs) == [(b, h) for b in range(w.B) for h in range(w.Hkv)]
    for b, h, n in runs:
        assert n == int(w.kv_len[b]) + w.T <= w.kv_cap
    cache_bytes = 2 * sum(n for _, _, n in runs) * w.D * 2
    assert cache_bytes == sum(int(w.kv_len[b]) + w.T for b in range(w.B)) * w.Hkv * w.D * 2 * 2
    src = np.arange(w.k.size, dtype=np.int64).reshape(w.k.shape)
    dst = np.full_like(src, -1)
    for b, h, n in runs:
        dst[b, h, :n] = src[b, h, :n]
    for b in range(w.B):
        n = int(w.kv_len[b]) + w.T
        assert (dst[b, :, :n] == src[b, :, :n]).all() and (dst[b, :, n:] == -1).all()


def test_default_workload_runs_both_acceptance_modes():
    assert bench.parse([]).workload == "fp8_long_context"
    assert [m[0] for m in bench.workload_modes("fp8_long_context")] == ["greedy", "onehot"]
    assert bench.workload_modes("qwen3_8b_stochastic") == [("prob", 1.0, True)]


def test_recorded_traffic_is_void_once_a_source_changes(tmp_path, monkeypatch):
    (tmp_path / "a.cu").write_text("x")
    (tmp_path / "b.cuh").write_text("y")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    key = bench.source_sha(["a.cu", "b.cuh"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"attn/wl": {"source_sha": key, "traffic_bytes_per_launch": 123}}))
    assert bench.traffic_from_profile("wl", "attn", ["a.cu", "b.cuh"]) == 123
    (tmp_path / "b.cuh").write_text("y2")                    # an included header changed
    assert bench.traffic_from_profile("wl", "attn", ["a.cu", "b.cuh"]) is None


def test_cpu_baseline_sample_on_the_tiny_workload():
    cpu = bench.cpu_baselines("tiny_chain", 0, 0.2)
    assert cpu["value"] > 0 and cpu["single_thread"]["value"] > 0 and cpu["single_thread"]["cores"] == 1
    assert cpu["kind"] == "oracle" and "one request" in cpu["sample"]
    import oracle
    assert oracle.num_threads() == cpu["cores"]              # the thread count is restored
