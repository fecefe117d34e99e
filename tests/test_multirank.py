"""The multi-rank path of bench.py on CPU: two gloo ranks (one process each, 127.0.0.1) agree on the
slowest rank's step time, the throughput counts every rank's batch, each rank draws its own batch, and the
reference arm runs on rank 0 only."""
import os
import socket
import sys
from pathlib import Path

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from speculative_decoding_tree_verify_gb300 import workloads as W
        ms = 1.0 + 0.5 * rank                           # rank 1 is the slow one
        m = bench.max_over_ranks(ms, world)
        w = W.make_workload("tiny_chain", seed=bench.rank_seed(0, rank))
        out[rank] = (m, bench.nodes_per_second(w.B, w.T, world, m), int(w.target_logits.view(np.uint32).sum() % 1000003))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    (m0, v0, h0), (m1, v1, h1) = out[0], out[1]
    assert m0 == m1 == 1.5                                   # max over ranks
    assert v0 == v1 == 1 * 6 * world / 1.5e-3               # B * T * world / max step time
    assert h0 != h1                                          # each rank has its own batch


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.nodes_per_second(8, 60, 1, 0.1) == 8 * 60 / 1e-4


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, str(ROOT))
    import bench

    class Args:
        workload, seed, steps, warmup = "tiny_chain", 0, 1, 0

    bench.run_reference(Args, rank=1, world=2)           # returns at once, prints nothing
    assert capsys.readouterr().out == ""
