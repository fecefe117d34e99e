"""sv_accept_noalloc against sv_accept: the allocation-free variant must give the same bits.

sv_accept_noalloc exists for callers that cannot allocate device memory for a workspace (a serving loop
whose allocator belongs to another framework, a plugin with no allocator of its own, a path that must never
call cudaMalloc).  It keeps its scratch in a fixed static device array inside the library instead.  This
file runs last so that a stop-at-first-failure run has already run every other test; it passes alone in a
fresh process as well as after the rest.

Each case makes two sv_accept_noalloc calls in a row on different inputs (the second finds the first's
leftovers in the shared array) and compares every integer output of both with sv_accept's, bit for bit, and
the first call's with the CPU oracle's as well.  One case uses the scratch to its last row.
"""
import numpy as np
import pytest
import torch

import oracle

from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

KEYS = ("status", "accept_len", "path", "out_tokens", "bonus", "argmax")


def _outputs(B, T):
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(accept_len=torch.full((B,), -9, **i32), path=torch.full((B, T), -9, **i32),
                out_tokens=torch.full((B, T), -9, **i32), bonus=torch.full((B,), -9, **i32),
                argmax=torch.full((B, T), -9, **i32), status=torch.full((B,), -9, **i32))


def _call(fn, w, temperature):
    B, T, V = w.B, w.T, w.V
    res = _outputs(B, T)
    tgt = dev(w.target_logits).view(B, T, V)
    dr = dev(w.draft_logits).view(B, T, V) if (temperature > 0 and w.draft_logits is not None) else None
    fn(tgt, dev(w.tokens), dev(w.parent), res["accept_len"], res["path"], res["out_tokens"], res["bonus"],
       draft_logits=dr, temperature=temperature, uniforms=dev(w.uniforms), argmax=res["argmax"],
       status=res["status"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


CASES = [
    # (workload, overrides for the first call, overrides for the second call)
    ("llama3_8b_tree", dict(seed=0), dict(seed=1)),
    ("qwen3_8b_stochastic", dict(seed=0), dict(seed=1, B=4)),
    ("tiny_chain", dict(seed=0, V=1000), dict(seed=2, V=4096, temperature=0.7, mode="prob")),
]


@pytest.mark.parametrize("name,first,second", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_accept_two_calls(name, first, second):
    for n, over in enumerate((first, second)):
        over = dict(over)
        seed = over.pop("seed")
        w = W.make_workload(name, seed=seed, with_attn=False, **over)
        want = _call(sv.accept, w, w.temperature)
        got = _call(sv.accept_noalloc, w, w.temperature)
        for k in KEYS:
            np.testing.assert_array_equal(got[k], want[k], err_msg=k)
        assert (got["status"] == 0).all()
        if n == 0:
            ref = oracle.accept_w(w)
            for k in KEYS:
                np.testing.assert_array_equal(got[k], ref[k], err_msg=f"oracle {k}")


def test_noalloc_uses_the_whole_scratch():
    # 16384 chains of 4 nodes = 65536 target rows, the scratch's limit, with draft rows (stochastic, PROB mode):
    # the array's last row records are written and read; then a small call reuses the array
    w = W.make_verify(11, B=16384, T=4, Hq=1, Hkv=1, D=16, L=(0, 0), V=16, q_dt="f32", kv_dt="f32",
                      logit_dt="bf16", tree="chain", mode="prob", temperature=0.9, with_attn=False)
    for case in (w, W.make_verify(12, B=3, T=4, Hq=1, Hkv=1, D=16, L=(0, 0), V=16, logit_dt="bf16", tree="chain",
                                  mode="prob", temperature=0.9, with_attn=False)):
        want = _call(sv.accept, case, case.temperature)
        got = _call(sv.accept_noalloc, case, case.temperature)
        for k in KEYS:
            np.testing.assert_array_equal(got[k], want[k], err_msg=k)
        assert (got["status"] == 0).all()
    ref = oracle.accept_w(w)
    got = _call(sv.accept_noalloc, w, w.temperature)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"oracle {k}")


def test_noalloc_rejects_oversized_batch():
    # 1100 x 60 target rows exceed the 65536-row scratch: refused on the host before any launch.
    B, T, V = 1100, 60, 16
    tgt = torch.zeros((B, T, V), dtype=torch.float32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    parent = torch.arange(-1, T - 1, **i32).repeat(B, 1)
    res = _outputs(B, T)
    with pytest.raises(sv.SVError) as e:
        sv.accept_noalloc(tgt, torch.zeros((B, T), **i32), parent, res["accept_len"], res["path"],
                          res["out_tokens"], res["bonus"])
    assert e.value.code == sv.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (res["accept_len"].cpu() == -9).all()
