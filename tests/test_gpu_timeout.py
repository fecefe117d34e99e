"""The time-out path of the tensor-core attention, driven on purpose without faulting or hanging the GPU.

sv_set_wait_limit shrinks the limit of the attention kernel's bounded waits so far that waits give up at once (the
copies and MMAs themselves run normally): the kernel winds down, waiting with the full limit for its own copies and
MMAs before it exits, and every request reports SV_ERR_TIMEOUT.  With the default limit restored, the same call on
the same context gives the oracle's result again."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_verify_gb300 import sv
from speculative_decoding_tree_verify_gb300 import workloads as W
from tests.gpu_util import run_attn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_dt,G", [("bf16", 4), ("e4m3", 8), ("bf16", 3)])
def test_forced_timeout_reports_status_and_leaves_the_context_usable(kv_dt, G):
    w = W.make_verify(41, B=3, T=13, Hq=2 * G, Hkv=2, D=128, L=(300, 900), V=16, q_dt="bf16", kv_dt=kv_dt,
                      tree=(3, 2, 2))
    try:
        sv.set_wait_limit(1)   # one SM cycle: a wait that is not already complete gives up
        out, lse, st = run_attn(w)
        assert (st == sv.ERR_TIMEOUT).all(), st
    finally:
        sv.set_wait_limit(0)
    out, lse, st = run_attn(w)
    ref, ref_lse, ref_st, _ = oracle.tree_attn_w(w)
    assert (st == 0).all()
    assert np.abs(out - ref).max() <= (6e-2 if kv_dt == "e4m3" else 2e-2)


def test_wait_limit_rejects_negative_values():
    with pytest.raises(sv.SVError):
        sv.set_wait_limit(-5)
