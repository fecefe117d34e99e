"""Helpers for the GPU parity tests: move generator arrays to the device and call the library."""
import numpy as np
import torch

from speculative_decoding_tree_verify_gb300 import sv


def dev(a):
    """numpy array from the generators -> CUDA tensor with the same bytes (bf16 bits travel as int16); tensors
    drawn on the GPU by the generator's device recipe pass through."""
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


def host_f32(t, dt):
    """Device output -> float64 numpy (bf16 outputs arrive as int16 bit patterns)."""
    x = t.cpu()
    if dt == "bf16":
        x = x.view(torch.int16).numpy().view(np.uint16)
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.numpy().astype(np.float64)


def run_attn(w, sm_scale=0.0, with_lse=True):
    q = dev(w.q)
    k = dev(w.k)
    v = dev(w.v)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.T, w.Hq), dtype=torch.float32, device="cuda") if with_lse else None
    status = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    sv.tree_attn(q, k, v, dev(w.kv_len), dev(w.parent), out, k_scale=dev(w.k_scale), v_scale=dev(w.v_scale),
                 sm_scale=sm_scale, lse=lse, status=status)
    torch.cuda.synchronize()
    return (host_f32(out, w.q_dt), None if lse is None else lse.cpu().numpy().astype(np.float64),
            status.cpu().numpy())


def run_accept(target, tokens, parent, *, V, temperature=0.0, draft=None, uniforms=None, want_argmax=True):
    B, T = parent.shape
    i32 = dict(dtype=torch.int32, device="cuda")
    res = dict(accept_len=torch.full((B,), -9, **i32), path=torch.full((B, T), -9, **i32),
               out_tokens=torch.full((B, T), -9, **i32), bonus=torch.full((B,), -9, **i32),
               argmax=torch.full((B, T), -9, **i32) if want_argmax else None, status=torch.full((B,), -9, **i32))
    tgt = dev(target).view(B, T, V)
    dr = None if draft is None else dev(draft).view(B, T, V)
    sv.accept(tgt, dev(tokens), dev(parent), res["accept_len"], res["path"], res["out_tokens"], res["bonus"],
              draft_logits=dr, temperature=temperature, uniforms=dev(uniforms), argmax=res["argmax"],
              status=res["status"])
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in res.items()}


def run_loss(lb, want_grad=True):
    N, T, V = lb.N, lb.T, lb.V
    row_loss = torch.full((N * T,), float("nan"), dtype=torch.float32, device="cuda")
    sums = torch.full((3,), float("nan"), dtype=torch.float32, device="cuda")
    grad = torch.full((N * T, V), 0x7FC0, dtype=torch.int16, device="cuda") if want_grad else None
    status = torch.full((N,), -9, dtype=torch.int32, device="cuda")
    sv.loss(dev(lb.logits), dev(lb.tokens), dev(lb.parent), dev(lb.labels), row_loss, sums, grad=grad, status=status)
    torch.cuda.synchronize()
    return dict(row_loss=row_loss.cpu().numpy().astype(np.float64), sums=sums.cpu().numpy().astype(np.float64),
                grad=None if grad is None else host_f32(grad, "bf16"), status=status.cpu().numpy())
