"""Thin Python binding of libsv.so (include/sv.h): argument marshalling only.

Every function takes torch tensors that already live on the GPU, passes their device pointers, sizes and
the current CUDA stream to the C entry point of the same name, and raises SVError on a non-OK status.  No
computation happens here, and there is no CPU fallback: if the CUDA library has not been built, loading
fails loudly.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "_build" / "libsv.so"

OK, ERR_INVALID_ARG, ERR_BAD_TREE, ERR_TREE_TOO_LARGE, ERR_UNSUPPORTED, ERR_NONFINITE, ERR_TIMEOUT, ERR_CUDA, \
    ERR_WORKSPACE = range(9)
F32, BF16, E4M3, E2M1 = 0, 1, 2, 3
OP_TREE_ATTN, OP_ACCEPT, OP_LOSS, OP_TREE_ATTN_BWD = 0, 1, 2, 3

_lib = None


class SVError(RuntimeError):
    def __init__(self, code: int, fn: str):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} (status {code})")


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"libsv.so is not built ({LIB_PATH}); run "
                               "`python -m speculative_decoding_tree_verify_gb300.build`")
        L = C.CDLL(str(LIB_PATH))
        P, i, f, z = C.c_void_p, C.c_int, C.c_float, C.c_size_t
        L.sv_status_string.argtypes = [i]
        L.sv_status_string.restype = C.c_char_p
        L.sv_version.restype = i
        L.sv_set_wait_limit.argtypes = [C.c_longlong]
        L.sv_set_wait_limit.restype = i
        L.sv_workspace_size.argtypes = [i] * 8
        L.sv_workspace_size.restype = z
        L.sv_tree_attn.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, P, P, f, P, P, P, P, z, P]
        L.sv_tree_attn.restype = i
        L.sv_accept.argtypes = [i, i, i, i, P, P, P, P, f, P, P, P, P, P, P, P, P, z, P]
        L.sv_accept.restype = i
        L.sv_loss.argtypes = [i, i, i, P, P, P, P, P, P, P, P, P, z, P]
        L.sv_loss.restype = i
        L.sv_accept_noalloc.argtypes = [i, i, i, i, P, P, P, P, f, P, P, P, P, P, P, P, P]
        L.sv_accept_noalloc.restype = i
        L.sv_tree_attn_paged.argtypes = [i, i, i, i, i, i, i, i, i, i, P, P, P, P, P, P, P, P, f, P, P, P, P, z, P]
        L.sv_tree_attn_paged.restype = i
        L.sv_tree_attn_fp4.argtypes = [i, i, i, i, i, i, i, P, P, P, P, P, P, P, P, P, f, P, P, P, P, z, P]
        L.sv_tree_attn_fp4.restype = i
        L.sv_tree_attn_bwd.argtypes = [i, i, i, i, i, i, i, i, P, P, P, P, P, f, P, P, P, P, P, P, P, P, z, P]
        L.sv_tree_attn_bwd.restype = i
        L.sv_kv_compact.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P]
        L.sv_kv_compact.restype = i
        L.sv_tree_expand.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, P, P, P]
        L.sv_tree_expand.restype = i
        _lib = L
    return _lib


def set_wait_limit(sm_cycles: int) -> None:
    """sv_set_wait_limit: bounded-wait limit of the attention kernels in SM cycles (0 = default, about 1 s)."""
    _check(lib().sv_set_wait_limit(int(sm_cycles)), "sv_set_wait_limit")


def status_string(code: int) -> str:
    return lib().sv_status_string(int(code)).decode()


def workspace_size(op: int, B: int, T: int, Hq: int = 0, Hkv: int = 0, D: int = 0, kv_cap: int = 0,
                   V: int = 0) -> int:
    return int(lib().sv_workspace_size(op, B, T, Hq, Hkv, D, kv_cap, V))


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype in (torch.bfloat16, torch.uint16, torch.int16):      # bf16 values or their bit patterns
        return BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libsv must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libsv must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ws(op, workspace, *dims):
    if workspace is not None:
        return workspace
    n = workspace_size(op, *dims)
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda") if n else None


def _check(code, fn):
    if code != OK:
        raise SVError(code, fn)


def tree_attn(q, k_cache, v_cache, kv_len, parent, out, *, k_scale=None, v_scale=None, sm_scale=0.0, lse=None,
              status=None, workspace=None, stream=None):
    """sv_tree_attn: q [B,T,Hq,D]; caches [B,Hkv,kv_cap,D]; out like q."""
    B, T, Hq, D = q.shape
    Hkv, kv_cap = k_cache.shape[1], k_cache.shape[2]
    ws = _ws(OP_TREE_ATTN, workspace, B, T, Hq, Hkv, D, kv_cap, 0)
    code = lib().sv_tree_attn(B, T, Hq, Hkv, D, kv_cap, dtype_code(q), dtype_code(k_cache), _ptr(q), _ptr(k_cache),
                              _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(kv_len), _ptr(parent),
                              float(sm_scale), _ptr(out), _ptr(lse), _ptr(status), _ptr(ws),
                              0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "sv_tree_attn")


def tree_attn_paged(q, k_pool, v_pool, page_table, kv_len, parent, out, *, k_scale=None, v_scale=None, sm_scale=0.0,
                    lse=None, status=None, workspace=None, stream=None):
    """sv_tree_attn_paged: q [B,T,Hq,D]; pools [num_pages,Hkv,page_size,D]; page_table [B,max_pages]; out like q."""
    B, T, Hq, D = q.shape
    num_pages, Hkv, page_size = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    max_pages = page_table.shape[1]
    ws = _ws(OP_TREE_ATTN, workspace, B, T, Hq, Hkv, D, page_size * max_pages, 0)
    code = lib().sv_tree_attn_paged(B, T, Hq, Hkv, D, page_size, max_pages, num_pages, dtype_code(q),
                                    dtype_code(k_pool), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(page_table), _ptr(kv_len), _ptr(parent), float(sm_scale),
                                    _ptr(out), _ptr(lse), _ptr(status), _ptr(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "sv_tree_attn_paged")


def tree_attn_fp4(q, k_codes, v_codes, k_block, v_block, k_scale, v_scale, kv_len, parent, out, *, sm_scale=0.0,
                  lse=None, status=None, workspace=None, stream=None):
    """sv_tree_attn_fp4: q [B,T,Hq,D] bf16; codes [B,Hkv,kv_cap,D/2] uint8; block scales [B,Hkv,kv_cap,D/16] uint8
    (E4M3); head scales [Hkv] float; out like q."""
    B, T, Hq, D = q.shape
    Hkv, kv_cap = k_codes.shape[1], k_codes.shape[2]
    ws = _ws(OP_TREE_ATTN, workspace, B, T, Hq, Hkv, D, kv_cap, 0)
    code = lib().sv_tree_attn_fp4(B, T, Hq, Hkv, D, kv_cap, dtype_code(q), _ptr(q), _ptr(k_codes), _ptr(v_codes),
                                  _ptr(k_block), _ptr(v_block), _ptr(k_scale), _ptr(v_scale), _ptr(kv_len),
                                  _ptr(parent), float(sm_scale), _ptr(out), _ptr(lse), _ptr(status), _ptr(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "sv_tree_attn_fp4")


def accept(target_logits, tokens, parent, accept_len, path, out_tokens, bonus, *, draft_logits=None,
           temperature=0.0, uniforms=None, argmax=None, status=None, workspace=None, stream=None):
    """sv_accept: logits [B,T,V]; tokens/parent [B,T]; outputs accept_len [B], path/out_tokens [B,T], bonus [B]."""
    B, T, V = target_logits.shape
    ws = _ws(OP_ACCEPT, workspace, B, T, 0, 0, 0, 0, V)
    code = lib().sv_accept(B, T, V, dtype_code(target_logits), _ptr(target_logits), _ptr(draft_logits),
                           _ptr(tokens), _ptr(parent), float(temperature), _ptr(uniforms), _ptr(accept_len),
                           _ptr(path), _ptr(out_tokens), _ptr(bonus), _ptr(argmax), _ptr(status), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "sv_accept")


def accept_noalloc(target_logits, tokens, parent, accept_len, path, out_tokens, bonus, *, draft_logits=None,
                   temperature=0.0, uniforms=None, argmax=None, status=None, stream=None):
    """sv_accept_noalloc: sv_accept using the library's built-in scratch (no workspace argument)."""
    B, T, V = target_logits.shape
    code = lib().sv_accept_noalloc(B, T, V, dtype_code(target_logits), _ptr(target_logits), _ptr(draft_logits),
                                   _ptr(tokens), _ptr(parent), float(temperature), _ptr(uniforms),
                                   _ptr(accept_len), _ptr(path), _ptr(out_tokens), _ptr(bonus), _ptr(argmax),
                                   _ptr(status), _stream(stream))
    _check(code, "sv_accept_noalloc")


def loss(draft_logits, tokens, parent, labels, row_loss, sums, *, grad=None, status=None, workspace=None,
         stream=None):
    """sv_loss: draft_logits [N*T,V] bf16; tokens/parent/labels [N,T]; row_loss [N*T]; sums [3]; grad like logits."""
    N, T = parent.shape
    V = draft_logits.shape[-1]
    ws = _ws(OP_LOSS, workspace, N, T, 0, 0, 0, 0, V)
    code = lib().sv_loss(N, T, V, _ptr(draft_logits), _ptr(tokens), _ptr(parent), _ptr(labels), _ptr(row_loss),
                         _ptr(sums), _ptr(grad), _ptr(status), _ptr(ws), ws.numel() * ws.element_size(),
                         _stream(stream))
    _check(code, "sv_loss")


def kv_compact(k_cache, v_cache, kv_len, parent, accept_len, path, new_kv_len, *, status=None, stream=None):
    """sv_kv_compact: caches [B,Hkv,kv_cap,D] (modified in place); kv_len/accept_len/new_kv_len [B]; parent/path [B,T]."""
    B, Hkv, kv_cap, D = k_cache.shape
    T = parent.shape[1]
    code = lib().sv_kv_compact(B, T, Hkv, D, kv_cap, dtype_code(k_cache), _ptr(k_cache), _ptr(v_cache), _ptr(kv_len),
                               _ptr(parent), _ptr(accept_len), _ptr(path), _ptr(new_kv_len), _ptr(status),
                               _stream(stream))
    _check(code, "sv_kv_compact")


def tree_expand(logits, front_score, k, n_keep, topk_token, topk_logprob, child_parent, child_token, child_score, *,
                status=None, stream=None):
    """sv_tree_expand: logits [B,n_front,V]; front_score [B,n_front]; topk_* [B,n_front,k]; child_* [B,n_keep]."""
    B, n_front, V = logits.shape
    code = lib().sv_tree_expand(B, n_front, V, int(k), int(n_keep), dtype_code(logits), _ptr(logits),
                                _ptr(front_score), _ptr(topk_token), _ptr(topk_logprob), _ptr(child_parent),
                                _ptr(child_token), _ptr(child_score), _ptr(status), _stream(stream))
    _check(code, "sv_tree_expand")


def tree_attn_bwd(q, k_cache, v_cache, kv_len, parent, out, lse, dout, dq, dk, dv, *, sm_scale=0.0, status=None,
                  workspace=None, stream=None):
    """sv_tree_attn_bwd: forward inputs plus out / lse / dout [B,T,Hq,D]; dq like q (fp32); dk, dv like the caches (fp32)."""
    B, T, Hq, D = q.shape
    Hkv, kv_cap = k_cache.shape[1], k_cache.shape[2]
    ws = _ws(OP_TREE_ATTN_BWD, workspace, B, T, Hq, Hkv, D, kv_cap, 0)
    code = lib().sv_tree_attn_bwd(B, T, Hq, Hkv, D, kv_cap, dtype_code(q), dtype_code(k_cache), _ptr(q), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(kv_len), _ptr(parent), float(sm_scale), _ptr(out), _ptr(lse),
                                  _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(status), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream))
    _check(code, "sv_tree_attn_bwd")
