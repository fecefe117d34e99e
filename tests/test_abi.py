"""The C ABI without a GPU: libsv.so builds and loads, exports every entry point include/sv.h declares,
and rejects bad host-visible arguments synchronously with the documented codes.

Every call below fails validation before anything is launched (each case carries at least one invalid
host-visible argument), so no device memory is touched and no GPU is needed.
"""
import ctypes as C
import re
from pathlib import Path

import pytest

from speculative_decoding_tree_verify_gb300 import build as sv_build
from speculative_decoding_tree_verify_gb300 import sv

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def L():
    sv_build.build()
    return sv.lib()


def declared_functions():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"sv_tree_attn", "sv_accept", "sv_loss", "sv_workspace_size", "sv_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    for code in range(9):
        assert sv.status_string(code) and sv.status_string(code) != "unknown status"
    assert sv.status_string(99) == "unknown status"
    assert L.sv_version() >= 100


def test_workspace_sizes(L):
    assert sv.workspace_size(sv.OP_ACCEPT, 8, 60, V=128256) >= 2 * 8 * 60 * 24
    assert sv.workspace_size(sv.OP_LOSS, 64, 32, V=128256) >= 2 * 64 * 32 * 4
    assert sv.workspace_size(sv.OP_ACCEPT, 8, 65, V=10) == 0      # T > 64 is never valid
    for op in (0, 1, 2):
        assert sv.workspace_size(op, 4, 8, 8, 2, 128, 512, 1000) % 256 == 0


FAKE = C.c_void_p(0x100000)      # 16-byte aligned, never dereferenced (validation fails first)
ODD = C.c_void_p(0x100002)       # misaligned


def attn(L, **kw):
    a = dict(B=2, T=4, Hq=4, Hkv=2, D=64, kv_cap=64, q_dt=sv.BF16, kv_dt=sv.BF16, q=FAKE, k=FAKE, v=FAKE, ks=None,
             vs=None, kv_len=FAKE, parent=FAKE, scale=0.0, out=FAKE, lse=None, status=None, ws=None, ws_bytes=0)
    a.update(kw)
    return L.sv_tree_attn(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["kv_cap"], a["q_dt"], a["kv_dt"], a["q"],
                          a["k"], a["v"], a["ks"], a["vs"], a["kv_len"], a["parent"], a["scale"], a["out"],
                          a["lse"], a["status"], a["ws"], a["ws_bytes"], None)


def test_tree_attn_host_validation(L):
    assert attn(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert attn(L, T=0) == sv.ERR_INVALID_ARG
    assert attn(L, Hq=3) == sv.ERR_INVALID_ARG                  # Hq % Hkv != 0
    assert attn(L, kv_cap=3) == sv.ERR_INVALID_ARG              # kv_cap < T
    assert attn(L, B=-1) == sv.ERR_INVALID_ARG
    assert attn(L, scale=float("nan")) == sv.ERR_INVALID_ARG
    assert attn(L, q_dt=sv.E4M3) == sv.ERR_UNSUPPORTED
    assert attn(L, kv_dt=7) == sv.ERR_UNSUPPORTED
    assert attn(L, q=None) == sv.ERR_INVALID_ARG
    assert attn(L, out=None) == sv.ERR_INVALID_ARG
    assert attn(L, kv_dt=sv.E4M3) == sv.ERR_INVALID_ARG         # scales required
    assert attn(L, k=ODD) == sv.ERR_UNSUPPORTED
    assert attn(L, B=0) == sv.OK                                # empty batch: nothing to do


def accept(L, **kw):
    a = dict(B=2, T=4, V=100, dt=sv.BF16, tgt=FAKE, dr=None, tok=FAKE, par=FAKE, temp=0.0, u=None, al=FAKE,
             path=FAKE, ot=FAKE, bonus=FAKE, am=None, st=None, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    return L.sv_accept(a["B"], a["T"], a["V"], a["dt"], a["tgt"], a["dr"], a["tok"], a["par"], a["temp"], a["u"],
                       a["al"], a["path"], a["ot"], a["bonus"], a["am"], a["st"], a["ws"], a["ws_bytes"], None)


def test_accept_host_validation(L):
    assert accept(L, T=70) == sv.ERR_TREE_TOO_LARGE
    assert accept(L, V=0) == sv.ERR_INVALID_ARG
    assert accept(L, temp=-1.0) == sv.ERR_INVALID_ARG
    assert accept(L, temp=float("inf")) == sv.ERR_INVALID_ARG
    assert accept(L, temp=1.0, u=None) == sv.ERR_INVALID_ARG    # stochastic needs uniforms
    assert accept(L, dt=sv.E4M3) == sv.ERR_UNSUPPORTED
    assert accept(L, tgt=None) == sv.ERR_INVALID_ARG
    assert accept(L, bonus=None) == sv.ERR_INVALID_ARG
    assert accept(L, tgt=ODD) == sv.ERR_UNSUPPORTED
    assert accept(L, ws=None) == sv.ERR_WORKSPACE
    assert accept(L, ws_bytes=16) == sv.ERR_WORKSPACE
    assert accept(L, B=0) == sv.OK


def loss(L, **kw):
    a = dict(N=2, T=4, V=100, z=FAKE, tok=FAKE, par=FAKE, lab=FAKE, rl=FAKE, sums=FAKE, g=None, st=None, ws=FAKE,
             ws_bytes=1 << 20)
    a.update(kw)
    return L.sv_loss(a["N"], a["T"], a["V"], a["z"], a["tok"], a["par"], a["lab"], a["rl"], a["sums"], a["g"],
                     a["st"], a["ws"], a["ws_bytes"], None)


def test_loss_host_validation(L):
    assert loss(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert loss(L, V=1) == sv.ERR_INVALID_ARG
    assert loss(L, N=-2) == sv.ERR_INVALID_ARG
    assert loss(L, sums=None) == sv.ERR_INVALID_ARG
    assert loss(L, lab=None) == sv.ERR_INVALID_ARG
    assert loss(L, g=ODD) == sv.ERR_UNSUPPORTED
    assert loss(L, ws=None) == sv.ERR_WORKSPACE


def paged(L, **kw):
    a = dict(B=2, T=4, Hq=4, Hkv=2, D=64, P=16, maxp=8, nump=20, q_dt=sv.BF16, kv_dt=sv.BF16, q=FAKE, k=FAKE, v=FAKE,
             ks=None, vs=None, pt=FAKE, kv_len=FAKE, parent=FAKE, scale=0.0, out=FAKE, lse=None, st=None, ws=None,
             ws_bytes=0)
    a.update(kw)
    return L.sv_tree_attn_paged(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["P"], a["maxp"], a["nump"], a["q_dt"],
                                a["kv_dt"], a["q"], a["k"], a["v"], a["ks"], a["vs"], a["pt"], a["kv_len"], a["parent"],
                                a["scale"], a["out"], a["lse"], a["st"], a["ws"], a["ws_bytes"], None)


def test_tree_attn_paged_host_validation(L):
    assert paged(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert paged(L, P=24) == sv.ERR_INVALID_ARG                # page size not a power of two
    assert paged(L, P=0) == sv.ERR_INVALID_ARG
    assert paged(L, maxp=0) == sv.ERR_INVALID_ARG
    assert paged(L, P=1, maxp=3) == sv.ERR_INVALID_ARG         # capacity below T
    assert paged(L, nump=0) == sv.ERR_INVALID_ARG
    assert paged(L, Hq=3) == sv.ERR_INVALID_ARG
    assert paged(L, q_dt=sv.E4M3) == sv.ERR_UNSUPPORTED
    assert paged(L, D=512) == sv.ERR_UNSUPPORTED
    assert paged(L, pt=None) == sv.ERR_INVALID_ARG
    assert paged(L, kv_dt=sv.E4M3) == sv.ERR_INVALID_ARG       # e4m3 needs its scales
    assert paged(L, k=ODD) == sv.ERR_UNSUPPORTED
    assert paged(L, B=0) == sv.OK


def attn_fp4(L, **kw):
    a = dict(B=2, T=4, Hq=4, Hkv=2, D=128, kv_cap=64, q_dt=sv.BF16, q=FAKE, kc=FAKE, vc=FAKE, kb=FAKE, vb=FAKE,
             ks=FAKE, vs=FAKE, kv_len=FAKE, parent=FAKE, scale=0.0, out=FAKE, lse=None, st=None, ws=None, ws_bytes=0)
    a.update(kw)
    return L.sv_tree_attn_fp4(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["kv_cap"], a["q_dt"], a["q"], a["kc"], a["vc"],
                              a["kb"], a["vb"], a["ks"], a["vs"], a["kv_len"], a["parent"], a["scale"], a["out"],
                              a["lse"], a["st"], a["ws"], a["ws_bytes"], None)


def test_tree_attn_fp4_host_validation(L):
    assert attn_fp4(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert attn_fp4(L, Hq=3) == sv.ERR_INVALID_ARG
    assert attn_fp4(L, kv_cap=2) == sv.ERR_INVALID_ARG          # capacity below T
    assert attn_fp4(L, D=64) == sv.ERR_UNSUPPORTED
    assert attn_fp4(L, q_dt=sv.F32) == sv.ERR_UNSUPPORTED
    assert attn_fp4(L, kv_cap=65) == sv.ERR_UNSUPPORTED         # odd capacity: block scales read two rows at a time
    assert attn_fp4(L, kb=None) == sv.ERR_INVALID_ARG
    assert attn_fp4(L, vs=None) == sv.ERR_INVALID_ARG
    assert attn_fp4(L, kc=ODD) == sv.ERR_UNSUPPORTED
    assert attn_fp4(L, B=0) == sv.OK


def attn_bwd(L, **kw):
    a = dict(B=2, T=4, Hq=4, Hkv=2, D=64, kv_cap=64, q_dt=sv.BF16, kv_dt=sv.BF16, q=FAKE, k=FAKE, v=FAKE,
             kv_len=FAKE, parent=FAKE, scale=0.0, out=FAKE, lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, st=None,
             ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    return L.sv_tree_attn_bwd(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["kv_cap"], a["q_dt"], a["kv_dt"], a["q"],
                              a["k"], a["v"], a["kv_len"], a["parent"], a["scale"], a["out"], a["lse"], a["dout"],
                              a["dq"], a["dk"], a["dv"], a["st"], a["ws"], a["ws_bytes"], None)


def test_tree_attn_bwd_host_validation(L):
    assert attn_bwd(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert attn_bwd(L, Hq=3) == sv.ERR_INVALID_ARG
    assert attn_bwd(L, kv_cap=2) == sv.ERR_INVALID_ARG
    assert attn_bwd(L, scale=-1.0) == sv.ERR_INVALID_ARG
    assert attn_bwd(L, kv_dt=sv.E4M3) == sv.ERR_UNSUPPORTED       # the backward takes bf16 / fp32 caches
    assert attn_bwd(L, D=96) == sv.ERR_UNSUPPORTED
    assert attn_bwd(L, Hq=64, Hkv=2, D=128) == sv.ERR_UNSUPPORTED  # G * D above 2048
    assert attn_bwd(L, lse=None) == sv.ERR_INVALID_ARG
    assert attn_bwd(L, dv=None) == sv.ERR_INVALID_ARG
    assert attn_bwd(L, dq=ODD) == sv.ERR_UNSUPPORTED
    assert attn_bwd(L, ws=None) == sv.ERR_WORKSPACE
    assert attn_bwd(L, ws_bytes=8) == sv.ERR_WORKSPACE
    assert attn_bwd(L, B=0) == sv.OK
    assert sv.workspace_size(sv.OP_TREE_ATTN_BWD, 8, 60, 32) >= 8 * 60 * 32 * 4


def compact(L, **kw):
    a = dict(B=2, T=4, Hkv=2, D=64, kv_cap=64, dt=sv.BF16, k=FAKE, v=FAKE, kv_len=FAKE, par=FAKE, al=FAKE, path=FAKE,
             nl=C.c_void_p(0x200000), st=None)
    a.update(kw)
    return L.sv_kv_compact(a["B"], a["T"], a["Hkv"], a["D"], a["kv_cap"], a["dt"], a["k"], a["v"], a["kv_len"],
                           a["par"], a["al"], a["path"], a["nl"], a["st"], None)


def test_kv_compact_host_validation(L):
    assert compact(L, T=65) == sv.ERR_TREE_TOO_LARGE
    assert compact(L, T=0) == sv.ERR_INVALID_ARG
    assert compact(L, kv_cap=3) == sv.ERR_INVALID_ARG
    assert compact(L, Hkv=0) == sv.ERR_INVALID_ARG
    assert compact(L, dt=5) == sv.ERR_UNSUPPORTED
    assert compact(L, D=12) == sv.ERR_UNSUPPORTED               # 24-byte rows are not 16-byte multiples
    assert compact(L, D=4096, dt=sv.F32) == sv.ERR_UNSUPPORTED  # rows above 8 KB
    assert compact(L, path=None) == sv.ERR_INVALID_ARG
    assert compact(L, nl=FAKE) == sv.ERR_INVALID_ARG            # new_kv_len aliases kv_len
    assert compact(L, k=ODD) == sv.ERR_UNSUPPORTED
    assert compact(L, B=0) == sv.OK


def expand(L, **kw):
    a = dict(B=2, NF=4, V=100, k=4, keep=8, dt=sv.BF16, z=FAKE, fs=FAKE, tt=FAKE, tl=FAKE, cp=FAKE, ct=FAKE, cs=FAKE,
             st=None)
    a.update(kw)
    return L.sv_tree_expand(a["B"], a["NF"], a["V"], a["k"], a["keep"], a["dt"], a["z"], a["fs"], a["tt"], a["tl"],
                            a["cp"], a["ct"], a["cs"], a["st"], None)


def test_tree_expand_host_validation(L):
    assert expand(L, k=0) == sv.ERR_INVALID_ARG
    assert expand(L, k=17) == sv.ERR_INVALID_ARG                # k above 16
    assert expand(L, V=3) == sv.ERR_INVALID_ARG                 # k > V
    assert expand(L, keep=17) == sv.ERR_INVALID_ARG             # more survivors than candidates
    assert expand(L, NF=300, k=4, keep=1) == sv.ERR_INVALID_ARG # more than 1024 candidates
    assert expand(L, NF=0) == sv.ERR_INVALID_ARG
    assert expand(L, dt=sv.E4M3) == sv.ERR_UNSUPPORTED
    assert expand(L, tt=None) == sv.ERR_INVALID_ARG
    assert expand(L, cs=None) == sv.ERR_INVALID_ARG
    assert expand(L, z=ODD) == sv.ERR_UNSUPPORTED
    assert expand(L, B=0) == sv.OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sv, "_lib", None)
    monkeypatch.setattr(sv, "LIB_PATH", tmp_path / "missing.so")
    with pytest.raises(RuntimeError, match="not built"):
        sv.lib()
