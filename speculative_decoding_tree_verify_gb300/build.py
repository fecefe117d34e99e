"""Build libsv.so (the CUDA library behind include/sv.h) in-tree for sm_103a.

Each .cu file is compiled in parallel to an object with nvcc, then linked into
speculative_decoding_tree_verify_gb300/_build/libsv.so with the CUDA runtime linked statically.
Usage: python -m speculative_decoding_tree_verify_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = BUILD / "libsv.so"
INCLUDE = PKG.parent / "include"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-Xcompiler", "-Wall"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _stale(obj: Path, src: Path, deps: list[Path]) -> bool:
    if not obj.exists():
        return True
    t = obj.stat().st_mtime
    return any(p.stat().st_mtime > t for p in [src, *deps])


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> Path:
    BUILD.mkdir(exist_ok=True)
    deps = list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    todo = []
    objs = []
    for src in sources():
        obj = BUILD / (src.stem + ".o")
        objs.append(obj)
        if force or verbose_ptxas or _stale(obj, src, deps):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [cc, *ARCH, *CFLAGS, *extra, "-I", str(INCLUDE), "-c", str(src), "-o", str(obj) + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stderr}")
        os.replace(str(obj) + ".tmp", obj)
        return src.name, r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for name, err in ex.map(compile_one, todo):
                if verbose_ptxas and err:
                    sys.stderr.write(f"--- {name}\n{err}")
    if todo or not LIB.exists():
        cmd = [cc, *ARCH, "-shared", "-o", str(LIB) + ".tmp", *map(str, objs), "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(str(LIB) + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas))
