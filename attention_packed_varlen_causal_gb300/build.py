"""Builds the in-tree CUDA library ``libbgattn.so`` for sm_103a.

Each translation unit is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a), then linked into one shared
library with the CUDA runtime linked statically, so loading it needs no
CUDA runtime on the library path.  Objects go to ``_build/`` at the
repository root (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libbgattn.so")
SOURCES = ["abi.cu", "prefill.cu", "decode.cu", "reorder.cu", "noalloc.cu", "lasttok.cu", "select.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _flags(verbose_ptxas: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _deps():
    files = [os.path.join(CSRC, n) for n in os.listdir(CSRC)] + [os.path.join(INCLUDE, "bg_attn.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _deps():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc()] + _flags(verbose_ptxas) + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose_ptxas or r.returncode != 0:
            sys.stderr.write(f"---- {s}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(s for s, _ in failed))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc()] + ARCH + ["-shared", "--cudart", "static", "-o", tmp] + [o for _, o, _ in results]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, verbose_ptxas="-v" in sys.argv)
    print(LIB_PATH)
