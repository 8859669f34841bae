"""Builds libbsa.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each translation unit is compiled in parallel into ``_build/`` and linked
into ``block_sparse_attention_bsa_gb300/libbsa.so``.  Run as
``python -m block_sparse_attention_bsa_gb300.build`` or call ``build()``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbsa.so")
SOURCES = ("bsa_api.cu", "bsa_select.cu", "bsa_fmha.cu", "bsa_bwd.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _flags(verbose_ptxas: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                "-I", os.path.join(ROOT, "include"), "-DNDEBUG"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, verbose_ptxas: bool) -> tuple:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + _flags(verbose_ptxas)
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "bsa.h"),
                                                                 os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = False) -> str:
    """Compiles the library if a source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, log in results:
        if log.strip() and (verbose_ptxas or rc != 0) and not quiet:
            print(f"--- {src} ---\n{log}", file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(r[0] for r in failed) + ":\n" +
                           "\n".join(r[3] for r in failed))
    tmp = LIB + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + [r[1] for r in results] + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
