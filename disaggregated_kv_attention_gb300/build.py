"""Build libforkkv.so in-tree: every CUDA/C++ source compiled for sm_103a with nvcc.

Objects are compiled in parallel into ``_build/`` at the repository root and
linked (with the static CUDA runtime) into ``libforkkv.so`` next to this file.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libforkkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]
CUDA_FLAGS = ARCH + COMMON + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]

SOURCES = [
    "allocator.cpp",
    "plan.cpp",
    "abi.cu",
    "kernels/rows.cu",
    "kernels/decode.cu",
    "kernels/prefill.cu",
    "kernels/fill.cu",
    "decode_static.cu",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libforkkv")


def _compile(src: str, verbose_ptxas: bool) -> str:
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src.replace("/", "_") + ".o")
    flags = list(CUDA_FLAGS)
    if verbose_ptxas and src.endswith(".cu"):
        flags += ["-Xptxas", "-v"]
    if src.endswith(".cpp"):
        flags = ARCH + COMMON + ["-x", "cu"]
    cmd = [nvcc()] + flags + ["-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {src}\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def _stale(objs_srcs) -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES]
    deps += [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "kernels", "common.cuh"),
             os.path.join(CSRC, "kernels", "tcgen05.cuh"),
             os.path.join(ROOT, "include", "forkkv.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link libforkkv.so; returns its path (skips work when up to date)."""
    if not force and not verbose_ptxas and not _stale(SOURCES):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
