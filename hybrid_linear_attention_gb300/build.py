"""Builds libkda.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc.

Each .cu under csrc/ is compiled to an object in parallel, then linked with nvcc -shared
(static CUDA runtime).  The result lands at hybrid_linear_attention_gb300/libkda.so.
Set KDA_PTXAS_VERBOSE=1 to print register/shared-memory usage per kernel.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the KDA library needs the CUDA 13 toolkit to build")


def _flags():
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "--expt-relaxed-constexpr"]
    if os.environ.get("KDA_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _deps_mtime():
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles every kernel source and links libkda.so; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources]

    def compile_one(src, obj):
        cmd = [nvcc, "-c", src, "-o", obj] + _flags()
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        logs = list(ex.map(compile_one, sources, objs))
    if verbose or os.environ.get("KDA_PTXAS_VERBOSE"):
        for src, log in zip(sources, logs):
            if log.strip():
                print(f"== {os.path.basename(src)}\n{log}", file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared", "-o", tmp] + objs + ARCH, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
