"""Compile the CUDA library in-tree for sm_103a (one translation unit, one -gencode)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libdtk_indexer_topk.so")
SOURCES = [os.path.join(CSRC, "itk_host.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("itk_common.cuh", "itk_scan.cuh", "itk_select.cuh", "itk_ptx.cuh")] + [
    os.path.join(ROOT, "include", "indexer_topk.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17", "-shared",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def nvcc_path() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build the library")
    return p


def build(force: bool = False, verbose: bool = False) -> str:
    newest = max(os.path.getmtime(f) for f in DEPS)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp, *SOURCES]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":  # pragma: no cover
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
