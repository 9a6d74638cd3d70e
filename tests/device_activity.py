"""Device activities (kernels, copies, memsets) a piece of code puts on the GPU, recorded
with the CUPTI activity API by the small C helper tests/cupti_activity.c (built here with
gcc against the CUDA toolkit's CUPTI)."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cupti_activity.c")
LIB = os.path.join(HERE, "libcupti_activity.so")
_lib = None


def _cuda_root():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        root = _cuda_root()
        libdir = os.path.join(root, "lib64")
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-shared", "-fPIC", SRC, f"-I{os.path.join(root, 'include')}", f"-L{libdir}",
                        "-lcupti", f"-Wl,-rpath,{libdir}", "-o", tmp], check=True)
        os.replace(tmp, LIB)
    lib = ctypes.CDLL(LIB)
    lib.dtk_activity_start.restype = ctypes.c_int
    lib.dtk_activity_stop.restype = ctypes.c_int
    lib.dtk_activity_get.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_int),
                                     ctypes.c_char_p, ctypes.c_int]
    _lib = lib
    return lib


KINDS = {0: "kernel", 1: "memcpy", 2: "memset"}


def record(fn, synchronize):
    """[(kind, name)] of the device activities fn issues, in start order; `synchronize`
    waits for the device before and after."""
    lib = load()
    synchronize()
    rc = lib.dtk_activity_start()
    if rc != 0:
        raise RuntimeError(f"CUPTI activity recording could not start (CUPTI status {rc})")
    try:
        fn()
        synchronize()
    finally:
        n = lib.dtk_activity_stop()
    if n < 0:
        raise RuntimeError("too many device activities to record")
    out = []
    buf = ctypes.create_string_buffer(256)
    for i in range(n):
        start, kind = ctypes.c_uint64(), ctypes.c_int()
        lib.dtk_activity_get(i, ctypes.byref(start), ctypes.byref(kind), buf, 256)
        out.append((start.value, KINDS[kind.value], buf.value.decode(errors="replace")))
    return [(k, name) for _, k, name in sorted(out)]
