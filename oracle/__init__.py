"""Oracle for the deterministic lightning-indexer top-k scan (ctypes loader).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package. The product path
(the CUDA library under ``deterministic_top_key_gb300``) never imports it, and
this package imports nothing from the product path.

The arithmetic lives in ``indexer_topk_oracle.c`` (plain C, fp64 sums, one
rounding to FP32, full sort with the larger-id tie-break). What it follows:
flashinfer PR #8691 ("perf(cake_dsa_indexer_det): ticket scheduling on sm_107a,
no fill kernel in eager entry"), opening description (dtypes, exact top-k ids
per query, ties to the larger id, partition independence) and the vendoring
note for cake_dsa_indexer_det ("lightning-indexer scores and deterministic exact
top-k").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "indexer_topk_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_indexer_topk.so")

# No fast-math and no FMA contraction: the fp64 sums are then the same on x86 and Arm.
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle library with gcc (idempotent unless ``force``)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32),
        ("Tkv", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("D", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("num_segments", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("q_causal_offsets", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        # DTK_ORACLE_LIB points the loader at another build of the same source; the
        # mutation test uses it to check that the pins reject planted mistakes.
        path = os.environ.get("DTK_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(_Problem)
        i32p = ctypes.c_void_p
        lib.dtk_oracle_topk.argtypes = [P, i32p, ctypes.c_int32, i32p, i32p, ctypes.c_int32]
        lib.dtk_oracle_scores.argtypes = [P, i32p, i32p, ctypes.c_int64, i32p, ctypes.c_int32]
        lib.dtk_oracle_visibility.argtypes = [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                              ctypes.POINTER(ctypes.c_int32)]
        lib.dtk_oracle_bruteforce.argtypes = [P, i32p, i32p]
        lib.dtk_oracle_max_threads.argtypes = []
        for f in (lib.dtk_oracle_topk, lib.dtk_oracle_scores, lib.dtk_oracle_visibility,
                  lib.dtk_oracle_bruteforce, lib.dtk_oracle_max_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


class Problem:
    """Host-side problem description; q/k are BF16 bit patterns (uint16)."""

    def __init__(self, q_bits, k_bits, w, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets=None):
        q_bits = np.asarray(q_bits)
        k_bits = np.asarray(k_bits)
        if q_bits.ndim != 3 or k_bits.ndim != 2:
            raise ValueError("q must be [T,H,D] and k must be [Tkv,D]")
        T, H, D = q_bits.shape
        Tkv = k_bits.shape[0]
        if k_bits.shape[1] != D or np.asarray(w).shape != (T, H):
            raise ValueError("shape mismatch between q, k and w")
        self._keep = []
        self.q, qp = _c(q_bits, np.uint16)
        self.k, kp = _c(k_bits, np.uint16)
        self.w, wp = _c(w, np.float32)
        self.cu_q, cqp = _c(cu_seqlens_q, np.int32)
        self.cu_k, ckp = _c(cu_seqlens_k, np.int32)
        if q_causal_offsets is None:
            self.offsets, op = None, None
        else:
            self.offsets, op = _c(q_causal_offsets, np.int32)
        self.T, self.Tkv, self.H, self.D, self.top_k = T, Tkv, H, D, int(top_k)
        self.num_segments = len(self.cu_q) - 1
        self._s = _Problem(T, Tkv, H, D, int(top_k), self.num_segments, cqp, ckp, op, qp, kp, wp)

    def _ptr(self):
        return ctypes.byref(self._s)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (status {rc})")


def topk(p: Problem, rows=None, nthreads: int = 0):
    """(ids [n,top_k] int32, scores [n,top_k] float32) for all rows or the listed query rows."""
    lib = _load()
    if rows is None:
        n, rp = p.T, None
    else:
        rows, rp = _c(rows, np.int32)
        n = len(rows)
    ids = np.empty((n, p.top_k), np.int32)
    sc = np.empty((n, p.top_k), np.float32)
    _check(lib.dtk_oracle_topk(p._ptr(), rp, n, ids.ctypes.data, sc.ctypes.data, int(nthreads)), "topk")
    return ids, sc


def scores(p: Problem, t_idx, s_idx, nthreads: int = 0):
    """FP32 scores of the (query row, global key row) pairs."""
    lib = _load()
    t_idx, tp = _c(t_idx, np.int32)
    s_idx, sp = _c(s_idx, np.int32)
    if t_idx.shape != s_idx.shape:
        raise ValueError("t_idx and s_idx differ in shape")
    out = np.empty(t_idx.shape, np.float32)
    _check(lib.dtk_oracle_scores(p._ptr(), tp, sp, t_idx.size, out.ctypes.data, int(nthreads)), "scores")
    return out


def visibility(p: Problem, t: int):
    """(first global key row of t's segment, number of keys query t sees)."""
    lib = _load()
    kb, nv = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.dtk_oracle_visibility(p._ptr(), int(t), ctypes.byref(kb), ctypes.byref(nv)), "visibility")
    return kb.value, nv.value


def bruteforce(p: Problem):
    """Rank-counting selection for tiny inputs (independent of the sort path)."""
    lib = _load()
    ids = np.empty((p.T, p.top_k), np.int32)
    sc = np.empty((p.T, p.top_k), np.float32)
    _check(lib.dtk_oracle_bruteforce(p._ptr(), ids.ctypes.data, sc.ctypes.data), "bruteforce")
    return ids, sc


def max_threads() -> int:
    return int(_load().dtk_oracle_max_threads())


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
