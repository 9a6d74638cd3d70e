"""Python binding of the C ABI in include/indexer_topk.h (argument marshalling only).

Every step of the scan runs in the CUDA library; this module only converts torch
tensors and streams to pointers and status codes to exceptions. PyTorch serves for
device memory and streams. If the compiled library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdtk_indexer_topk.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "indexer_topk.h")

ITK_OK = 0
STATUS_NAMES = {}


class IndexerTopkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


class _Desc(ctypes.Structure):
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
        ("key_id_base", ctypes.c_int32),
    ]


_lib = None


def _status_constants():
    consts = {}
    with open(HEADER) as f:
        for m in re.finditer(r"\b(ITK_[A-Z_]+)\s*=\s*(\d+)", f.read()):
            consts[m.group(1)] = int(m.group(2))
    return consts


def header_functions():
    """Names of the functions the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:ITK_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**(indexer_topk_[a-z_]+)\s*\(",
                                 text, re.M)))


def load():
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library {LIB_PATH} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
    DP = ctypes.POINTER(_Desc)
    sig = {
        "indexer_topk_prepare": (ctypes.c_int, [DP, vp, ctypes.POINTER(vp)]),
        "indexer_topk_workspace_bytes": (sz, [vp]),
        "indexer_topk_run": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "indexer_topk_eager_workspace_bytes": (sz, [DP]),
        "indexer_topk_eager": (ctypes.c_int, [DP, vp, vp, vp, vp, vp, vp, sz, vp]),
        "indexer_topk_destroy": (None, [vp]),
        "indexer_topk_device_status": (ctypes.c_int, [vp, vp]),
        "indexer_topk_validate": (ctypes.c_int, [DP]),
        "indexer_topk_num_units": (i64, [DP]),
        "indexer_topk_unit_table": (i64, [DP, vp, i64]),
        "indexer_topk_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "indexer_topk_last_error": (ctypes.c_char_p, []),
        "indexer_topk_version": (ctypes.c_char_p, []),
        "indexer_topk_debug_inject": (ctypes.c_int, [vp, ctypes.c_int, vp]),
        "indexer_topk_run_noalloc": (ctypes.c_int, [DP, vp, vp, vp, vp, vp, vp]),
        "indexer_topk_noalloc_scratch_bytes": (sz, []),
        "indexer_topk_noalloc_device_status": (ctypes.c_int, [vp]),
        "indexer_topk_eager_device_status": (ctypes.c_int, [DP, vp, sz, vp]),
        "indexer_topk_set_split_event": (ctypes.c_int, [vp, vp]),
        "indexer_topk_bench_hold": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _ = i32
    _lib = lib
    return lib


def _check(rc: int):
    if rc != ITK_OK:
        lib = load()
        detail = lib.indexer_topk_last_error().decode()
        name = lib.indexer_topk_status_string(rc).decode()
        raise IndexerTopkError(rc, f"{name}: {detail}")


class Desc:
    """Host descriptor; keeps the int32 arrays alive while the C side may read them."""

    def __init__(self, T, Tkv, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets=None, H=64, D=128, key_id_base=0):
        import numpy as np

        self.cu_q = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.cu_k = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
        self.offs = None if q_causal_offsets is None else np.ascontiguousarray(q_causal_offsets, dtype=np.int32)
        self.c = _Desc(int(T), int(Tkv), int(H), int(D), int(top_k), len(self.cu_q) - 1, self.cu_q.ctypes.data,
                       self.cu_k.ctypes.data, None if self.offs is None else self.offs.ctypes.data, int(key_id_base))
        self.T, self.Tkv, self.top_k, self.H, self.D = int(T), int(Tkv), int(top_k), int(H), int(D)
        self.key_id_base = int(key_id_base)

    def ref(self):
        return ctypes.byref(self.c)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _current_cuda_device():
    """The CUDA device the library will launch on (the calling thread's current device)."""
    import torch

    return torch.device("cuda", torch.cuda.current_device())


def _check_buffers(desc: Desc, q, k, w, out_ids, out_scores, workspace=None):
    """The checks the C ABI cannot make on plain pointers: every tensor given is a
    contiguous CUDA tensor of the expected dtype, on the current CUDA device (the library
    launches there, on that device's stream), holding at least the elements the call reads
    or writes (a flat buffer is fine: the library reads rows of H*D, D and H elements and
    writes rows of top_k). A missing buffer (None) is left to the library, which reports
    ITK_ERR_NULL_POINTER; alignment is checked there too."""
    import torch

    T, Tkv, K, H, D = desc.T, desc.Tkv, desc.top_k, desc.H, desc.D
    want = (("q", q, torch.bfloat16, T * H * D), ("k", k, torch.bfloat16, Tkv * D), ("w", w, torch.float32, T * H),
            ("out_ids", out_ids, torch.int32, T * K), ("out_scores", out_scores, torch.float32, T * K),
            ("workspace", workspace, None, 0))
    dev = next((t.device for _, t, _, _ in want if t is not None), None)
    if dev is not None and dev.type == "cuda":
        cur = _current_cuda_device()
        if dev != cur:
            raise IndexerTopkError(STATUS_NAMES.get("ITK_ERR_INVALID_ARGUMENT", 1),
                                   f"buffers on {dev}, but the current CUDA device is {cur}: the library launches "
                                   "on the current device (use torch.cuda.device(...) around the call)")
    for name, t, dtype, n in want:
        if t is None:
            continue
        bad = []
        if not t.is_cuda:
            bad.append(f"on {t.device}, not a CUDA device")
        elif t.device != dev:
            bad.append(f"on {t.device}, the other buffers on {dev}")
        if dtype is not None and t.dtype != dtype:
            bad.append(f"dtype {t.dtype}, want {dtype}")
        if not t.is_contiguous():
            bad.append("not contiguous")
        if t.numel() < n:
            bad.append(f"{t.numel()} elements, want at least {n}")
        if bad:
            raise IndexerTopkError(STATUS_NAMES.get("ITK_ERR_INVALID_ARGUMENT", 1), f"{name}: " + "; ".join(bad))


class Plan:
    """A prepared runner (owns the plan's device block)."""

    def __init__(self, desc: Desc, stream=None):
        lib = load()
        h = ctypes.c_void_p()
        _check(lib.indexer_topk_prepare(desc.ref(), _stream_handle(stream), ctypes.byref(h)))
        self._h = h
        self.desc = desc

    @property
    def handle(self):
        return self._h

    def workspace_bytes(self) -> int:
        return int(load().indexer_topk_workspace_bytes(self._h))

    def device_status(self, stream=None):
        _check(load().indexer_topk_device_status(self._h, _stream_handle(stream)))

    def destroy(self):
        if self._h:
            load().indexer_topk_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def indexer_topk_prepare(T, Tkv, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets=None, H=64, D=128,
                         stream=None, key_id_base=0) -> Plan:
    return Plan(Desc(T, Tkv, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets, H, D, key_id_base), stream)


def indexer_topk_workspace_bytes(plan: Plan) -> int:
    return plan.workspace_bytes()


def indexer_topk_run(plan: Plan, q, k, w, out_ids, out_scores, workspace, stream=None):
    """q BF16 [T,64,128], k BF16 [Tkv,128], w FP32 [T,64], out_ids INT32 [T,top_k], out_scores FP32 [T,top_k]."""
    _check_buffers(plan.desc, q, k, w, out_ids, out_scores, workspace)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().indexer_topk_run(plan.handle, _ptr(q), _ptr(k), _ptr(w), _ptr(out_ids), _ptr(out_scores),
                                   _ptr(workspace), nbytes, _stream_handle(stream)))


def indexer_topk_eager_workspace_bytes(desc: Desc) -> int:
    return int(load().indexer_topk_eager_workspace_bytes(desc.ref()))


def indexer_topk_eager(desc: Desc, q, k, w, out_ids, out_scores, workspace, stream=None):
    _check_buffers(desc, q, k, w, out_ids, out_scores, workspace)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().indexer_topk_eager(desc.ref(), _ptr(q), _ptr(k), _ptr(w), _ptr(out_ids), _ptr(out_scores),
                                     _ptr(workspace), nbytes, _stream_handle(stream)))


def indexer_topk_eager_device_status(desc: Desc, workspace, stream=None):
    """Raise if an eager call with this descriptor and workspace gave up a bounded wait or
    failed an internal check (reads and clears the status word kept in the workspace)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().indexer_topk_eager_device_status(desc.ref(), _ptr(workspace), nbytes, _stream_handle(stream)))


def indexer_topk_validate(desc: Desc) -> int:
    return int(load().indexer_topk_validate(desc.ref()))


def indexer_topk_unit_table(desc: Desc):
    import numpy as np

    lib = load()
    n = int(lib.indexer_topk_num_units(desc.ref()))
    if n < 0:
        _check(-n)
    out = np.zeros((max(n, 1), 6), np.int32)
    m = int(lib.indexer_topk_unit_table(desc.ref(), out.ctypes.data, n))
    if m < 0:
        _check(-m)
    return out[:n]


def indexer_topk_run_noalloc(desc: Desc, q, k, w, out_ids, out_scores, stream=None):
    """The scan through the entry point that allocates nothing (static device scratch).

    For callers that must not allocate device memory at call time, e.g. a runtime that has
    already reserved the device memory for its own pool. Calls share one scratch array, so
    calls that overlap on the GPU race; keep them on one stream or ordered."""
    _check_buffers(desc, q, k, w, out_ids, out_scores)
    _check(load().indexer_topk_run_noalloc(desc.ref(), _ptr(q), _ptr(k), _ptr(w), _ptr(out_ids), _ptr(out_scores),
                                           _stream_handle(stream)))


def indexer_topk_noalloc_device_status(stream=None):
    """Raise if the last no-allocation call on the current device gave up a bounded wait or
    failed an internal check (reads and clears the status word of the static scratch)."""
    _check(load().indexer_topk_noalloc_device_status(_stream_handle(stream)))


def indexer_topk_set_split_event(plan: Plan, event=None):
    """Record `event` (a torch.cuda.Event that has been recorded once, or a raw
    cudaEvent_t handle) between the scan and the selection launch of later runs; None
    stops it."""
    handle = None if event is None else (event.cuda_event if hasattr(event, "cuda_event") else int(event))
    _check(load().indexer_topk_set_split_event(plan.handle, handle))


def indexer_topk_bench_hold(n_ctas: int, microseconds: int, stream=None):
    """Keep n_ctas SMs busy for `microseconds` with a kernel on `stream` (benchmark aid)."""
    _check(load().indexer_topk_bench_hold(int(n_ctas), int(microseconds), _stream_handle(stream)))


def indexer_topk_debug_inject(plan, what: int, stream=None):
    """Test hook (see the header); plan None targets the next eager or no-allocation call (what = 5)."""
    handle = None if plan is None else plan.handle
    _check(load().indexer_topk_debug_inject(handle, int(what), _stream_handle(stream)))


def indexer_topk(q, k, w, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets=None, stream=None, key_id_base=0):
    """One-shot scan through the eager entry; allocates outputs and workspace with torch."""
    import torch

    T, Tkv = q.shape[0], k.shape[0]
    desc = Desc(T, Tkv, cu_seqlens_q, cu_seqlens_k, top_k, q_causal_offsets, q.shape[1], q.shape[2], key_id_base)
    ids = torch.empty((T, top_k), dtype=torch.int32, device=q.device)
    scores = torch.empty((T, top_k), dtype=torch.float32, device=q.device)
    ws = torch.empty(max(indexer_topk_eager_workspace_bytes(desc), 1), dtype=torch.uint8, device=q.device)
    indexer_topk_eager(desc, q, k, w, ids, scores, ws, stream)
    return ids, scores


STATUS_NAMES.update(_status_constants())
globals().update(STATUS_NAMES)
