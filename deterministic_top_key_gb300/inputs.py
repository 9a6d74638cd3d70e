"""Seeded synthetic inputs for the indexer top-k scan.

This module only draws numbers. It holds none of the scan's arithmetic, so the
CUDA path and the CPU oracle can both take their inputs from it.

Shapes follow the workload rows of flashinfer PR #8691's tables (single causal
documents S1/S2, the CP tail C1, the packed CP16 rows Z2cp and Z3cp and the split-tail
rows A1-A3); the
distributions are the ones the rows are benchmarked with here: q, k ~ N(0,1)
rounded to BF16 and w ~ N(0,1)/8 (the tiny case uses w ~ U(-1,1)). Every case
also has an integer variant, q, k uniform over {-2..2} and w uniform over
{-1, 0.5, 1, 2}, for which every FP32 sum in the scan is exact.

Streams: q draws from ``seed``, k from ``seed + 1``, w from ``seed + 2``
(numpy PCG64), so the inputs are identical on every machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

H_HEADS = 64
D_HEAD = 128


@dataclass
class Workload:
    name: str
    q_bits: np.ndarray  # [T,H,D] uint16 (BF16 bit patterns)
    k_bits: np.ndarray  # [Tkv,D] uint16
    w: np.ndarray  # [T,H] float32
    cu_seqlens_q: np.ndarray  # [B+1] int32
    cu_seqlens_k: np.ndarray  # [B+1] int32
    q_causal_offsets: np.ndarray | None  # [B] int32 or None (bottom-right alignment)
    top_k: int
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.q_bits.shape[0])

    @property
    def Tkv(self) -> int:
        return int(self.k_bits.shape[0])

    @property
    def H(self) -> int:
        return int(self.q_bits.shape[1])

    @property
    def D(self) -> int:
        return int(self.q_bits.shape[2])

    @property
    def num_segments(self) -> int:
        return int(len(self.cu_seqlens_q) - 1)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    flat = out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat.size, step):  # chunked to bound peak host memory
        n = min(step, flat.size - i)
        flat[i:i + n] = f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32))
    return out


def _int_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    vals = rng.integers(-2, 3, size=shape, dtype=np.int8).astype(np.float32)
    return f32_to_bf16_bits(vals)


def draw(T, Tkv, cu_seqlens_q, cu_seqlens_k, top_k, *, q_causal_offsets=None, seed=0, kind="normal",
         w_dist="normal8", H=H_HEADS, D=D_HEAD, name="custom") -> Workload:
    """Draw one workload. kind: "normal" or "int"; w_dist: "normal8" (N(0,1)/8) or "uniform" (U(-1,1))."""
    rq = np.random.Generator(np.random.PCG64(seed))
    rk = np.random.Generator(np.random.PCG64(seed + 1))
    rw = np.random.Generator(np.random.PCG64(seed + 2))
    if kind == "normal":
        q = _normal_bf16(rq, (T, H, D))
        k = _normal_bf16(rk, (Tkv, D))
        if w_dist == "normal8":
            w = (rw.standard_normal((T, H), dtype=np.float32) / np.float32(8.0)).astype(np.float32)
        elif w_dist == "uniform":
            w = rw.uniform(-1.0, 1.0, size=(T, H)).astype(np.float32)
        else:
            raise ValueError(f"unknown w_dist {w_dist!r}")
    elif kind == "int":
        q = _int_bf16(rq, (T, H, D))
        k = _int_bf16(rk, (Tkv, D))
        choices = np.array([-1.0, 0.5, 1.0, 2.0], np.float32)
        w = choices[rw.integers(0, 4, size=(T, H))]
    else:
        raise ValueError(f"unknown kind {kind!r}")
    offs = None if q_causal_offsets is None else np.asarray(q_causal_offsets, np.int32)
    return Workload(name=name, q_bits=q, k_bits=k, w=np.ascontiguousarray(w, np.float32),
                    cu_seqlens_q=np.asarray(cu_seqlens_q, np.int32), cu_seqlens_k=np.asarray(cu_seqlens_k, np.int32),
                    q_causal_offsets=offs, top_k=int(top_k), meta={"seed": seed, "kind": kind, "w_dist": w_dist})


def cp_rank0_layout(doc_lens, cp=16):
    """Packed-varlen layout of context-parallel rank 0 under a zigzag split: every document
    of length L is cut into 2 * cp chunks of L / (2 cp) tokens and rank 0 holds the first
    and the last chunk of each.

    Each query segment has its own key segment: the first chunk sees the document's first
    chunk of keys (offset 0), the last chunk sees all L keys (offset L - chunk, the
    bottom-right default)."""
    tq, tk = [], []
    for L in doc_lens:
        chunk = L // (2 * cp)
        assert chunk * 2 * cp == L, "document length must split into 2 * cp equal chunks"
        tq += [chunk, chunk]
        tk += [chunk, L]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    return cu_q, cu_k


def z2_layout(n_docs=8, doc_len=32768):
    """Z2cp: 8 documents of 32768 tokens at CP16 (1024-query chunks): T = 16384, Tkv = 270336."""
    return cp_rank0_layout([doc_len] * n_docs)


# Z3cp ("packed 4k-64k documents, CP16 zigzag rank 0", T = 10624, Tkv = 175296). The page
# gives the totals but not the document mix. Rank 0 holds L/16 queries and L/32 + L keys of
# a document of length L, so T = sum(L)/16 and Tkv = 33 sum(L)/32, and both totals give
# sum(L) = 169984. These eight lengths, 4k to 50k and multiples of 1024, have that sum.
Z3_DOCS = (4096, 8192, 12288, 16384, 20480, 24576, 32768, 51200)


# name -> (T, Tkv, cu_q, cu_k, offsets, top_k, w_dist, description)
def config(name: str):
    if name == "tiny":
        return dict(T=512, Tkv=512, cu_seqlens_q=[0, 512], cu_seqlens_k=[0, 512], top_k=128, w_dist="uniform",
                    q_causal_offsets=None, desc="tiny single causal document N=512, top_k=128")
    if name == "S1":
        return dict(T=8192, Tkv=8192, cu_seqlens_q=[0, 8192], cu_seqlens_k=[0, 8192], top_k=2048,
                    w_dist="normal8", q_causal_offsets=None, desc="single causal document N=8192, top_k=2048")
    if name == "S2":
        return dict(T=16384, Tkv=16384, cu_seqlens_q=[0, 16384], cu_seqlens_k=[0, 16384], top_k=2048,
                    w_dist="normal8", q_causal_offsets=None, desc="single causal document N=16384, top_k=2048")
    if name == "C1":
        return dict(T=4096, Tkv=65536, cu_seqlens_q=[0, 4096], cu_seqlens_k=[0, 65536], top_k=2048,
                    w_dist="normal8", q_causal_offsets=[61440],
                    desc="CP tail: 4096 queries at positions 61440..65535 of a 65536-key document, top_k=2048")
    if name == "Z2":
        cu_q, cu_k = z2_layout()
        return dict(T=int(cu_q[-1]), Tkv=int(cu_k[-1]), cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, top_k=2048,
                    w_dist="normal8", q_causal_offsets=None,
                    desc="packed 8 x 32k documents, first and last 1024-query chunk of each (16 segments), top_k=2048")
    if name == "Z3":
        cu_q, cu_k = cp_rank0_layout(Z3_DOCS)
        return dict(T=int(cu_q[-1]), Tkv=int(cu_k[-1]), cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, top_k=2048,
                    w_dist="normal8", q_causal_offsets=None,
                    desc="packed 4k-50k documents at CP16 zigzag rank 0 (16 segments), top_k=2048")
    if name in SPLIT_TAIL:
        tkv = SPLIT_TAIL[name]
        return dict(T=4, Tkv=tkv, cu_seqlens_q=[0, 4], cu_seqlens_k=[0, tkv], top_k=2048, w_dist="normal8",
                    q_causal_offsets=None, desc=f"split tail: the last 4 queries of a {tkv}-key document, top_k=2048")
    raise KeyError(name)


# split-tail rows: 4 queries at the end of one document (bottom-right offsets)
SPLIT_TAIL = {"A1": 22018, "A2": 30466, "A3": 41986}

CONFIG_NAMES = ("tiny", "S1", "S2", "C1", "Z2", "Z3", "A1", "A2", "A3")


def make(name: str, kind: str = "normal", seed: int = 0) -> Workload:
    c = config(name)
    return draw(c["T"], c["Tkv"], c["cu_seqlens_q"], c["cu_seqlens_k"], c["top_k"], q_causal_offsets=c["q_causal_offsets"],
                seed=seed, kind=kind, w_dist=c["w_dist"], name=name)
