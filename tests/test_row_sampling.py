"""The full-size parity tests compare a sample of rows with the oracle; the sample must
reach every kind of work unit the scan runs on that configuration (host logic only)."""
from types import SimpleNamespace

import numpy as np

from deterministic_top_key_gb300 import inputs
from tests.test_gpu_full_configs import _row_visible, _sample_rows


def _layout(name):
    c = inputs.config(name)
    offs = None if c["q_causal_offsets"] is None else np.asarray(c["q_causal_offsets"], np.int32)
    cu_q = np.asarray(c["cu_seqlens_q"], np.int32)
    return SimpleNamespace(T=c["T"], cu_seqlens_q=cu_q, cu_seqlens_k=np.asarray(c["cu_seqlens_k"], np.int32),
                           q_causal_offsets=offs, num_segments=len(cu_q) - 1)


def test_sampled_rows_cover_every_unit_kind():
    # kinds: at most 4096 visible keys (direct), at most 16384 (dense), more (filtered)
    for name, kinds in (("S1", 2), ("S2", 2), ("C1", 1), ("Z2", 2), ("Z3", 3)):
        wl = _layout(name)
        _, vis = _row_visible(wl)
        rows = _sample_rows(wl)
        assert len(rows) >= 512 and len(np.unique(rows)) == len(rows)
        v = vis[rows]
        got = int((v <= 4096).any()) + int(((v > 4096) & (v <= 16384)).any()) + int((v > 16384).any())
        assert got == kinds, (name, got)
        for b in range(wl.num_segments):  # first and last query of every segment
            q0, q1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
            assert q0 in rows and q1 - 1 in rows


def test_split_tails_compare_every_row():
    for name in ("A1", "A2", "A3"):
        assert list(_sample_rows(_layout(name))) == [0, 1, 2, 3]
