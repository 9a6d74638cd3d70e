"""Comparison of the CUDA path's output with the oracle's.

Integer-valued inputs: every FP32 sum in the scan is exact, so ids and scores must be
bit-identical.

Random inputs: both sides select on FP32 scores, but the CUDA path sums in FP32 (tensor
core dot products, then a fixed-order FMA chain over heads) while the oracle sums in
fp64 and rounds once. Tolerance on a score o of row r:
    |gpu - o| <= RTOL * max(|o|, mean |o| over row r's returned entries)
with RTOL = 1e-3. Ids may differ only at the selection boundary: where the oracle's
k-th and (k+1)-th scores lie within that tolerance, and then only among ids whose
oracle scores lie within it of the k-th score.
"""
from __future__ import annotations

import numpy as np

import oracle

RTOL = 1e-3


def to_device(wl, device):
    import torch

    q = torch.from_numpy(wl.q_bits.view(np.int16)).view(torch.bfloat16).to(device)
    k = torch.from_numpy(wl.k_bits.view(np.int16)).view(torch.bfloat16).to(device)
    w = torch.from_numpy(wl.w).to(device)
    return q, k, w


def oracle_problem(wl, top_k=None):
    return oracle.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k,
                          wl.top_k if top_k is None else top_k, wl.q_causal_offsets)


def assert_exact(g_ids, g_sc, r_ids, r_sc, rows=None):
    g_ids = np.asarray(g_ids)
    g_sc = np.asarray(g_sc)
    if rows is not None:
        g_ids, g_sc = g_ids[rows], g_sc[rows]
    bad = np.nonzero(np.any(g_ids != r_ids, axis=1) | np.any(g_sc.view(np.uint32) != r_sc.view(np.uint32), axis=1))[0]
    if len(bad):
        i = bad[0]
        raise AssertionError(f"{len(bad)} rows differ; first local row {i}:\n gpu ids {g_ids[i][:12]}\n ref ids "
                             f"{r_ids[i][:12]}\n gpu sc {g_sc[i][:12]}\n ref sc {r_sc[i][:12]}")


def check_row_format(ids, sc, keff):
    """Validity of one returned row: k_eff entries in the total order, then the fill."""
    assert np.all(ids[keff:] == -1), "fill ids must be -1"
    assert np.all(np.isneginf(sc[keff:])), "fill scores must be -inf"
    i, s = ids[:keff], sc[:keff]
    assert np.all(i >= 0)
    assert len(np.unique(i)) == keff, "duplicate ids in a row"
    if keff > 1:
        ok = (s[:-1] > s[1:]) | ((s[:-1] == s[1:]) & (i[:-1] > i[1:]))
        assert np.all(ok), "row is not sorted by (score desc, id desc)"
    assert not np.any(np.signbit(s) & (s == 0)), "-0.0 must be returned as +0.0"


def assert_close(g_ids, g_sc, wl, rows, top_k=None, nthreads=0):
    """Random-input parity on the listed query rows (g_ids/g_sc are full [T, top_k] arrays)."""
    top_k = wl.top_k if top_k is None else top_k
    rows = np.asarray(rows, np.int32)
    p1 = oracle_problem(wl, top_k + 1)
    r_ids, r_sc = oracle.topk(p1, rows=rows, nthreads=nthreads)
    p = oracle_problem(wl)
    for li, t in enumerate(rows):
        gi, gs = np.asarray(g_ids[t]), np.asarray(g_sc[t])
        _, n_vis = oracle.visibility(p, int(t))
        keff = min(top_k, n_vis)
        check_row_format(gi, gs, keff)
        ri, rs = r_ids[li, :keff], r_sc[li, :keff]
        scale = max(float(np.mean(np.abs(rs))), 1e-30)
        tol = lambda o: RTOL * np.maximum(np.abs(o), scale)  # noqa: E731
        # every returned score against the oracle's score of the same id
        o_of_g = oracle.scores(p, np.full(keff, t, np.int32), gi[:keff], nthreads=nthreads)
        err = np.abs(gs[:keff] - o_of_g)
        assert np.all(err <= tol(o_of_g)), f"row {t}: score error {err.max()} beyond tolerance"
        # position-wise scores
        assert np.all(np.abs(gs[:keff] - rs) <= tol(rs)), f"row {t}: ranked scores differ beyond tolerance"
        # set agreement except at a near-tie boundary
        gset, rset = set(gi[:keff].tolist()), set(ri.tolist())
        if gset != rset:
            assert keff == top_k and n_vis > top_k, f"row {t}: id sets differ with no boundary"
            s_k, s_k1 = float(r_sc[li, keff - 1]), float(r_sc[li, keff])
            assert abs(s_k - s_k1) <= tol(s_k), f"row {t}: ids differ but k-th/(k+1)-th scores are apart"
            diff = np.array(sorted(gset ^ rset), np.int32)
            o = oracle.scores(p, np.full(len(diff), t, np.int32), diff, nthreads=nthreads)
            assert np.all(np.abs(o - s_k) <= tol(s_k)), f"row {t}: a differing id is not at the boundary"
