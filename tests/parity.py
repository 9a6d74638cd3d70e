"""Comparison of the CUDA path's output with the oracle's.

Integer-valued inputs: every FP32 sum in the scan is exact, so ids and scores must be
bit-identical.

Random inputs: both sides select on FP32 scores, but the CUDA path sums in FP32 (tensor
core dot products, then a fixed-order FMA chain over heads) while the oracle sums in
fp64 and rounds once. A score o = I[t,s] of the oracle may differ from the GPU's by

    tol(t,s) = max(RTOL * |o|, B(t,s)),   RTOL = 1e-3,

where B is an upper bound of the FP32 path's own rounding error for that score:

    B(t,s) = g(128, 2^-23) * sum_h |w_h| * sum_d |q_hd * k_sd|
           + g(12, 2^-24)  * sum_h |w_h * x_h|
           + 2^-23 * |o|,                      g(n, u) = n u / (1 - n u).

First term: x_h = q[t,h,:].k[s,:] is a sum of 128 products of BF16 values, each exact in
FP32; in whatever order and grouping the tensor core adds them, each of its at most 128
roundings (to nearest or toward zero) errs by at most 2^-23 of a partial sum of
|products|, so |x^_h - x_h| <= g(128, 2^-23) sum_d |q_hd k_sd|, and ReLU does not enlarge
that difference. Second term: each w_h * ReLU(x_h) passes through at most 8 FMA roundings
and 3 tree additions (round to nearest). Third: the oracle's one rounding to FP32 and the
GPU's last one. RTOL is the relative tolerance asked of the scan; B takes over only where
FP32 itself cannot resolve a score to 1e-3 (cancellation among heads).

Ids may differ only at the selection boundary: where the oracle's k-th and (k+1)-th
scores lie within tolerance of each other, and then only among ids whose oracle scores
lie within it of the k-th score.
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


def _fp32_bound(wl, t, ids, o):
    """B(t, s) of the module docstring for query row t and key rows ids (o: oracle scores)."""
    from deterministic_top_key_gb300 import inputs

    q = inputs.bf16_bits_to_f32(wl.q_bits[t]).astype(np.float64)           # [H, D]
    k = inputs.bf16_bits_to_f32(wl.k_bits[np.asarray(ids)]).astype(np.float64)  # [n, D]
    w = np.abs(wl.w[t].astype(np.float64))                                  # [H]
    D = q.shape[1]
    g = lambda n, u: n * u / (1.0 - n * u)  # noqa: E731
    s_abs = w @ (np.abs(q) @ np.abs(k).T)         # sum_h |w_h| sum_d |q_hd k_sd|
    s_x = w @ np.abs(q @ k.T)                      # sum_h |w_h x_h|
    return g(D, 2.0 ** -23) * s_abs + g(12, 2.0 ** -24) * s_x + 2.0 ** -23 * np.abs(np.asarray(o, np.float64))


def tolerance(wl, t, ids, o):
    """max(RTOL |o|, B(t, s)) for the oracle scores o of the key rows ids of query row t."""
    o = np.asarray(o, np.float64)
    return np.maximum(RTOL * np.abs(o), _fp32_bound(wl, t, ids, o))


def assert_close(g_ids, g_sc, wl, rows, top_k=None, nthreads=0, key_id_base=0):
    """Random-input parity on the listed query rows (g_ids/g_sc are full [T, top_k] arrays;
    returned ids are key_id_base + key row)."""
    top_k = wl.top_k if top_k is None else top_k
    rows = np.asarray(rows, np.int32)
    p1 = oracle_problem(wl, top_k + 1)
    r_ids, r_sc = oracle.topk(p1, rows=rows, nthreads=nthreads)
    p = oracle_problem(wl)
    for li, t in enumerate(rows):
        gi, gs = np.asarray(g_ids[t]), np.asarray(g_sc[t])
        gi = np.where(gi >= 0, gi - key_id_base, gi)
        _, n_vis = oracle.visibility(p, int(t))
        keff = min(top_k, n_vis)
        check_row_format(gi, gs, keff)
        ri, rs = r_ids[li, :keff], r_sc[li, :keff]
        # every returned score against the oracle's score of the same id
        o_of_g = oracle.scores(p, np.full(keff, t, np.int32), gi[:keff], nthreads=nthreads)
        err = np.abs(gs[:keff].astype(np.float64) - o_of_g)
        tol_g = tolerance(wl, t, gi[:keff], o_of_g)
        assert np.all(err <= tol_g), f"row {t}: score error {err.max()} beyond tolerance"
        # position-wise scores
        tol_r = tolerance(wl, t, ri, rs)
        assert np.all(np.abs(gs[:keff].astype(np.float64) - rs) <= tol_r), \
            f"row {t}: ranked scores differ beyond tolerance"
        # set agreement except at a near-tie boundary
        gset, rset = set(gi[:keff].tolist()), set(ri.tolist())
        if gset != rset:
            assert keff == top_k and n_vis > top_k, f"row {t}: id sets differ with no boundary"
            s_k, s_k1 = float(r_sc[li, keff - 1]), float(r_sc[li, keff])
            tk = float(tolerance(wl, t, r_ids[li, keff - 1:keff + 1], r_sc[li, keff - 1:keff + 1]).max())
            assert abs(s_k - s_k1) <= tk, f"row {t}: ids differ but k-th/(k+1)-th scores are apart"
            diff = np.array(sorted(gset ^ rset), np.int32)
            o = oracle.scores(p, np.full(len(diff), t, np.int32), diff, nthreads=nthreads)
            tol_d = np.maximum(tolerance(wl, t, diff, o), tk)
            assert np.all(np.abs(o - s_k) <= tol_d), f"row {t}: a differing id is not at the boundary"
