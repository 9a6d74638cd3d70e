"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Contract (flashinfer PR #8691, opening description): BF16 q/k, FP32 w and
scores, top-k key ids per query, ties to the larger id, results independent of
partition or chunking. Score form: the lightning-indexer sum over heads of
w * ReLU(q . k).

Each pin is chosen so that a plausible slip in the oracle (a dropped ReLU, a
swapped w index, a transposed q or k, an off-by-one causal bound, a reversed
tie-break, a wrong fill value or order) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from deterministic_top_key_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(oracle_mod, q, k, w, cu_q, cu_k, top_k, offsets=None):
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    return oracle_mod.Problem(inputs.f32_to_bf16_bits(q), inputs.f32_to_bf16_bits(k), np.asarray(w, np.float32),
                              cu_q, cu_k, top_k, offsets)


def _to_float(v):
    return -math.inf if v == "-inf" else float(v)


def test_worked_example(oracle_mod):
    """Hand-derived example in tests/golden/worked_example.json (values worked out by hand)."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    p = _problem(oracle_mod, g["q"], g["k"], g["w"], g["cu_seqlens_q"], g["cu_seqlens_k"], g["top_k"],
                 g["q_causal_offsets"])
    ids, sc = oracle_mod.topk(p)
    np.testing.assert_array_equal(ids, np.array(g["expected_ids"], np.int32))
    exp = np.array([[_to_float(v) for v in row] for row in g["expected_scores"]], np.float32)
    np.testing.assert_array_equal(sc, exp)
    # the zero score of query 3 is +0.0, not -0.0
    assert not np.signbit(sc[3, 0])
    bi, bs = oracle_mod.bruteforce(p)
    np.testing.assert_array_equal(bi, ids)
    np.testing.assert_array_equal(bs, sc)


def test_unit_vector_closed_form(oracle_mod):
    """H=1, w=1, q_t = e_a(t), k_s = e_b(s): the score is 1 if a(t) == b(s) else 0.

    Expected rows: the visible keys with b(s) == a(t) in descending id order, then the
    other visible keys in descending id order, then the fill."""
    D, T, top_k = 8, 24, 40
    rng = np.random.default_rng(5)
    a = rng.integers(0, D, size=T)
    b = rng.integers(0, D, size=T)
    q = np.zeros((T, 1, D), np.float32)
    q[np.arange(T), 0, a] = 1.0
    k = np.zeros((T, D), np.float32)
    k[np.arange(T), b] = 1.0
    w = np.ones((T, 1), np.float32)
    p = _problem(oracle_mod, q, k, w, [0, T], [0, T], top_k)
    ids, sc = oracle_mod.topk(p)
    for t in range(T):
        vis = np.arange(t + 1)
        hit = [s for s in vis[::-1] if b[s] == a[t]]
        miss = [s for s in vis[::-1] if b[s] != a[t]]
        exp_ids = hit + miss + [-1] * (top_k - t - 1)
        exp_sc = [1.0] * len(hit) + [0.0] * len(miss) + [-math.inf] * (top_k - t - 1)
        np.testing.assert_array_equal(ids[t], exp_ids)
        np.testing.assert_array_equal(sc[t], np.array(exp_sc, np.float32))


def test_all_scores_zero_gives_largest_ids(oracle_mod):
    """q >= 0 and k <= 0 make every dot product <= 0, so every score is +0.0 and the
    tie-break alone orders the row: the k_eff largest visible ids, descending."""
    rng = np.random.default_rng(1)
    T, H, D, top_k = 40, 4, 16, 7
    q = np.abs(rng.standard_normal((T, H, D))).astype(np.float32)
    k = -np.abs(rng.standard_normal((T, D))).astype(np.float32)
    w = rng.standard_normal((T, H)).astype(np.float32)
    p = _problem(oracle_mod, q, k, w, [0, T], [0, T], top_k)
    ids, sc = oracle_mod.topk(p)
    for t in range(T):
        keff = min(top_k, t + 1)
        np.testing.assert_array_equal(ids[t, :keff], np.arange(t, t - keff, -1))
        assert np.all(sc[t, :keff] == 0.0) and not np.any(np.signbit(sc[t, :keff]))
        assert np.all(ids[t, keff:] == -1) and np.all(np.isneginf(sc[t, keff:]))


def test_negative_weights_only_give_nonpositive_scores(oracle_mod):
    """w < 0 everywhere: each term w*ReLU(.) is <= 0, so the best key is one whose heads
    all have non-positive dot products (score 0) if any, and no score exceeds 0."""
    rng = np.random.default_rng(2)
    T, H, D = 30, 3, 8
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = rng.standard_normal((T, D)).astype(np.float32)
    w = -np.abs(rng.standard_normal((T, H))).astype(np.float32) - 0.1
    p = _problem(oracle_mod, q, k, w, [0, T], [0, T], T)
    ids, sc = oracle_mod.topk(p)
    valid = ids >= 0
    assert np.all(sc[valid] <= 0.0)


def test_causal_counts_and_offsets(oracle_mod):
    """Query i of a segment with offset off sees exactly off+i+1 keys, all inside its own segment."""
    rng = np.random.default_rng(3)
    tq = [3, 5, 4]
    tk = [7, 5, 9]
    offs = [2, 0, 5]
    cu_q = np.concatenate([[0], np.cumsum(tq)])
    cu_k = np.concatenate([[0], np.cumsum(tk)])
    T, Tkv, H, D = int(cu_q[-1]), int(cu_k[-1]), 2, 4
    q = rng.standard_normal((T, H, D)).astype(np.float32)
    k = rng.standard_normal((Tkv, D)).astype(np.float32)
    w = rng.standard_normal((T, H)).astype(np.float32)
    top_k = 16
    p = _problem(oracle_mod, q, k, w, cu_q, cu_k, top_k, offs)
    ids, _ = oracle_mod.topk(p)
    for b in range(3):
        for i in range(tq[b]):
            t = cu_q[b] + i
            n_vis = offs[b] + i + 1
            got = ids[t][ids[t] >= 0]
            assert len(got) == min(top_k, n_vis)
            assert set(got.tolist()) == set(range(cu_k[b], cu_k[b] + n_vis))
            assert oracle_mod.visibility(p, t) == (cu_k[b], n_vis)


def test_default_offset_is_bottom_right(oracle_mod):
    """Without offsets, segment b's queries end at its last key: off_b = Tk_b - Tq_b."""
    rng = np.random.default_rng(4)
    tq, tk = [2, 3], [6, 3]
    cu_q = np.concatenate([[0], np.cumsum(tq)])
    cu_k = np.concatenate([[0], np.cumsum(tk)])
    q = rng.standard_normal((5, 2, 4)).astype(np.float32)
    k = rng.standard_normal((9, 4)).astype(np.float32)
    w = rng.standard_normal((5, 2)).astype(np.float32)
    p0 = _problem(oracle_mod, q, k, w, cu_q, cu_k, 8)
    p1 = _problem(oracle_mod, q, k, w, cu_q, cu_k, 8, [4, 0])
    for a, b in zip(oracle_mod.topk(p0), oracle_mod.topk(p1)):
        np.testing.assert_array_equal(a, b)
    assert oracle_mod.visibility(p0, 1) == (0, 6)
    assert oracle_mod.visibility(p0, 2) == (6, 1)


def test_invalid_offsets_rejected(oracle_mod):
    q = np.zeros((2, 1, 2), np.float32)
    k = np.zeros((3, 2), np.float32)
    w = np.ones((2, 1), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.topk(_problem(oracle_mod, q, k, w, [0, 2], [0, 3], 2, [2]))  # 2 + 2 > 3
    with pytest.raises(ValueError):
        oracle_mod.topk(_problem(oracle_mod, q, k, w, [0, 2], [0, 3], 2, [-1]))
    with pytest.raises(ValueError):
        oracle_mod.topk(_problem(oracle_mod, q, np.zeros((1, 2)), w, [0, 2], [0, 1], 2))  # Tq > Tk, default offset < 0


@pytest.mark.parametrize("kind", ["normal", "int"])
def test_sort_path_matches_bruteforce(oracle_mod, kind):
    """The sort path and the rank-counting path select and order identically."""
    w_dist = "uniform"
    wl = inputs.draw(37, 53, [0, 12, 12, 37], [0, 20, 23, 53], 9, q_causal_offsets=[3, 0, 5], seed=11, kind=kind,
                     w_dist=w_dist, H=5, D=12)
    p = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k,
                           wl.q_causal_offsets)
    a = oracle_mod.topk(p)
    b = oracle_mod.bruteforce(p)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_top_k_at_least_visible_returns_every_visible_key(oracle_mod):
    wl = inputs.draw(20, 20, [0, 20], [0, 20], 64, seed=3, kind="normal", w_dist="uniform", H=3, D=8)
    p = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ids, sc = oracle_mod.topk(p)
    for t in range(20):
        assert sorted(ids[t, : t + 1].tolist()) == list(range(t + 1))
        assert np.all(ids[t, t + 1:] == -1)
        # descending by score, equal scores by descending id
        s, i = sc[t, : t + 1], ids[t, : t + 1]
        for j in range(t):
            assert s[j] > s[j + 1] or (s[j] == s[j + 1] and i[j] > i[j + 1])


def test_integer_inputs_are_exact(oracle_mod):
    """Integer q, k in [-2,2] and w in {-1,0.5,1,2}: every score is a multiple of 0.5 and
    equals the exact integer arithmetic value (int64 dot products, doubled weights)."""
    wl = inputs.draw(16, 16, [0, 16], [0, 16], 16, seed=7, kind="int", H=64, D=128)
    p = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ids, sc = oracle_mod.topk(p)
    qi = inputs.bf16_bits_to_f32(wl.q_bits).astype(np.int64)
    ki = inputs.bf16_bits_to_f32(wl.k_bits).astype(np.int64)
    w2 = (wl.w * 2).astype(np.int64)  # exact: w in {-1, .5, 1, 2}
    for t in range(16):
        for j in range(t + 1):
            s = ids[t, j]
            dots = qi[t] @ ki[s]
            twice = int(np.sum(w2[t] * np.maximum(dots, 0)))
            assert sc[t, j] * 2 == twice
    assert np.all(np.mod(sc[ids >= 0] * 2, 1) == 0)


def test_weight_scaling_is_exact(oracle_mod):
    """Doubling w doubles every score exactly and keeps every id."""
    wl = inputs.draw(30, 30, [0, 30], [0, 30], 10, seed=9, kind="normal", w_dist="uniform", H=4, D=16)
    p1 = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    p2 = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w * 2, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    i1, s1 = oracle_mod.topk(p1)
    i2, s2 = oracle_mod.topk(p2)
    np.testing.assert_array_equal(i1, i2)
    np.testing.assert_array_equal(s1 * 2, s2)


def test_rechunking_invariance(oracle_mod):
    """Splitting a segment's queries into two chunks (each with its own copy of the keys and
    the matching causal offset) leaves every row unchanged up to the id shift of the copy."""
    wl = inputs.draw(24, 30, [0, 24], [0, 30], 12, seed=13, kind="normal", w_dist="uniform", H=3, D=8)
    base = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, [0, 24], [0, 30], 12)  # offset 6
    ids0, sc0 = oracle_mod.topk(base)
    k2 = np.concatenate([wl.k_bits, wl.k_bits])
    split = oracle_mod.Problem(wl.q_bits, k2, wl.w, [0, 10, 24], [0, 30, 60], 12, [6, 16])
    ids1, sc1 = oracle_mod.topk(split)
    np.testing.assert_array_equal(sc0, sc1)
    np.testing.assert_array_equal(ids0[:10], ids1[:10])
    shifted = np.where(ids1[10:] >= 0, ids1[10:] - 30, -1)
    np.testing.assert_array_equal(ids0[10:], shifted)


def test_segments_are_independent(oracle_mod):
    """Concatenating two problems as two segments reproduces each problem's rows."""
    a = inputs.draw(9, 14, [0, 9], [0, 14], 6, seed=21, kind="int", H=2, D=8)
    b = inputs.draw(7, 7, [0, 7], [0, 7], 6, seed=22, kind="int", H=2, D=8)
    pa = oracle_mod.Problem(a.q_bits, a.k_bits, a.w, [0, 9], [0, 14], 6)
    pb = oracle_mod.Problem(b.q_bits, b.k_bits, b.w, [0, 7], [0, 7], 6)
    pab = oracle_mod.Problem(np.concatenate([a.q_bits, b.q_bits]), np.concatenate([a.k_bits, b.k_bits]),
                             np.concatenate([a.w, b.w]), [0, 9, 16], [0, 14, 21], 6)
    ia, sa = oracle_mod.topk(pa)
    ib, sb = oracle_mod.topk(pb)
    iab, sab = oracle_mod.topk(pab)
    np.testing.assert_array_equal(iab[:9], ia)
    np.testing.assert_array_equal(sab[:9], sa)
    np.testing.assert_array_equal(np.where(iab[9:] >= 0, iab[9:] - 14, -1), ib)
    np.testing.assert_array_equal(sab[9:], sb)


def test_row_subset_matches_full(oracle_mod):
    wl = inputs.draw(40, 40, [0, 40], [0, 40], 8, seed=4, kind="normal", w_dist="uniform", H=2, D=8)
    p = oracle_mod.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ids, sc = oracle_mod.topk(p)
    rows = np.array([39, 0, 17, 17, 5], np.int32)
    ri, rs = oracle_mod.topk(p, rows=rows)
    np.testing.assert_array_equal(ri, ids[rows])
    np.testing.assert_array_equal(rs, sc[rows])
    s = oracle_mod.scores(p, np.full(3, 39), ids[39, :3])
    np.testing.assert_array_equal(s, sc[39, :3])
