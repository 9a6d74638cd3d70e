"""The random-input tolerance of the parity tests (tests/parity.py) against an FP32
computation of the same scores: an FP32 path summing in the GPU's head order stays inside
the bound B, and an error twice as large as the tolerance is caught."""
import numpy as np

import oracle
from deterministic_top_key_gb300 import inputs
from tests import parity


def _fp32_scores(wl, t, ids):
    """I[t,s] the way an FP32 path computes it: each dot product summed in FP32 (one
    order the tensor core may take), then eight FMA chains over heads h = m, m+8, ...,
    combined by a fixed tree."""
    q = inputs.bf16_bits_to_f32(wl.q_bits[t])            # [H, D] float32
    k = inputs.bf16_bits_to_f32(wl.k_bits[np.asarray(ids)])  # [n, D]
    w = wl.w[t]
    x = np.zeros((q.shape[0], len(ids)), np.float32)
    for d in range(q.shape[1]):  # BF16 x BF16 products are exact in FP32
        x = (x + np.outer(q[:, d], k[:, d]).astype(np.float32)).astype(np.float32)
    r = np.maximum(x, np.float32(0))
    p = np.zeros((8, len(ids)), np.float32)
    for h in range(q.shape[0]):
        m = h % 8
        p[m] = (np.float64(w[h]) * r[h].astype(np.float64) + p[m].astype(np.float64)).astype(np.float32)
    s = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]))
    return (s + np.float32(0)).astype(np.float32)


def test_fp32_path_inside_the_bound_and_planted_error_outside():
    wl = inputs.make("tiny", seed=4)
    p = parity.oracle_problem(wl)
    rows = np.array([3, 40, 200, 511], np.int32)
    ids, sc = oracle.topk(p, rows=rows)
    worst = 0.0
    for li, t in enumerate(rows):
        keff = min(wl.top_k, int(t) + 1)
        i, o = ids[li, :keff], sc[li, :keff].astype(np.float64)
        f = _fp32_scores(wl, t, i).astype(np.float64)
        tol = parity.tolerance(wl, t, i, o)
        worst = max(worst, float(np.max(np.abs(f - o) / tol)))
        assert np.all(np.abs(f - o) <= tol)
        assert np.all(tol >= parity.RTOL * np.abs(o))
        # a score off by twice its tolerance is rejected
        assert not np.any(np.abs((o + 2 * tol) - o) <= tol)
    assert worst < 0.5  # the FP32 path sits well inside the bound


def test_bound_grows_with_cancellation():
    """B is what takes over for a near-zero score: there rel 1e-3 would ask for more than
    FP32 can give, and B is positive and scales with sum_h |w_h| sum_d |q k|."""
    wl = inputs.make("tiny", seed=4)
    t, ids = 300, np.arange(301, dtype=np.int32)
    o = oracle.scores(parity.oracle_problem(wl), np.full(301, t, np.int32), ids).astype(np.float64)
    b = parity._fp32_bound(wl, t, ids, o)
    j = int(np.argmin(np.abs(o)))
    assert b[j] > parity.RTOL * abs(o[j])
    assert np.all(b > 0)
