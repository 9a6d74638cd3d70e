"""Full-size configurations, in the launch configuration the benchmark times.

Every row is checked for validity (sorted by the total order, unique ids inside the
query's visible range, fill after k_eff). Against the oracle: on the integer variant,
every row of every configuration, bit-exact (the oracle takes about 15 s for S1, 55 s for
S2 and Z2, 65 s for Z3 and 110 s for C1 on 16 cores); on random inputs at least 512 rows
per configuration (all rows of the split tails), within tolerance. The sampled rows cover
every kind of work unit the scan runs -- queries that see at most 4096 keys (appended
straight to the store), at most 16384 (positional working buffer, one threshold raise) and
more (filtered with sync points) -- and the first and last query of every segment.
"""
import numpy as np
import pytest

from deterministic_top_key_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu



def _sample_rows(wl, n=512, seed=0):
    """About n rows: the segment edges, then an even share of random rows from each kind
    of unit (by the number of keys the query sees), all rows if T <= n."""
    if wl.T <= n:
        return np.arange(wl.T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    _, vis = _row_visible(wl)
    rows = set()
    for b in range(wl.num_segments):  # segment edges
        q0, q1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
        if q1 > q0:
            rows.update({q0, q1 - 1})
    kinds = [np.nonzero(vis <= 4096)[0], np.nonzero((vis > 4096) & (vis <= 16384))[0], np.nonzero(vis > 16384)[0]]
    kinds = [x for x in kinds if len(x)]
    per = max(1, (n - len(rows)) // len(kinds))
    for x in kinds:
        rows.update(rng.choice(x, size=min(per, len(x)), replace=False).tolist())
    rest = np.setdiff1d(np.arange(wl.T), np.fromiter(rows, np.int64))
    if len(rows) < n:  # top up with rows of any kind
        rows.update(rng.choice(rest, size=min(n - len(rows), len(rest)), replace=False).tolist())
    return np.array(sorted(rows), np.int32)


def _row_visible(wl):
    vis = np.zeros(wl.T, np.int64)
    begin = np.zeros(wl.T, np.int64)
    for b in range(wl.num_segments):
        q0, q1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
        tq, tk = q1 - q0, int(wl.cu_seqlens_k[b + 1] - wl.cu_seqlens_k[b])
        off = int(wl.q_causal_offsets[b]) if wl.q_causal_offsets is not None else tk - tq
        vis[q0:q1] = off + np.arange(tq) + 1
        begin[q0:q1] = wl.cu_seqlens_k[b]
    return begin, vis


def _check_all_rows(ids, sc, wl):
    begin, vis = _row_visible(wl)
    keff = np.minimum(vis, wl.top_k)
    pos = np.arange(wl.top_k)[None, :]
    valid = pos < keff[:, None]
    assert np.all(ids[~valid] == -1) and np.all(np.isneginf(sc[~valid]))
    lo, hi = begin[:, None], (begin + vis)[:, None]
    assert np.all(((ids >= lo) & (ids < hi))[valid]), "an id outside the query's visible keys"
    s0, s1 = sc[:, :-1], sc[:, 1:]
    i0, i1 = ids[:, :-1], ids[:, 1:]
    pair_valid = valid[:, 1:]
    ordered = (s0 > s1) | ((s0 == s1) & (i0 > i1))
    assert np.all(ordered[pair_valid]), "a row is not in (score desc, id desc) order"
    assert not np.any((sc == 0) & np.signbit(sc))
    # ids unique within a row (sorted copy, ignoring fill)
    srt = np.sort(np.where(valid, ids, -1 - pos), axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1])


def _run(wl, dev):
    import torch

    from deterministic_top_key_gb300 import binding

    q, k, w = parity.to_device(wl, dev)
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k,
                                        wl.q_causal_offsets)
    ws = torch.empty(max(plan.workspace_bytes(), 1), dtype=torch.uint8, device=dev)
    ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    ids2 = torch.empty_like(ids)
    sc2 = torch.empty_like(sc)
    binding.indexer_topk_run(plan, q, k, w, ids2, sc2, ws)
    torch.cuda.synchronize()
    plan.device_status()
    assert torch.equal(ids, ids2) and torch.equal(sc.view(torch.int32), sc2.view(torch.int32)), "repeat differs"
    plan.destroy()
    return ids.cpu().numpy(), sc.cpu().numpy()


@pytest.fixture(scope="module")
def dev(cuda_lib):
    import torch

    return torch.device("cuda:0")


@pytest.mark.parametrize("name", ["S1", "S2", "C1", "Z2", "Z3", "A1", "A2", "A3"])
def test_full_config_random(name, dev, oracle_mod):
    wl = inputs.make(name)
    ids, sc = _run(wl, dev)
    _check_all_rows(ids, sc, wl)
    parity.assert_close(ids, sc, wl, _sample_rows(wl))


@pytest.mark.parametrize("name", ["S1", "S2", "C1", "Z2", "Z3", "A1", "A2", "A3"])
def test_full_config_integer(name, dev, oracle_mod):
    wl = inputs.make(name, kind="int")
    ids, sc = _run(wl, dev)
    _check_all_rows(ids, sc, wl)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)
