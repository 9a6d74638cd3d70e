"""CUDA path vs oracle, through the C ABI, on small and ragged cases."""
import numpy as np
import pytest

from deterministic_top_key_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def run_plan(binding, wl, dev, top_k=None, runs=1):
    import torch

    q, k, w = parity.to_device(wl, dev)
    top_k = wl.top_k if top_k is None else top_k
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, top_k, wl.q_causal_offsets)
    ws = torch.empty(max(plan.workspace_bytes(), 1), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(runs):
        ids = torch.full((wl.T, top_k), 7, dtype=torch.int32, device=dev)
        sc = torch.full((wl.T, top_k), 7.0, dtype=torch.float32, device=dev)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
        outs.append((ids, sc))
    torch.cuda.synchronize()
    plan.device_status()
    plan.destroy()
    res = [(i.cpu().numpy(), s.cpu().numpy()) for i, s in outs]
    return res if runs > 1 else res[0]


@pytest.fixture(scope="module")
def dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def binding(cuda_lib):
    from deterministic_top_key_gb300 import binding as b

    return b


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_integer_bit_exact(binding, dev, oracle_mod, seed):
    wl = inputs.make("tiny", kind="int", seed=seed)
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_random_within_tolerance(binding, dev, oracle_mod, seed):
    wl = inputs.make("tiny", seed=seed)
    ids, sc = run_plan(binding, wl, dev)
    parity.assert_close(ids, sc, wl, np.arange(wl.T))


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_ragged_segments(binding, dev, oracle_mod, kind):
    # segment sizes leave partial query blocks (nq < 4) and partial key tiles; one empty
    # query segment; explicit offsets that are neither 0 nor bottom-right
    tq = [1, 6, 0, 130, 67, 2]
    tk = [5, 6, 3, 333, 67, 900]
    offs = [4, 0, 1, 200, 0, 897]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    wl = inputs.draw(int(cu_q[-1]), int(cu_k[-1]) + 37, cu_q, cu_k, 96, q_causal_offsets=offs, seed=5, kind=kind,
                     w_dist="uniform")
    ids, sc = run_plan(binding, wl, dev)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
        parity.assert_exact(ids, sc, r_ids, r_sc)
    else:
        parity.assert_close(ids, sc, wl, np.arange(wl.T))


def test_default_offsets_bottom_right(binding, dev, oracle_mod):
    tq, tk = [50, 9, 128], [300, 9, 129]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    wl = inputs.draw(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, 40, seed=8, kind="int")
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


def test_weights_down_to_two_to_the_minus_125_are_exact(binding, dev, oracle_mod):
    """The epilogue multiplies w / 2 by x + |x|; halving is exact for |w| >= 2^-125, so
    integer q and k with weights in {0, +-2^-125, +-2^-124} (every product and sum an exact
    multiple of 2^-125 below 2^-100) give the oracle's bits."""
    wl = inputs.draw(300, 700, [0, 300], [0, 700], 200, seed=41, kind="int")
    rng = np.random.default_rng(41)
    tiny = np.float32(2.0 ** -125)
    w = (rng.choice(np.array([-2, -1, 0, 1, 2], np.float32), size=wl.w.shape) * tiny).astype(np.float32)
    wl = inputs.Workload("tiny-w", wl.q_bits, wl.k_bits, w, wl.cu_seqlens_q, wl.cu_seqlens_k, None, wl.top_k)
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


@pytest.mark.parametrize("top_k", [1, 3, 128, 2048])
def test_top_k_values(binding, dev, oracle_mod, top_k):
    wl = inputs.draw(70, 2100, [0, 70], [0, 2100], top_k, seed=2, kind="int")
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


def _monotone_problem(n_keys, T, direction, top_k):
    """Scores strictly monotone in the key id (every key enters the candidate buffer when
    increasing), or all equal (direction 0: pure tie-break)."""
    H, D = 64, 128
    q = np.zeros((T, H, D), np.float32)
    q[:, :, 0] = 1.0
    k = np.zeros((n_keys, D), np.float32)
    if direction == 0:
        k[:, 0] = 1.0
    else:
        # distinct positive BF16 values, monotone in the row index
        base = np.arange(n_keys, dtype=np.uint32) + np.uint32(0x3F80)
        vals = (base << np.uint32(16)).view(np.float32)
        k[:, 0] = vals if direction > 0 else vals[::-1]
    w = np.ones((T, H), np.float32)
    wl = inputs.Workload("monotone", inputs.f32_to_bf16_bits(q), inputs.f32_to_bf16_bits(k), w,
                         np.array([0, T], np.int32), np.array([0, n_keys], np.int32), None, top_k)
    return wl


@pytest.mark.parametrize("direction", [1, -1, 0])
def test_monotone_and_tied_scores(binding, dev, oracle_mod, direction):
    """Increasing scores and all-equal scores insert every key and force many compactions."""
    wl = _monotone_problem(9000, 9, direction, 2048)
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


@pytest.mark.parametrize("direction", [1, -1, 0])
def test_monotone_and_tied_scores_on_a_split_tail(binding, dev, oracle_mod, direction):
    """Four queries over 9000 keys run as a split tail (18 units). With all-equal scores
    every key lands in one score bin, so the merge narrows its threshold over several
    digit levels, down to the key ids; monotone scores keep every key of a chunk."""
    wl = _monotone_problem(9000, 4, direction, 2048)
    assert len(binding.indexer_topk_unit_table(binding.Desc(4, 9000, [0, 4], [0, 9000], 2048))) > 2
    ids, sc = run_plan(binding, wl, dev)
    r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids, sc, r_ids, r_sc)


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_direct_store_boundary(binding, dev, oracle_mod, kind):
    """Query blocks whose queries see at most 4096 keys append every visible key straight
    to the store; one more visible key takes the filtered path. Segments with 4093-4096,
    4094-4097 and 3-6 visible keys sit beside a 260-query segment (so nothing is split)."""
    tq = [4, 4, 4, 260]
    tk = [4096, 4097, 6, 300]
    offs = [4092, 4093, 2, 40]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    wl = inputs.draw(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, 2048, q_causal_offsets=offs, seed=31, kind=kind)
    units = binding.indexer_topk_unit_table(binding.Desc(wl.T, wl.Tkv, cu_q, cu_k, 2048, offs))
    assert len(units) == 3 + 65 and (units[:, 4] == 0).all()  # one unit per query block
    ids, sc = run_plan(binding, wl, dev)
    rows = np.arange(12)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl), rows=rows.astype(np.int32))
        parity.assert_exact(ids, sc, r_ids, r_sc, rows=rows)
    else:
        parity.assert_close(ids, sc, wl, rows)


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_filtered_unit_boundary(binding, dev, oracle_mod, kind):
    """A query block whose last query sees 16385 keys is filtered: its first 128 tiles go
    to positional slots, then it compacts and filters. Its first three queries see
    16382-16384 keys, so their positional prefix ends early. Beside it: a block whose
    queries see 16381-16384 keys (no sync points at all), and a 260-query segment so that
    nothing is split."""
    tq = [4, 4, 260]
    tk = [16385, 16384, 300]
    offs = [16381, 16380, 40]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    wl = inputs.draw(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, 2048, q_causal_offsets=offs, seed=37, kind=kind)
    units = binding.indexer_topk_unit_table(binding.Desc(wl.T, wl.Tkv, cu_q, cu_k, 2048, offs))
    assert len(units) == 2 + 65 and (units[:, 4] == 0).all()  # one unit per query block
    ids, sc = run_plan(binding, wl, dev)
    rows = np.arange(8)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl), rows=rows.astype(np.int32))
        parity.assert_exact(ids, sc, r_ids, r_sc, rows=rows)
    else:
        parity.assert_close(ids, sc, wl, rows)


@pytest.mark.parametrize("top_k", [1, 7, 300])
@pytest.mark.parametrize("kind", ["int", "normal"])
def test_small_top_k_in_every_append_mode(binding, dev, oracle_mod, top_k, kind):
    """Small top_k through the three append modes of the scan: query blocks that see at
    most 4096 keys (straight to the store), at most 16384 (positional, no sync points)
    and 20000 (positional prefix, then filtered with sync points and compactions)."""
    tq = [4, 4, 4, 260]
    tk = [3000, 10000, 20000, 300]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    wl = inputs.draw(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, top_k, seed=41, kind=kind)
    assert len(binding.indexer_topk_unit_table(binding.Desc(wl.T, wl.Tkv, cu_q, cu_k, top_k))) == 3 + 65
    ids, sc = run_plan(binding, wl, dev)
    rows = np.arange(12)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl), rows=rows.astype(np.int32))
        parity.assert_exact(ids, sc, r_ids, r_sc, rows=rows)
    else:
        parity.assert_close(ids, sc, wl, rows)


def test_repeat_runs_bit_identical(binding, dev):
    wl = inputs.draw(200, 1500, [0, 200], [0, 1500], 256, seed=4, kind="normal")
    outs = run_plan(binding, wl, dev, runs=3)
    for ids, sc in outs[1:]:
        np.testing.assert_array_equal(ids, outs[0][0])
        np.testing.assert_array_equal(sc.view(np.uint32), outs[0][1].view(np.uint32))


def test_rechunked_rows_bit_identical(binding, dev):
    """Partition independence: the same queries run as one segment or split into two
    segments (second one on a copy of the keys, matching offset) give identical rows."""
    wl = inputs.draw(96, 800, [0, 96], [0, 800], 300, seed=9, kind="normal")
    ids0, sc0 = run_plan(binding, wl, dev)
    k2 = np.concatenate([wl.k_bits, wl.k_bits])
    split = inputs.Workload("split", wl.q_bits, k2, wl.w, np.array([0, 37, 96], np.int32),
                            np.array([0, 800, 1600], np.int32), np.array([704, 741], np.int32), 300)
    ids1, sc1 = run_plan(binding, split, dev)
    np.testing.assert_array_equal(sc0.view(np.uint32), sc1.view(np.uint32))
    np.testing.assert_array_equal(ids0[:37], ids1[:37])
    np.testing.assert_array_equal(ids0[37:], np.where(ids1[37:] >= 0, ids1[37:] - 800, -1))


@pytest.mark.parametrize("kind", ["normal", "int"])
def test_packed_segments_match_each_segment_alone(binding, dev, kind):
    """Segment independence: four problems packed as four segments of one call give each
    problem's rows, with the ids moved by the problem's first key row. The packing changes
    how the work is cut: alone, the 64-query problem over 24000 keys and the 3-query
    problem over 9000 keys are split tails (key-split units finished by the merge); packed
    with the 260-query problem (65 query blocks) nothing is split, and those queries run as
    filtered and dense units finished by the selection."""
    top_k = 300
    parts = [
        inputs.draw(260, 260, [0, 260], [0, 260], top_k, seed=31, kind=kind),  # direct units
        inputs.draw(64, 24000, [0, 64], [0, 24000], top_k, seed=32, kind=kind),  # filtered units
        inputs.draw(3, 9000, [0, 3], [0, 9000], top_k, seed=33, kind=kind),  # one dense unit
        inputs.draw(5, 7000, [0, 5], [0, 7000], top_k, q_causal_offsets=np.array([100], np.int32), seed=34,
                    kind=kind),  # explicit offset: 101-105 visible keys
    ]
    alone = [run_plan(binding, p, dev) for p in parts]
    cu_q = np.concatenate([[0], np.cumsum([p.T for p in parts])]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum([p.Tkv for p in parts])]).astype(np.int32)
    packed = inputs.Workload(
        "packed", np.concatenate([p.q_bits for p in parts]), np.concatenate([p.k_bits for p in parts]),
        np.concatenate([p.w for p in parts]), cu_q, cu_k,
        np.array([p.Tkv - p.T if p.q_causal_offsets is None else int(p.q_causal_offsets[0]) for p in parts],
                 np.int32), top_k)
    def split(wl):  # some query block is scanned by more than one unit
        first_rows = binding.indexer_topk_unit_table(
            binding.Desc(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, top_k, wl.q_causal_offsets))[:, 0]
        return len(np.unique(first_rows)) < len(first_rows)

    assert [split(p) for p in parts] == [False, True, True, False]
    assert not split(packed)
    ids, sc = run_plan(binding, packed, dev)
    for i, (a_ids, a_sc) in enumerate(alone):
        rows = slice(cu_q[i], cu_q[i + 1])
        np.testing.assert_array_equal(sc[rows].view(np.uint32), a_sc.view(np.uint32))
        np.testing.assert_array_equal(np.where(ids[rows] >= 0, ids[rows] - cu_k[i], -1), a_ids)


def test_eager_matches_prepared(binding, dev):
    import torch

    wl = inputs.draw(130, 600, [0, 130], [0, 600], 64, seed=12, kind="normal")
    ids0, sc0 = run_plan(binding, wl, dev)
    q, k, w = parity.to_device(wl, dev)
    ids1, sc1 = binding.indexer_topk(q, k, w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids1.cpu().numpy(), ids0)
    np.testing.assert_array_equal(sc1.cpu().numpy().view(np.uint32), sc0.view(np.uint32))


@pytest.mark.parametrize("kind", ["normal", "int"])
def test_split_tail_matches_unsplit(binding, dev, oracle_mod, kind):
    """Four queries over 5000 keys form a split tail (10 units of about 4 key tiles,
    merged per query); the same four queries inside a descriptor of 66 query blocks run
    as one unit. Rows are bit-identical, and equal to the oracle on integer inputs."""
    tq, tk = [4, 260], [5000, 300]
    cu_q = np.concatenate([[0], np.cumsum(tq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(tk)]).astype(np.int32)
    big = inputs.draw(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, 2048, seed=21, kind=kind)
    assert len(binding.indexer_topk_unit_table(binding.Desc(big.T, big.Tkv, cu_q, cu_k, 2048))) == 66
    small = inputs.Workload("split", big.q_bits[:4], big.k_bits[:5000], big.w[:4], np.array([0, 4], np.int32),
                            np.array([0, 5000], np.int32), None, 2048)
    assert len(binding.indexer_topk_unit_table(binding.Desc(4, 5000, [0, 4], [0, 5000], 2048))) == 10
    ids_b, sc_b = run_plan(binding, big, dev)
    ids_s, sc_s = run_plan(binding, small, dev)
    np.testing.assert_array_equal(ids_s, ids_b[:4])
    np.testing.assert_array_equal(sc_s.view(np.uint32), sc_b[:4].view(np.uint32))
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(small))
        parity.assert_exact(ids_s, sc_s, r_ids, r_sc)
    else:
        parity.assert_close(ids_s, sc_s, small, np.arange(4))


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_split_tail_with_fewer_keys_than_top_k(binding, dev, oracle_mod, kind):
    """Four queries over 1500 keys, top_k 2048: the split tail's merge keeps every key and
    fills the rest of each row."""
    wl = inputs.draw(4, 1500, [0, 4], [0, 1500], 2048, seed=43, kind=kind)
    assert len(binding.indexer_topk_unit_table(binding.Desc(4, 1500, [0, 4], [0, 1500], 2048))) > 1
    ids, sc = run_plan(binding, wl, dev)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
        parity.assert_exact(ids, sc, r_ids, r_sc)
    else:
        parity.assert_close(ids, sc, wl, np.arange(4))
    assert (ids[:, 1500:] == -1).all()


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_split_tail_at_the_chunk_budget(binding, dev, oracle_mod, kind):
    """Four queries over 200000 keys: the one query block is split into the whole budget of
    256 key-range units (6-7 tiles each), and the merge selects each row from 256 candidate
    lists (about 200 K keys per query)."""
    wl = inputs.draw(4, 200000, [0, 4], [0, 200000], 2048, seed=44, kind=kind)
    units = binding.indexer_topk_unit_table(binding.Desc(4, 200000, [0, 4], [0, 200000], 2048))
    assert len(units) == 256 and (units[:, 0] == 0).all()
    ids, sc = run_plan(binding, wl, dev)
    if kind == "int":
        r_ids, r_sc = oracle_mod.topk(parity.oracle_problem(wl))
        parity.assert_exact(ids, sc, r_ids, r_sc)
    else:
        parity.assert_close(ids, sc, wl, np.arange(4))


def test_eager_matches_prepared_on_a_split_tail(binding, dev):
    """The eager entry runs the same launches (the scan, then the merge) for a split tail."""
    import torch

    wl = inputs.draw(8, 7000, [0, 8], [0, 7000], 300, seed=13, kind="normal")
    assert len(binding.indexer_topk_unit_table(binding.Desc(8, 7000, [0, 8], [0, 7000], 300))) > 2
    ids0, sc0 = run_plan(binding, wl, dev)
    q, k, w = parity.to_device(wl, dev)
    ids1, sc1 = binding.indexer_topk(q, k, w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids1.cpu().numpy(), ids0)
    np.testing.assert_array_equal(sc1.cpu().numpy().view(np.uint32), sc0.view(np.uint32))
    parity.assert_close(ids0, sc0, wl, np.arange(8))
