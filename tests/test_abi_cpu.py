"""The C-ABI library loads on a machine without a GPU, exports every function the public
header declares, and its host-only entry points (validation, unit planning) behave."""
import ctypes

import numpy as np
import pytest

from deterministic_top_key_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    from deterministic_top_key_gb300 import build

    build.build()
    return binding.load()


def test_exports_every_declared_function(lib):
    names = binding.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/indexer_topk.h but not exported"


def test_status_strings_and_version(lib):
    assert lib.indexer_topk_status_string(0) == b"ok"
    assert b"workspace" in lib.indexer_topk_status_string(binding.ITK_ERR_WORKSPACE_TOO_SMALL)
    assert lib.indexer_topk_version().decode().count(".") == 2


def _desc(**kw):
    d = dict(T=10, Tkv=20, cu_seqlens_q=[0, 10], cu_seqlens_k=[0, 20], top_k=8)
    d.update(kw)
    return binding.Desc(**d)


def test_validation(lib):
    assert binding.indexer_topk_validate(_desc()) == 0
    assert binding.indexer_topk_validate(_desc(H=32)) == binding.ITK_ERR_UNSUPPORTED
    assert binding.indexer_topk_validate(_desc(D=64)) == binding.ITK_ERR_UNSUPPORTED
    assert binding.indexer_topk_validate(_desc(top_k=0)) == binding.ITK_ERR_INVALID_ARGUMENT
    assert binding.indexer_topk_validate(_desc(top_k=2049)) == binding.ITK_ERR_UNSUPPORTED
    assert binding.indexer_topk_validate(_desc(cu_seqlens_q=[0, 9])) == binding.ITK_ERR_INVALID_SEQLENS
    assert binding.indexer_topk_validate(_desc(cu_seqlens_q=[1, 10])) == binding.ITK_ERR_INVALID_SEQLENS
    assert binding.indexer_topk_validate(_desc(cu_seqlens_k=[0, 21])) == binding.ITK_ERR_INVALID_SEQLENS
    assert binding.indexer_topk_validate(_desc(q_causal_offsets=[11])) == binding.ITK_ERR_INVALID_OFFSETS
    assert binding.indexer_topk_validate(_desc(q_causal_offsets=[-1])) == binding.ITK_ERR_INVALID_OFFSETS
    assert binding.indexer_topk_validate(_desc(q_causal_offsets=[10])) == 0
    assert binding.indexer_topk_validate(_desc(key_id_base=5)) == 0
    assert binding.indexer_topk_validate(_desc(key_id_base=2**31 - 1 - 20)) == 0  # last id 2^31 - 2
    assert binding.indexer_topk_validate(_desc(key_id_base=2**31 - 20)) == binding.ITK_ERR_INVALID_ARGUMENT
    assert binding.indexer_topk_validate(_desc(key_id_base=-1)) == binding.ITK_ERR_INVALID_ARGUMENT
    assert binding.indexer_topk_validate(
        _desc(T=4, cu_seqlens_q=[0, 4, 2], cu_seqlens_k=[0, 5, 6])) == binding.ITK_ERR_INVALID_SEQLENS
    assert lib.indexer_topk_validate(None) == binding.ITK_ERR_INVALID_ARGUMENT
    assert len(lib.indexer_topk_last_error()) > 0


def _check_unit_table(u, cu_q, cu_k, offs):
    """Every query block appears as consecutive units whose key-tile ranges partition its
    visible tiles [0, ceil((pos0 + nq) / 128)); blocks come longest first."""
    blocks = []  # (q0, nq, tiles)
    covered = np.zeros(int(cu_q[-1]), int)
    i = 0
    while i < len(u):
        q0, nq, k0, pos0, t0, t1 = (int(x) for x in u[i])
        assert 1 <= nq <= 4
        b = int(np.searchsorted(cu_q, q0, side="right") - 1)
        assert k0 == cu_k[b] and q0 + nq <= cu_q[b + 1]
        assert pos0 == offs[b] + (q0 - cu_q[b])
        tiles = (pos0 + nq + 127) // 128
        assert t0 == 0
        end = t1
        j = i + 1
        while j < len(u) and int(u[j][0]) == q0:  # the block's further chunks
            assert int(u[j][4]) == end and int(u[j][5]) > end
            end = int(u[j][5])
            j += 1
        assert end == tiles
        covered[q0:q0 + nq] += 1
        blocks.append((q0, nq, tiles, j - i))
        i = j
    assert np.all(covered == 1)
    tiles = [b[2] for b in blocks]
    assert tiles == sorted(tiles, reverse=True)
    return blocks


def test_unit_table_covers_every_query_once_longest_first(lib):
    tq = [3, 0, 9, 130, 1]
    tk = [10, 2, 9, 4000, 1]
    offs = [7, 0, 0, 3870, 0]
    cu_q = np.concatenate([[0], np.cumsum(tq)])
    cu_k = np.concatenate([[0], np.cumsum(tk)])
    d = binding.Desc(int(cu_q[-1]), int(cu_k[-1]), cu_q, cu_k, 16, offs)
    u = binding.indexer_topk_unit_table(d)
    blocks = _check_unit_table(u, cu_q, cu_k, offs)
    # 38 query blocks: a split tail; the 4000-key blocks (32 tiles) split into 6 chunks
    # (256 // 38 units per block), the short ones stay whole
    assert len(blocks) == 38
    assert all(n == (6 if t >= 8 else 1) for _, _, t, n in blocks)


def test_unit_table_without_split(lib):
    """More than 64 query blocks: one unit per block, covering all its visible tiles."""
    T = 4 * 65
    cu = np.array([0, T], np.int32)
    d = binding.Desc(T, T, cu, cu, 16)
    u = binding.indexer_topk_unit_table(d)
    assert len(u) == 65
    blocks = _check_unit_table(u, cu, cu, [0])
    assert all(n == 1 for *_, n in blocks)


def test_split_tail_chunks(lib):
    """A1: one block of 173 tiles becomes 44 consecutive units of 3-4 tiles."""
    from deterministic_top_key_gb300 import inputs

    c = inputs.config("A1")
    d = binding.Desc(c["T"], c["Tkv"], c["cu_seqlens_q"], c["cu_seqlens_k"], c["top_k"])
    u = binding.indexer_topk_unit_table(d)
    assert len(u) == 44
    sizes = u[:, 5] - u[:, 4]
    assert sizes.min() >= 3 and sizes.max() <= 4 and sizes.sum() == 173


def test_unit_count_for_configs(lib):
    from deterministic_top_key_gb300 import inputs

    for name, n in [("tiny", 128), ("S1", 2048), ("S2", 4096), ("C1", 1024), ("Z2", 4096), ("Z3", 2656),
                    ("A1", 44), ("A2", 60), ("A3", 83)]:
        c = inputs.config(name)
        d = binding.Desc(c["T"], c["Tkv"], c["cu_seqlens_q"], c["cu_seqlens_k"], c["top_k"], c["q_causal_offsets"])
        assert lib.indexer_topk_num_units(d.ref()) == n


def test_host_only_entry_points_reject_null_plan(lib):
    assert lib.indexer_topk_set_split_event(None, None) == binding.ITK_ERR_INVALID_ARGUMENT
    assert lib.indexer_topk_workspace_bytes(None) == 0
    assert lib.indexer_topk_status_string(binding.ITK_ERR_INTERNAL) == b"internal device check failed"


def test_prepare_without_device_fails_cleanly(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    rc = lib.indexer_topk_prepare(_desc().ref(), None, ctypes.byref(h))
    assert rc == binding.ITK_ERR_NO_DEVICE and not h.value
