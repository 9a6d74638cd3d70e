"""The entry point that allocates nothing, checked against the prepared entry point and,
on integer inputs, against the oracle.

Some callers cannot call cudaMalloc when they run the scan -- for example a serving
runtime that has already reserved the device memory for its own pool. For them the
library offers indexer_topk_run_noalloc, whose scratch lives in one static device array.
This file is collected last so that a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes
import numpy as np
import pytest

from deterministic_top_key_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(cuda_lib):
    import torch

    from deterministic_top_key_gb300 import binding

    return binding, torch, torch.device("cuda:0")


def _prepared(binding, torch, dev, wl, q, k, w):
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k,
                                        wl.q_causal_offsets)
    ws = torch.empty(max(plan.workspace_bytes(), 1), dtype=torch.uint8, device=dev)
    ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    plan.device_status()
    plan.destroy()
    return ids.cpu().numpy(), sc.cpu().numpy()


def _noalloc(binding, torch, dev, wl, q, k, w):
    desc = binding.Desc(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, wl.q_causal_offsets)
    ids = torch.full((wl.T, wl.top_k), 9, dtype=torch.int32, device=dev)
    sc = torch.full((wl.T, wl.top_k), 9.0, dtype=torch.float32, device=dev)
    binding.indexer_topk_run_noalloc(desc, q, k, w, ids, sc)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


def test_noalloc_matches_prepared_on_two_calls(env):
    binding, torch, dev = env
    # two different problems in a row: the second call must not see the first one's
    # scratch contents (ticket block, unit table, candidate buffers)
    cu_q = np.array([0, 700, 1500], np.int32)
    cu_k = np.array([0, 2600, 4000], np.int32)
    first = inputs.draw(1500, 4000, cu_q, cu_k, 512, q_causal_offsets=[1900, 500], seed=31, kind="normal")
    second = inputs.draw(900, 900, [0, 900], [0, 900], 256, seed=32, kind="int")
    # more than 512 work units: the static candidate store takes them in two launch pairs
    third = inputs.draw(2600, 3000, [0, 1300, 2600], [0, 1500, 3000], 128, seed=33, kind="normal")
    # a split tail: 8 queries over 6000 keys (two blocks of 12 units, then a merge launch)
    fourth = inputs.draw(8, 6000, [0, 8], [0, 6000], 512, seed=34, kind="int")
    for wl in (first, second, third, fourth):
        q, k, w = parity.to_device(wl, dev)
        ref_ids, ref_sc = _prepared(binding, torch, dev, wl, q, k, w)
        got_ids, got_sc = _noalloc(binding, torch, dev, wl, q, k, w)
        # the same kernel on the same inputs: identical bits, well within the tolerance
        # of the random-input parity tests
        parity.assert_exact(got_ids, got_sc, ref_ids, ref_sc)
        binding.indexer_topk_noalloc_device_status()
        if wl.meta["kind"] == "int":  # every FP32 sum exact: bit-identical to the oracle too
            import oracle

            o_ids, o_sc = oracle.topk(parity.oracle_problem(wl))
            parity.assert_exact(got_ids, got_sc, o_ids, o_sc)


def test_noalloc_reports_a_wait_timeout_then_runs_exact(env):
    """A call whose scan CTA 0 withholds a key-tile load with every wait cut to about
    1 ms (test hook): its status reader reports the timeout, which the call itself cannot
    return (its kernels run after it returns), and the next call is exact again."""
    binding, torch, dev = env
    import oracle

    wl = inputs.draw(300, 900, [0, 300], [0, 900], 128, seed=35, kind="int")
    q, k, w = parity.to_device(wl, dev)
    o_ids, o_sc = oracle.topk(parity.oracle_problem(wl))
    binding.indexer_topk_debug_inject(None, 5)
    _noalloc(binding, torch, dev, wl, q, k, w)
    with pytest.raises(binding.IndexerTopkError) as err:
        binding.indexer_topk_noalloc_device_status()
    assert err.value.status == binding.ITK_ERR_DEVICE_TIMEOUT
    binding.indexer_topk_noalloc_device_status()  # reading cleared the word
    for _ in range(2):
        got_ids, got_sc = _noalloc(binding, torch, dev, wl, q, k, w)
        binding.indexer_topk_noalloc_device_status()
        parity.assert_exact(got_ids, got_sc, o_ids, o_sc)


def test_noalloc_rejects_too_many_units(env):
    binding, torch, dev = env
    T = 4 * 65536 + 4  # one work unit past the static scratch's unit table
    desc = binding.Desc(T, T, [0, T], [0, T], 8)
    # through the C entry point itself, with dummy buffers: the unit count is refused
    # before any buffer is read (the binding would refuse buffers this small first)
    e = torch.empty(16, dtype=torch.float32, device=dev)
    p = ctypes.c_void_p(e.data_ptr())
    with pytest.raises(binding.IndexerTopkError) as err:
        binding._check(binding.load().indexer_topk_run_noalloc(desc.ref(), p, p, p, p, p, binding._stream_handle(None)))
    assert err.value.status == binding.ITK_ERR_UNSUPPORTED
    assert "static scratch" in str(err.value)
    assert binding.load().indexer_topk_noalloc_scratch_bytes() > 0
