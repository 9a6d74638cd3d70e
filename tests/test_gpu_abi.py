"""C-ABI behaviour on the GPU: argument errors, ticket-block recovery, stream ordering."""
import numpy as np
import pytest

from deterministic_top_key_gb300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(cuda_lib):
    import torch

    from deterministic_top_key_gb300 import binding

    dev = torch.device("cuda:0")
    wl = inputs.draw(150, 900, [0, 50, 150], [0, 400, 900], 32, seed=21, kind="int")
    q, k, w = parity.to_device(wl, dev)
    import oracle

    ref = oracle.topk(parity.oracle_problem(wl))
    return binding, torch, dev, wl, (q, k, w), ref


def _bufs(torch, dev, wl):
    ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    return ids, sc


def test_argument_errors(env):
    binding, torch, dev, wl, (q, k, w), _ = env
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ids, sc = _bufs(torch, dev, wl)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws[: plan.workspace_bytes() // 2])
    assert e.value.status == binding.ITK_ERR_WORKSPACE_TOO_SMALL
    kb = torch.empty(k.numel() + 8, dtype=torch.bfloat16, device=dev)[1:]
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_run(plan, q, kb, w, ids, sc, ws)
    assert e.value.status == binding.ITK_ERR_MISALIGNED
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_run(plan, q, k, None, ids, sc, ws)
    assert e.value.status == binding.ITK_ERR_NULL_POINTER
    # refused by the binding: a strided q and a BF16 w would be read as the wrong layout or type
    for bad in ((q.transpose(1, 2), k, w), (q, k, w.to(torch.bfloat16))):
        with pytest.raises(binding.IndexerTopkError) as e:
            binding.indexer_topk_run(plan, *bad, ids, sc, ws)
        assert e.value.status == binding.ITK_ERR_INVALID_ARGUMENT
    plan.destroy()
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, 4096)
    assert e.value.status == binding.ITK_ERR_UNSUPPORTED


def test_recovery_after_failed_launch(env):
    """A poisoned ticket block plus a refused launch: the next run zeroes the block first
    and returns correct rows."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    binding.indexer_topk_debug_inject(plan, 2)  # leave the block nonzero
    binding.indexer_topk_debug_inject(plan, 1)  # next launch is refused
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    assert e.value.status == binding.ITK_ERR_CUDA
    ids.fill_(5)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.device_status()
    # and the block is left at zero again: another run is still correct
    ids.fill_(5)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.destroy()


def test_prepare_and_run_on_ordered_streams(env):
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, stream=s1)
    ev = torch.cuda.Event()
    ev.record(s1)
    s2.wait_event(ev)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    torch.cuda.synchronize()
    for _ in range(3):
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws, stream=s2)
    s2.synchronize()
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.destroy()


def test_empty_query_set(env):
    binding, torch, dev, wl, (q, k, w), _ = env
    plan = binding.indexer_topk_prepare(0, 10, [0, 0], [0, 10], 8)
    assert plan.workspace_bytes() == 0
    e = torch.empty((0, 8), dtype=torch.int32, device=dev)
    binding.indexer_topk_run(plan, q, k, w, e, e.float(), None)
    plan.destroy()


def test_split_event_brackets_the_two_kernels(env):
    """The plan's split event is recorded between the scan and the selection launches."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    s = torch.cuda.current_stream()
    a, mid, b = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    mid.record(s)  # creates the event
    binding.indexer_topk_set_split_event(plan, mid)
    a.record(s)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    b.record(s)
    binding.indexer_topk_set_split_event(plan, None)
    torch.cuda.synchronize()
    t_scan, t_sel, t_all = a.elapsed_time(mid), mid.elapsed_time(b), a.elapsed_time(b)
    assert t_scan > 0 and t_sel > 0 and abs(t_scan + t_sel - t_all) < 1e-3 + 1e-3 * t_all
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.destroy()


def test_cuda_graph_capture_and_replay(env):
    """A prepared run captured into a CUDA graph replays with bit-identical rows: both
    launches take their arguments by value and both ticket blocks reset themselves at the
    end of every run, so each replay starts from zero."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first run outside the capture (kernel attributes, module load)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws, stream=s)
    for _ in range(3):
        ids.fill_(5)
        sc.fill_(0.0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.device_status()
    del g
    plan.destroy()


def test_runs_correct_while_sms_are_held(env):
    """A kernel of another stream holds 32 SMs while the scan runs, with the ticket schedule
    and with the fixed one: the call completes and every row stays exact."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    side = torch.cuda.Stream()
    for what in (4, 3, 4):  # ticket, fixed, ticket again
        binding.indexer_topk_debug_inject(plan, what)
        ids.fill_(5)
        torch.cuda.synchronize()
        binding.indexer_topk_bench_hold(32, 2000, side)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
        torch.cuda.synchronize()
        parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.device_status()
    plan.destroy()
