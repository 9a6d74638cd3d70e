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


@pytest.mark.parametrize("base", [1000, 2**31 - 1 - 900])
def test_key_id_base(env, base):
    """Ids are key_id_base + key row: the prepared and eager entries return the oracle's
    ids shifted by the base (the fill stays -1) and the same scores. The env problem is a
    split tail, so the merge writes these rows; a second problem runs the selection."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    shifted = np.where(r_ids >= 0, r_ids + base, -1)
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, key_id_base=base)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), shifted, r_sc)
    plan.destroy()
    ids2, sc2 = binding.indexer_topk(q, k, w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, key_id_base=base)
    torch.cuda.synchronize()
    parity.assert_exact(ids2.cpu().numpy(), sc2.cpu().numpy(), shifted, r_sc)
    # 300 queries (75 query blocks, no split): the selection kernel writes the rows
    wl2 = inputs.draw(300, 700, [0, 300], [0, 700], 64, seed=22, kind="int")
    q2, k2, w2 = parity.to_device(wl2, dev)
    import oracle

    i2, s2 = oracle.topk(parity.oracle_problem(wl2))
    ids3, sc3 = binding.indexer_topk(q2, k2, w2, wl2.cu_seqlens_q, wl2.cu_seqlens_k, wl2.top_k, key_id_base=base)
    torch.cuda.synchronize()
    parity.assert_exact(ids3.cpu().numpy(), sc3.cpu().numpy(), np.where(i2 >= 0, i2 + base, -1), s2)
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, key_id_base=-1)
    assert e.value.status == binding.ITK_ERR_INVALID_ARGUMENT


def _device_activities(torch, fn):
    """[(kind, name)] of the device activities (kernels, copies, memsets) that fn issues, in
    start order, recorded through the CUPTI activity API."""
    from tests import device_activity

    return device_activity.record(fn, torch.cuda.synchronize)


def _expected_kernels(binding, desc):
    """Kernels of one run of `desc`: the scan, then the merge if some query block is split
    and the selection if some block is whole (the header's contract)."""
    ut = binding.indexer_topk_unit_table(desc)
    _, per_block = np.unique(ut[:, 0], return_counts=True)
    return ["scan"] + (["merge"] if (per_block > 1).any() else []) + (["select"] if (per_block == 1).any() else [])


@pytest.mark.parametrize("shape", ["whole", "split", "mixed"])
def test_launches_per_call(env, shape):
    """A prepared run issues exactly the scan and its finishing kernel(s), the scan first,
    and no copy or memset; an eager call adds one host-to-device copy of its tables before
    them. Counted from the device activities (CUPTI), as the page's eager test counts its
    profiled device activities."""
    binding, torch, dev, *_ = env
    if shape == "whole":    # 75 query blocks: scan + selection
        wl = inputs.draw(300, 700, [0, 300], [0, 700], 64, seed=23, kind="int")
    elif shape == "split":  # 2 query blocks of 3000 keys: scan + merge
        wl = inputs.draw(8, 3000, [0, 8], [0, 3000], 64, seed=24, kind="int")
    else:                   # 3 blocks: one long (split), two short (whole): all three
        wl = inputs.draw(12, 3000, [0, 4, 12], [0, 2900, 3000], 64, seed=25, kind="int")
    desc = binding.Desc(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    want = _expected_kernels(binding, desc)
    assert want == {"whole": ["scan", "select"], "split": ["scan", "merge"],
                    "mixed": ["scan", "merge", "select"]}[shape]
    q, k, w = parity.to_device(wl, dev)
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(max(plan.workspace_bytes(), 1), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)  # first run outside the recording
    acts = _device_activities(torch, lambda: binding.indexer_topk_run(plan, q, k, w, ids, sc, ws))
    assert len(acts) == len(want), acts  # no copy, no memset
    for (what, name), kind in zip(acts, want):
        assert what == "kernel" and f"indexer_topk_{kind}_kernel" in name, acts
    import oracle

    r_ids, r_sc = oracle.topk(parity.oracle_problem(wl))
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.destroy()
    ews = torch.empty(binding.indexer_topk_eager_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    acts = _device_activities(torch, lambda: binding.indexer_topk_eager(desc, q, k, w, ids, sc, ews))
    assert len(acts) == 1 + len(want), acts
    assert acts[0][0] == "memcpy", acts  # the unit table with zeroed ticket blocks
    for (what, name), kind in zip(acts[1:], want):
        assert what == "kernel" and f"indexer_topk_{kind}_kernel" in name, acts
    binding.indexer_topk_eager_device_status(desc, ews)
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)


@pytest.mark.parametrize("shape", ["whole", "split"])
def test_wait_timeout_is_reported_and_the_next_run_is_exact(env, shape):
    """A run in which scan CTA 0 withholds a key-tile load, with every in-kernel wait cut
    to about 1 ms: the waits on that tile run out, the CTA unwinds (copies and tensor-core
    work drained, tensor memory freed), the status word reports the timeout, and the next
    run of the same plan is bit-exact against the oracle."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    if shape == "whole":
        wl = inputs.draw(300, 700, [0, 300], [0, 700], 64, seed=26, kind="int")
        q, k, w = parity.to_device(wl, dev)
        import oracle

        r_ids, r_sc = oracle.topk(parity.oracle_problem(wl))
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(plan.workspace_bytes(), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    plan.device_status()
    binding.indexer_topk_debug_inject(plan, 5)
    binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    with pytest.raises(binding.IndexerTopkError) as e:
        plan.device_status()
    assert e.value.status == binding.ITK_ERR_DEVICE_TIMEOUT
    plan.device_status()  # reading cleared the word
    for _ in range(2):
        ids.fill_(5)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws)
        torch.cuda.synchronize()
        parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
    plan.device_status()
    plan.destroy()


def test_eager_status_reader_reports_a_wait_timeout(env):
    """The eager entry keeps its status word in the caller's workspace; its reader reports a
    call whose scan CTA 0 withholds a key-tile load with waits cut to about 1 ms (test
    hook), and the next eager call with the same workspace is exact again."""
    binding, torch, dev, wl, (q, k, w), (r_ids, r_sc) = env
    desc = binding.Desc(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k)
    ws = torch.empty(binding.indexer_topk_eager_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    ids, sc = _bufs(torch, dev, wl)
    binding.indexer_topk_debug_inject(None, 5)
    binding.indexer_topk_eager(desc, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    with pytest.raises(binding.IndexerTopkError) as e:
        binding.indexer_topk_eager_device_status(desc, ws)
    assert e.value.status == binding.ITK_ERR_DEVICE_TIMEOUT
    binding.indexer_topk_eager_device_status(desc, ws)  # reading cleared the word
    ids.fill_(5)
    binding.indexer_topk_eager(desc, q, k, w, ids, sc, ws)
    torch.cuda.synchronize()
    binding.indexer_topk_eager_device_status(desc, ws)
    parity.assert_exact(ids.cpu().numpy(), sc.cpu().numpy(), r_ids, r_sc)
