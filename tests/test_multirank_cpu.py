"""The benchmark's multi-process path on CPU: two gloo ranks, and the reference arm
under torchrun with two processes (rank 0 alone prints the JSON line)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from deterministic_top_key_gb300 import inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank times its own replica; the slowest rank sets the job time
        ms = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
        # replicas differ by seed: rank r draws seed r
        wl = inputs.make("tiny", seed=rank)
        digest = float(wl.q_bits[:4].astype("float64").sum())
        flops = 2.0 * bench.visible_pairs(wl) * wl.H * wl.D
        q.put((rank, ms, digest, bench.job_tflops(flops, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_replicate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[1] for o in out] == [2.5, 2.5]  # MAX over ranks
    assert out[0][2] != out[1][2]  # different replicas
    # tiny: 131328 visible pairs x 64 x 128 x 2 FLOP per rank, two ranks, 2.5 ms
    assert out[0][3] == pytest.approx(2 * 2.0 * 131328 * 64 * 128 / 2.5e-3 / 1e12)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--config",
           "tiny", "--steps", "2", "--warmup", "1", "--ref-budget", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
