"""Benchmark of the deterministic indexer top-k scan on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config S1]

One step = one full scan, the indexer_topk_run call (the scan kernel, then the selection
kernel -- or the merge kernel for split tails), over the workload's synthetic inputs. The
metric is effective TFLOP/s of useful causal MACs (2 * visible (query, key) pairs * H * D
per call), with ms per call (median over the timed steps) beside it. Inputs are resident
in HBM; L2 is flushed between timed steps. Under torchrun each rank runs its own replica
of the workload (seed + rank) on its own GPU: no collective touches the data path; the
timing is reduced with a MAX over ranks.

`--impl reference` times the CPU oracle (test infrastructure) on the host cores on a
bounded sample of the same workload; its per-call figure is extrapolated from the sample.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer top-k ms/call and effective TFLOP/s (causal MACs) vs BF16 tensor peak"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "scan_kernel_traffic.json")
# the device sources of the scan kernel (the selection and merge kernels, in itk_select.cuh,
# and the host code do not change the scan kernel's DRAM traffic)
KERNEL_SOURCES = [os.path.join(ROOT, "deterministic_top_key_gb300", "csrc", f)
                  for f in ("itk_common.cuh", "itk_scan.cuh", "itk_ptx.cuh")]


def _code_only(text: str) -> str:
    """The source without its comments and with whitespace collapsed: a comment-only edit
    does not change the compiled kernel, so it keeps the recorded traffic."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def visible_pairs(wl) -> int:
    cu_q, cu_k = wl.cu_seqlens_q.astype(np.int64), wl.cu_seqlens_k.astype(np.int64)
    total = 0
    for b in range(wl.num_segments):
        tq, tk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        off = wl.q_causal_offsets[b] if wl.q_causal_offsets is not None else tk - tq
        # query i sees off + i + 1 keys
        total += int(tq * (off + 1) + tq * (tq - 1) // 2)
    return total


def row_visible(wl) -> np.ndarray:
    out = np.zeros(wl.T, np.int64)
    for b in range(wl.num_segments):
        q0, q1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
        tq, tk = q1 - q0, int(wl.cu_seqlens_k[b + 1] - wl.cu_seqlens_k[b])
        off = int(wl.q_causal_offsets[b]) if wl.q_causal_offsets is not None else tk - tq
        out[q0:q1] = off + np.arange(tq) + 1
    return out


def finish_kernels(binding, wl) -> str:
    """The launches after the scan: the merge for split queries, the selection for the rest."""
    ut = binding.indexer_topk_unit_table(binding.Desc(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k,
                                                      wl.q_causal_offsets))
    _, per_block = np.unique(ut[:, 0], return_counts=True)
    names = (["merge"] if (per_block > 1).any() else []) + (["selection"] if (per_block == 1).any() else [])
    return " + ".join(names)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


def load_traffic():
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None  # counters were taken on another version of the kernel
    return d


def pci_bus_id(props):
    """nvidia-smi's name of a CUDA device ("00000000:1B:00.0"), from its properties."""
    try:
        return f"{int(props.pci_domain_id):08X}:{int(props.pci_bus_id):02X}:{int(props.pci_device_id):02X}.0"
    except (AttributeError, TypeError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int, bus_id: str | None = None):
        # nvidia-smi numbers the physical GPUs and ignores CUDA_VISIBLE_DEVICES: name the
        # device by its PCI bus id when it is known, so that the samples are of this GPU
        self.gpu = gpu_index
        self.bus_id = bus_id
        self.proc = None
        # raw samples: $ITK_CLOCKS_DIR if set, else the temporary directory
        out_dir = os.environ.get("ITK_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"itk_clocks_rank{gpu_index}.csv")
        self.timed = None  # (t0, t1) host wall clock of the timed region

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.bus_id or self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # wait (bounded) for the first sample so that sampling is live before any timed work
        t_end = time.time() + 10.0
        while time.time() < t_end and self.proc.poll() is None:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        return self

    def mark_timed(self, t0: float, t1: float):
        self.timed = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def _samples(self):
        import datetime

        out = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm, smax = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                reasons = {n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")}
                out.append((ts, sm, smax, reasons))
        return out

    def summary(self):
        """Median SM clock of the samples taken inside the timed region; when that region is
        shorter than the sampling period, of all samples taken while this benchmark kept the
        GPU busy (warm-up, timed steps, end-to-end and per-config runs), as `window` says."""
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        samples = self._samples()
        window = "timed region"
        if self.timed is not None:
            # 100 ms of slack: a sample's timestamp is when nvidia-smi started its query
            inside = [x for x in samples if self.timed[0] - 0.1 <= x[0] <= self.timed[1] + 0.1]
            if inside:
                samples_used = inside
            else:
                samples_used = samples
                window = "all GPU work of this run (timed region shorter than the sampling period)"
        else:
            samples_used = samples
            window = "all GPU work of this run"
        if not samples_used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set().union(*[x[3] for x in samples_used])
        return {"sm_mhz": float(np.median([x[1] for x in samples_used])),
                "sm_max_mhz": float(max(x[2] for x in samples_used)), "reasons": sorted(reasons),
                "samples": len(samples_used), "window": window, "period_ms": self.PERIOD_MS,
                "gpu": self.bus_id or f"index {self.gpu}"}


def cpu_oracle_sample(wl, budget_s: float, seed_rows: int = 32):
    """Time the oracle on a growing, evenly spaced sample of query rows until it has run
    for at least budget_s / 3 seconds; returns (flops of the sample, seconds, rows, threads)."""
    import oracle

    oracle.build()
    p = oracle.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, wl.q_causal_offsets)
    vis = row_visible(wl)
    n = min(seed_rows, wl.T)
    while True:
        rows = np.unique(np.linspace(0, wl.T - 1, n).astype(np.int32))
        t0 = time.perf_counter()
        oracle.topk(p, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 3 or len(rows) >= wl.T:
            flops = 2.0 * float(vis[rows].sum()) * wl.H * wl.D
            return flops, dt, len(rows), oracle.max_threads()
        n = min(wl.T, int(n * max(2.0, budget_s / 3 / max(dt, 1e-3))))


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank runs its own replica, timed by the slowest rank."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The oracle on the host cores: each step scans a bounded sample of the workload."""
    world, rank, _ = dist_init()
    if rank != 0:
        return 0
    from deterministic_top_key_gb300 import inputs

    wl = inputs.make(args.config, seed=0)
    # size one step's sample so that all steps together take about a minute
    per_step_s = max(0.5, min(args.ref_budget, 60.0 / max(args.steps, 1)))
    flops, dt, nrows, threads = cpu_oracle_sample(wl, 3 * per_step_s)
    import oracle

    p = oracle.Problem(wl.q_bits, wl.k_bits, wl.w, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k, wl.q_causal_offsets)
    rows = np.unique(np.linspace(0, wl.T - 1, nrows).astype(np.int32))
    for _ in range(args.warmup):
        oracle.topk(p, rows=rows[: max(1, len(rows) // 8)])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.topk(p, rows=rows)
        times.append(time.perf_counter() - t0)
    t = float(np.median(times))
    value = flops / t / 1e12
    full_flops = 2.0 * visible_pairs(wl) * wl.H * wl.D
    sample = f"{len(rows)} of {wl.T} query rows, evenly spaced ({flops / full_flops:.4%} of the call's MACs)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_flops / (value * 1e12) * 1e3,
        "ms_per_step_kind": "extrapolated: the whole call's MACs at the sample's measured rate",
        "sample_ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, world):
    from deterministic_top_key_gb300 import inputs

    return {"workload": f"{wl.name}: {inputs.config(wl.name)['desc']}", "T": wl.T, "Tkv": wl.Tkv, "H": wl.H,
            "D": wl.D, "top_k": wl.top_k, "segments": wl.num_segments, "l2": "flushed between timed steps",
            "replicas": world, "inputs": "q,k ~ N(0,1) BF16, w ~ N(0,1)/8, seed 0 (+rank)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="S1")
    ap.add_argument("--per-config", default="tiny,S2,C1,Z2,Z3,A1,A2,A3",
                    help="extra configs timed and reported in per_config ('' = none)")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--cpu-budget-per-config", type=float, default=3.0,
                    help="seconds of oracle work for each per_config cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--residency", action="store_true",
                    help="instead of the standard line: time the call while a kernel on another stream holds 1 or "
                         "32 SMs, with the ticket schedule and with a fixed schedule")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.residency:
        return run_residency(args)
    return run_ours(args)


def _to_device(torch, wl, dev):
    q = torch.from_numpy(wl.q_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    k = torch.from_numpy(wl.k_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(wl.w).to(dev)
    return q, k, w


def _measure(binding, torch, wl, dev, steps, warmup, flush_buf):
    q, k, w = _to_device(torch, wl, dev)
    plan = binding.indexer_topk_prepare(wl.T, wl.Tkv, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.top_k,
                                        wl.q_causal_offsets)
    ws = torch.empty(max(plan.workspace_bytes(), 1), dtype=torch.uint8, device=dev)
    ids = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device=dev)
    sc = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush_buf.fill_(1)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws, stream)
    torch.cuda.synchronize()
    plan.device_status()
    return plan, (q, k, w, ids, sc, ws), stream


def _timed_steps(binding, torch, plan, bufs, stream, steps, flush_buf, split=False):
    """Times `steps` runs with CUDA events on the launching stream, the L2 flushed before
    every step outside the events. Without `split`: the whole call (start..end), launched
    exactly as a caller launches it. With `split`: the library also records an event right
    after the scan launch, so start..split is the scan kernel and split..end the rest. That
    event sits between two kernels that otherwise overlap their launch (programmatic
    dependent launch), so split runs serve the per-kernel figures only."""
    starts, splits, ends = ([torch.cuda.Event(enable_timing=True) for _ in range(steps)] for _ in range(3))
    for e in splits:  # create the events' device handles
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        flush_buf.fill_(i & 0xFF)
        if split:
            binding.indexer_topk_set_split_event(plan, splits[i])
        starts[i].record(stream)
        binding.indexer_topk_run(plan, *bufs, stream)
        ends[i].record(stream)
    if split:
        binding.indexer_topk_set_split_event(plan, None)
    return starts, (splits if split else None), ends


def _step_ms(starts, splits, ends):
    """Median over the timed steps of the whole call, and (with splits) of its two parts."""
    ends[-1].synchronize()
    total = np.array([a.elapsed_time(b) for a, b in zip(starts, ends)])
    if splits is None:
        return float(np.median(total)), None, None
    scan = np.array([a.elapsed_time(b) for a, b in zip(starts, splits)])
    sel = np.array([a.elapsed_time(b) for a, b in zip(splits, ends)])
    return float(np.median(total)), float(np.median(scan)), float(np.median(sel))


def _e2e(binding, torch, wl, plan, bufs, stream, args, flush_buf, flops, world, dist, dev):
    """End to end through the public API: every step copies its inputs from pinned host
    memory, runs the scan and copies the ids and scores back to pinned host memory.

    Two measurements. `serial`: copy in, run, copy out, one after another on one stream.
    `value` (pipelined): the way a serving loop would overlap them: the copy-in of step
    i + 1 and the copy-out of step i - 1 run on their own streams while step i computes
    (double-buffered device inputs and outputs); a timed window spans the first copy-in to
    the last copy-out of `steps` steps, so it holds every step's copies, and the median of
    three windows is reported."""
    q, k, w, ids, sc, ws = bufs
    hq = torch.from_numpy(wl.q_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hk = torch.from_numpy(wl.k_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(wl.w).pin_memory()
    hid = [torch.empty(ids.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    hsc = [torch.empty(sc.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = hq.numel() * 2 + hk.numel() * 2 + hw.numel() * 4
    d2h = hid[0].numel() * 4 + hsc[0].numel() * 4

    # serial: one stream, steps back to back
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        flush_buf.fill_(i & 0xFF)
        if i >= args.warmup:
            e_s[i - args.warmup].record(stream)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        w.copy_(hw, non_blocking=True)
        binding.indexer_topk_run(plan, q, k, w, ids, sc, ws, stream)
        hid[0].copy_(ids, non_blocking=True)
        hsc[0].copy_(sc, non_blocking=True)
        if i >= args.warmup:
            e_e[i - args.warmup].record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(float(np.median([a.elapsed_time(b) for a, b in zip(e_s, e_e)])), dist, dev)

    # pipelined: copy-in stream, compute stream, copy-out stream, two buffer sets
    dq = [q, torch.empty_like(q)]
    dk = [k, torch.empty_like(k)]
    dw = [w, torch.empty_like(w)]
    did = [ids, torch.empty_like(ids)]
    dsc = [sc, torch.empty_like(sc)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    loaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def pipeline(n_steps, t0=None, t1=None):
        for i in range(n_steps):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[b])  # step i - 2 has read this input set
                if i == 0 and t0 is not None:
                    t0.record(s_in)
                dq[b].copy_(hq, non_blocking=True)
                dk[b].copy_(hk, non_blocking=True)
                dw[b].copy_(hw, non_blocking=True)
                loaded[b].record(s_in)
            stream.wait_event(loaded[b])
            if i >= 2:
                stream.wait_event(drained[b])  # step i - 2's outputs are on the host
            binding.indexer_topk_run(plan, dq[b], dk[b], dw[b], did[b], dsc[b], ws, stream)
            computed[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[b])
                hid[b].copy_(did[b], non_blocking=True)
                hsc[b].copy_(dsc[b], non_blocking=True)
                drained[b].record(s_out)
        if t1 is not None:
            t1.record(s_out)

    torch.cuda.synchronize()
    pipeline(args.warmup)
    torch.cuda.synchronize()
    # three windows of `steps` pipelined steps; the median window is reported (the host
    # link is shared, and one window can catch another job's transfers)
    windows = []
    for _ in range(3):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipeline(args.steps, t0, t1)
        torch.cuda.synchronize()
        windows.append(t0.elapsed_time(t1) / args.steps)
    pipe_ms = max_over_ranks(float(np.median(windows)), dist, dev)
    return {"value": job_tflops(flops, world, pipe_ms), "unit": "TFLOP/s", "ms_per_step": pipe_ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": True, "window_ms_per_step": [round(x, 4) for x in windows],
            "serial": {"value": job_tflops(flops, world, serial_ms), "ms_per_step": serial_ms},
            "note": "copies of step i + 1 (in) and i - 1 (out) overlap step i's compute; median of three windows of "
                    "`steps` steps; serial = no overlap"}


def run_residency(args):
    """Side-stream residency benchmark (flashinfer PR #8691, opening description and the
    side-stream table): a kernel on a second stream holds n SMs (so that n scan CTAs cannot
    start) for about one call's time, launched just before each call. With the ticket
    schedule the running CTAs take every unit and the held CTAs find none left; with a
    fixed schedule (CTA b owns units b, b + grid, ...) the held CTAs' units run as a second
    wave after the holder leaves. Prints one JSON line of per-call times and ratios."""
    import torch

    from deterministic_top_key_gb300 import binding, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2_bytes, 256 << 20), dtype=torch.uint8, device=dev)
    wl = inputs.make(args.config)
    plan, bufs, stream = _measure(binding, torch, wl, dev, args.steps, args.warmup, flush_buf)
    side = torch.cuda.Stream()

    def timed(hold_sms, hold_us, static):
        binding.indexer_topk_debug_inject(plan, 3 if static else 4)
        ms = []
        for i in range(args.warmup + args.steps):
            flush_buf.fill_(i & 0xFF)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            binding.indexer_topk_bench_hold(hold_sms, hold_us, side)
            a.record(stream)
            binding.indexer_topk_run(plan, *bufs, stream)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                ms.append(a.elapsed_time(b))
        binding.indexer_topk_debug_inject(plan, 4)
        plan.device_status()
        return float(np.median(ms))

    base = timed(0, 0, False)
    base_static = timed(0, 0, True)
    hold_us = int(base * 1000)
    rows = {}
    for n in (1, 32):
        t_ticket = timed(n, hold_us, False)
        t_static = timed(n, hold_us, True)
        rows[f"hold_{n}"] = {"ticket_ms": t_ticket, "fixed_ms": t_static, "ticket_ratio": t_ticket / base,
                             "fixed_ratio": t_static / base_static}
    plan.destroy()
    line = {"metric": "call time with n SMs held by another stream, relative to none held", "unit": "ratio",
            "config": {"workload": f"{wl.name}: {inputs.config(wl.name)['desc']}", "hold_us": hold_us},
            "base_ms": {"ticket": base, "fixed": base_static}, "rows": rows, "steps": args.steps,
            "warmup": args.warmup, "data": "synthetic"}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    from deterministic_top_key_gb300 import binding, inputs

    world, rank, local = dist_init()
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()

    peaks, peak_src = load_peaks()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2_bytes, 256 << 20), dtype=torch.uint8, device=dev)

    wl = inputs.make(args.config, seed=rank)
    flops = 2.0 * visible_pairs(wl) * wl.H * wl.D
    clocks = ClockSampler(local, pci_bus_id(torch.cuda.get_device_properties(dev))).__enter__()
    # (sampling covers warm-up through the per-config runs)
    plan, bufs, stream = _measure(binding, torch, wl, dev, args.steps, args.warmup, flush_buf)
    q, k, w, ids, sc, ws = bufs

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    wall0 = time.perf_counter()
    t_timed0 = time.time()
    starts, splits, ends = _timed_steps(binding, torch, plan, bufs, stream, args.steps, flush_buf)
    barrier()
    clocks.mark_timed(t_timed0, time.time())
    wall = time.perf_counter() - wall0
    plan.device_status()
    total_ms, _, _ = _step_ms(starts, splits, ends)
    ms = max_over_ranks(total_ms, dist, dev)
    value = job_tflops(flops, world, ms)
    # per-kernel figures: the same steps again with the split event between the launches
    split_ms, scan_ms, sel_ms = _step_ms(*_timed_steps(binding, torch, plan, bufs, stream, args.steps, flush_buf,
                                                       split=True))
    torch.cuda.synchronize()
    plan.device_status()
    split_ms = max_over_ranks(split_ms, dist, dev)
    scan_ms = max_over_ranks(scan_ms, dist, dev)
    sel_ms = max_over_ranks(sel_ms, dist, dev)

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = _e2e(binding, torch, wl, plan, bufs, stream, args, flush_buf, flops, world, dist, dev)

    # per-config figures (same method; parity-test configs, reported for the roofline)
    traffic = load_traffic()
    per_config = {}
    for name in [c for c in args.per_config.split(",") if c and c != args.config]:
        wl2 = inputs.make(name, seed=rank)
        f2 = 2.0 * visible_pairs(wl2) * wl2.H * wl2.D
        plan2, b2, st2 = _measure(binding, torch, wl2, dev, args.steps, args.warmup, flush_buf)
        m2, _, _ = _step_ms(*_timed_steps(binding, torch, plan2, b2, st2, args.steps, flush_buf))
        _, m2_scan, m2_sel = _step_ms(*_timed_steps(binding, torch, plan2, b2, st2, args.steps, flush_buf, split=True))
        torch.cuda.synchronize()
        plan2.device_status()
        tf2 = f2 / (m2 * 1e-3) / 1e12
        tf2_scan = f2 / (m2_scan * 1e-3) / 1e12
        pc = {"ms": m2, "tflops": tf2, "frac": tf2 / peaks["bf16_tflops"],
              "scan_ms": m2_scan, "scan_tflops": tf2_scan, "scan_frac": tf2_scan / peaks["bf16_tflops"],
              "finish_ms": m2_sel, "finish": finish_kernels(binding, wl2), "T": wl2.T, "Tkv": wl2.Tkv,
              "top_k": wl2.top_k, "gflop": f2 / 1e9,
              "scan_traffic_bytes": None if traffic is None else traffic.get("per_config_bytes", {}).get(name)}
        plan2.destroy()
        del b2
        if rank == 0 and args.cpu_budget_per_config > 0:
            fs, ds, nr, th = cpu_oracle_sample(wl2, args.cpu_budget_per_config)
            pc["cpu_baseline"] = {"value": fs / ds / 1e12, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                                  "sample": f"{nr} of {wl2.T} query rows, evenly spaced; {ds:.1f} s"}
        per_config[name] = pc

    clocks.__exit__(None, None, None)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    finish = [{"merge": "merge", "selection": "select"}[f] for f in finish_kernels(binding, wl).split(" + ")]
    achieved = flops / (scan_ms * 1e-3) / 1e12  # the dominant kernel alone
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json bf16_tflops)" if peak_src == "measured"
                else "fallback 1.9 PFLOP/s bf16 burst",
                "traffic": None if traffic is None else traffic["bytes_per_launch_scaled"],
                "algorithmic_flops_per_launch": flops, "kernel": "indexer_topk_scan_kernel",
                "kernel_ms": scan_ms, "step_frac": value / world / peaks["bf16_tflops"]}
    if traffic is not None:
        roofline["traffic_note"] = traffic.get("note", "")
    flops_s, dt_s, nrows, threads = cpu_oracle_sample(wl, args.cpu_budget)
    cpu = {"value": flops_s / dt_s / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"{nrows} of {wl.T} query rows of {wl.name}, evenly spaced; {dt_s:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(wl, world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks.summary(),
        "gpu_launches": (1 + len(finish)) * args.steps,
        "kernels": {"indexer_topk_scan_kernel": {"ms": scan_ms, "launches": args.steps},
                    " + ".join(f"indexer_topk_{f}_kernel" for f in finish): {"ms": sel_ms, "launches": args.steps},
                    "split_run_ms_per_step": split_ms,
                    "note": "separate runs of the same steps with an event between the launches"},
        "per_config": per_config, "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
