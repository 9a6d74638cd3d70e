"""The benchmark's clock record: samples parsed from nvidia-smi's CSV, restricted to the
timed region when it holds any, with every throttle reason reported."""
import datetime
import os

import bench


def _line(ts, sm, reasons=("Not Active",) * 4):
    t = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{t}, 0, {sm}, 2070, 900.5, 0x0000000000000000, " + ", ".join(reasons) + "\n"


def _sampler(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = os.path.join(tmp_path, "clocks.csv")
    with open(s.path, "w") as f:
        f.writelines(lines)
    s.proc = object()  # stands in for the nvidia-smi process, already finished
    return s


def test_timed_region_samples_only(tmp_path):
    t0 = 1_700_000_000.0
    lines = [_line(t0 + i * 0.05, 1000 + i) for i in range(40)]  # 2 s of samples
    s = _sampler(tmp_path, lines)
    s.mark_timed(t0 + 1.0, t0 + 1.2)
    out = s.summary()
    assert out["window"] == "timed region"
    # samples from 0.9 s to 1.3 s (100 ms slack each side): 1018 .. 1026
    assert out["samples"] == 9 and out["sm_mhz"] == 1022.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == []


def test_short_region_falls_back_and_keeps_reasons(tmp_path):
    t0 = 1_700_000_000.0
    lines = [_line(t0, 2070), _line(t0 + 0.05, 1900, ("Not Active", "Not Active", "Not Active", "Active")),
             "garbage line\n"]
    s = _sampler(tmp_path, lines)
    s.mark_timed(t0 + 10.0, t0 + 10.01)
    out = s.summary()
    assert out["window"].startswith("all GPU work")
    assert out["samples"] == 2 and out["reasons"] == ["sw_power_cap"]


def test_sampler_names_the_gpu_by_pci_bus_id():
    """nvidia-smi numbers physical GPUs and ignores CUDA_VISIBLE_DEVICES, so the sampler
    asks for the CUDA device's PCI bus id, built from its properties."""
    from types import SimpleNamespace

    props = SimpleNamespace(pci_domain_id=0, pci_bus_id=0x1B, pci_device_id=0)
    assert bench.pci_bus_id(props) == "00000000:1B:00.0"
    assert bench.pci_bus_id(SimpleNamespace()) is None
    s = bench.ClockSampler(3, "00000000:1B:00.0")
    assert s.bus_id == "00000000:1B:00.0"
