"""bench.py keeps its one-JSON-line contract: the reference (oracle) arm on
CPU, and the GPU arm with every leg (route timing, Ulysses, e2e, CPU
baseline) on the tiny workload."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMMON = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
          "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=timeout, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_contract():
    d = _run(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"], 300)
    assert COMMON <= set(d)
    assert d["impl"] == "reference" and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["higher_is_better"] is True and d["value"] > 0


@pytest.mark.gpu
def test_gpu_arm_contract():
    d = _run(["--workload", "tiny", "--steps", "3", "--warmup", "3", "--cpu-budget", "1"], 600)
    assert COMMON | {"roofline", "gpu_launches", "clocks", "route_build_us"} <= set(d)
    assert "impl" not in d
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["gpu_launches"] == 3 * (2 + 2 * 48)
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["swap_us_distribution"]["p10"] <= d["swap_us_distribution"]["p90"]


def test_clock_sampler_targets_the_benchmarked_gpu(monkeypatch):
    """nvidia-smi is asked about the GPU the benchmark runs on: its PCI
    address when torch reports one, else the index through CUDA_VISIBLE_DEVICES."""
    import types
    import torch
    import bench
    dev = torch.device("cuda", 1)
    props = types.SimpleNamespace(pci_domain_id=0, pci_bus_id=0x1B, pci_device_id=0)
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda d: props)
    assert bench.smi_gpu_id(dev) == "00000000:1B:00.0"

    def no_props(d):
        raise AttributeError("no pci fields")
    monkeypatch.setattr(torch.cuda, "get_device_properties", no_props)
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.smi_gpu_id(dev) == "5"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.smi_gpu_id(dev) == "1"
