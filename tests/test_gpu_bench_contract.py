"""bench.py prints the one JSON line the benchmark contract asks for (small run on the GPU)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
def test_bench_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "5", "--warmup", "3",
                        "--cpu-seconds", "0.5", "--workloads", "mla,asym_remap"], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny" and d["value"] > 0
    assert d["config"]["l2"].startswith("flushed")  # a step this small is timed with L2 flushed between steps
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    ac = d["cpu_baseline_all_cores"]
    assert ac["kind"] == "oracle" and ac["cores"] >= 1 and ac["value"] > 0
    for name, k in d["kernels"].items():
        assert k["ms_best"] <= k["ms_median"] and k["ms_best"] <= k["ms"], name
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 5 * 5  # slot_mapping, reshape_and_cache, builder, pack, unpack per step
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    # the roofline describes the slowest of the bandwidth-bound calls
    copies = {k: d["kernels"][k]["ms"] for k in ("reshape_and_cache", "pack", "unpack") if k in d["kernels"]}
    assert rf["kernel"] == max(copies, key=copies.get)
    # the other presets, each at full size with its own timed steps, clocks and roofline
    w = d["workloads"]
    assert set(w) == {"mla", "asym_remap"}
    for name, e in w.items():
        assert e["config"]["workload"] == name and e["steps"] >= 5 and e["value"] > 0
        assert e["roofline"]["kernel"] in e["kernels"] and e["roofline"]["frac"] > 0
        assert set(e["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert w["mla"]["config"]["layers"] == 61 and w["mla"]["config"]["num_blocks"] == 8192
    assert set(w["mla"]["kernels"]) >= {"pack", "reshape_and_cache"} and "unpack" not in w["mla"]["kernels"]
    assert w["mla"]["decode_write"]["tokens"] == 256
    assert all(v > 0 for v in w["mla"]["decode_write"]["device_us_per_write_back_to_back"].values())
    assert w["asym_remap"]["config"]["dst_block_size"] == 64 and "unpack" in w["asym_remap"]["kernels"]


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
@pytest.mark.parametrize("flags", [["--stage", "host"], ["--sw-window", "24"], ["--workload", "mid", "--layers", "1",
                                                                            "--num-blocks", "2048"]],
                         ids=["host_staging", "sliding_window", "mid_shrunk"])
def test_bench_modes_print_one_line(flags):
    args = [sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--no-cpu-baseline", "--no-workloads"]
    if "--workload" not in flags:
        args += ["--workload", "tiny"]
    r = subprocess.run(args + flags, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["value"] > 0 and d["roofline"]["achieved"] > 0 and d["gpu_launches"] > 0
    if "--stage" in flags:
        assert d["config"]["stage"] == "pinned host memory" and "host_link" in d


@pytest.mark.skipif(not torch.cuda.is_available(), reason="no CUDA device")
@pytest.mark.parametrize("workload,extra", [("tiny", []), ("mla", ["--num-blocks", "512"])], ids=["tiny", "mla_small"])
def test_bench_write_only(workload, extra):
    """--write-only (the write kernels' profiling driver) prints one line with both write forms timed."""
    r = subprocess.run([sys.executable, "bench.py", "--write-only", "--workload", workload, "--steps", "3"] + extra,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["tokens"] > 0 and d["bytes_per_write"] > 0
    assert set(d["device_us_per_write_back_to_back"]) == {"two_calls", "fused"}
    assert all(v > 0 for v in d["device_us_per_write_back_to_back"].values())
