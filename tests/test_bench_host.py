"""Host-side logic of bench.py that needs no GPU: the DRAM traffic record behind roofline.traffic
and the parsing of the nvidia-smi clock samples taken during the timed region."""
from __future__ import annotations

import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _write_record(root, kernels: dict):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "wl_dram.json"), "w") as f:
        json.dump({"workload": "wl", "kernels": kernels}, f)


def test_traffic_reported_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    hashes = {"pack": "a" * 16, "reshape_and_cache": "b" * 16}
    monkeypatch.setattr(bench, "source_hash", lambda paths: hashes["pack" if paths == bench.COPY_SOURCES
                                                                   else "reshape_and_cache"])
    _write_record(str(tmp_path), {"pack": {"source_hash": "a" * 16, "bytes_per_launch_full": 123},
                                  "unpack": {"source_hash": "0" * 16, "bytes_per_launch_full": 456},
                                  "reshape_and_cache": {"source_hash": "b" * 16, "bytes_per_launch_full": 789}})
    assert bench.ncu_traffic("wl", "pack") == 123
    assert bench.ncu_traffic("wl", "unpack") is None  # taken on other copy sources
    assert bench.ncu_traffic("wl", "reshape_and_cache") == 789
    assert bench.ncu_traffic("wl", "slot_mapping") is None  # no record for this kernel
    assert bench.ncu_traffic("no_such_workload", "pack") is None


def test_committed_traffic_records_are_plausible():
    """Every committed DRAM record holds, per kernel, the capture's bytes and the full-size
    figure scaled from it by the stated factor, near the kernel's algorithmic bytes."""
    algorithmic = {"page_shaped": {"pack": 3_623_878_656, "unpack": 3_623_878_656,
                                   "reshape_and_cache": 3_624_468_480}}
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        if not name.endswith("_dram.json"):
            continue
        with open(os.path.join(ROOT, "profiles", name)) as f:
            rec = json.load(f)
        scale = rec["scale"]
        assert scale >= 1
        for kernel, e in rec["kernels"].items():
            assert kernel in bench.KERNEL_SOURCES
            assert re.fullmatch(r"[0-9a-f]{16}", e["source_hash"])
            per_launch = (e["dram_read_bytes"] + e["dram_write_bytes"]) / e["launches"]
            assert abs(e["bytes_per_launch_full"] - round(per_launch * scale)) <= 1
            want = algorithmic.get(rec["workload"], {}).get(kernel)
            if want:
                assert 0.9 < e["bytes_per_launch_full"] / want < 1.05, (name, kernel)


def test_source_hash_follows_every_copy_source(tmp_path, monkeypatch):
    files = []
    for i, name in enumerate(("a.cu", "b.cuh")):
        p = tmp_path / name
        p.write_text(f"source {i}\n")
        files.append(name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.source_hash(files)
    (tmp_path / "b.cuh").write_text("source 1 changed\n")
    assert bench.source_hash(files) != before
    assert re.fullmatch(r"[0-9a-f]{16}", before)


def test_clock_summary(tmp_path):
    rows = [
        "0, 2070, 2070, 450.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 470.1, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 480.9, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.path = str(path)
    out = s.summary(0.0, 1.0)
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_max"] == 480.9
    assert not path.exists()  # the sample file is removed once read
    empty = bench.ClockSampler(0)
    empty.path = str(tmp_path / "missing.csv")
    assert empty.summary(0.0, 1.0)["reasons"] == ["no nvidia-smi samples"]
