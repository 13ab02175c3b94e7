"""Host-side logic of bench.py that needs no GPU: the DRAM traffic record behind roofline.traffic
and the parsing of the nvidia-smi clock samples taken during the timed region."""
from __future__ import annotations

import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _record():
    with open(os.path.join(ROOT, "profiles", "page_shaped_pack_dram.md")) as f:
        text = f.read()
    h = re.search(r"^source_hash: (\w+)$", text, re.M).group(1)
    b = int(re.search(r"^pack_dram_bytes_per_launch: (\d+)$", text, re.M).group(1))
    return h, b


def test_traffic_reported_only_for_the_sources_it_was_taken_on(monkeypatch):
    h, b = _record()
    # the record is plausible: DRAM bytes of one full-size pack launch, near its algorithmic bytes
    assert 0.9 < b / 3_623_878_656 < 1.02
    monkeypatch.setattr(bench, "source_hash", lambda paths: h)
    assert bench.ncu_traffic("page_shaped") == b
    monkeypatch.setattr(bench, "source_hash", lambda paths: "0" * 16)  # the copy kernels changed
    assert bench.ncu_traffic("page_shaped") is None
    assert bench.ncu_traffic("no_such_workload") is None


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
