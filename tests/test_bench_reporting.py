"""CPU checks of the benchmark's reporting helpers: the clock summary taken
from nvidia-smi samples, the DRAM traffic figure taken from a committed ncu
capture (null once the hashed kernel sources differ from the captured ones),
and the consistency of the committed capture files themselves."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    s.sel = []
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def test_clock_summary_median_and_reasons(tmp_path):
    rows = [
        "0, 2070, 2070, 850.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 910.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 880.2, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    d = _sampler_with(tmp_path, rows).summary()
    assert d["samples"] == 3
    assert d["sm_mhz"] == 2070.0 and d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["sw_power_cap"]
    assert d["power_w_max"] == 910.0
    assert not os.path.exists(str(tmp_path / "clocks.csv"))  # the sample file is removed


def test_clock_summary_flags_thermal_slowdown(tmp_path):
    rows = ["0, 1500, 2070, 700, 0x40, Not Active, Active, Not Active, Not Active"]
    d = _sampler_with(tmp_path, rows).summary()
    assert d["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_without_samples(tmp_path):
    d = _sampler_with(tmp_path, []).summary()
    assert d["samples"] == 0 and d["reasons"] == ["unsampled"]


def test_traffic_follows_the_kernel_sources(monkeypatch):
    path = os.path.join(ROOT, "profiles", "decode_packed_w2_traffic.json")
    t = json.load(open(path))
    monkeypatch.setattr(bench, "kernel_sha", lambda: t["source_sha256"])
    # the captured launch size gives the captured bytes; another size scales by the ratio
    assert bench.traffic_for("w2", t["algorithmic_bytes_per_launch"]) == t["traffic_bytes_per_launch"]
    assert bench.traffic_for("w2", 10**9) == round(t["traffic_ratio"] * 10**9)
    # changed sources: no traffic figure
    monkeypatch.setattr(bench, "kernel_sha", lambda: "0" * 64)
    assert bench.traffic_for("w2", t["algorithmic_bytes_per_launch"]) is None
    # no capture for a workload: no traffic figure
    assert bench.traffic_for("no_such_workload", 1) is None


TRAFFIC_FILES = ("decode_packed_w2_traffic.json", "decode_packed_w5_traffic.json",
                 "decode_packed_w5_d256_traffic.json", "decode_packed_w5_d64_traffic.json")


def test_committed_traffic_files_are_consistent():
    for name in TRAFFIC_FILES:
        t = json.load(open(os.path.join(ROOT, "profiles", name)))
        assert tuple(t["source_files"]) == tuple(bench.DECODE_SRCS)
        assert len(t["source_sha256"]) == 64
        total = t["dram_bytes_read"] + t["dram_bytes_write"]
        alg = t.get("algorithmic_bytes_per_launch", t.get("algorithmic_bytes_per_launch_b1"))
        captured = t.get("traffic_bytes_per_launch", t.get("traffic_bytes_per_launch_b1"))
        assert captured == total
        assert abs(t["traffic_ratio"] - total / alg) < 1e-5
        # DRAM traffic within 2% of the algorithmic bytes: no re-reads
        assert 1.0 <= t["traffic_ratio"] < 1.02
        assert t["command"].startswith("ncu ") and "--clock-control none" in t["command"]


def test_committed_traffic_files_match_the_committed_kernel():
    """Every committed capture was taken on the decode sources as committed, so
    the benchmark's roofline carries a traffic figure; a change to those
    sources needs a new capture (and this fails until it is taken)."""
    sha = bench.kernel_sha()
    for name in TRAFFIC_FILES:
        t = json.load(open(os.path.join(ROOT, "profiles", name)))
        assert t["source_sha256"] == sha, name
    assert bench.traffic_for("w5", 69656903680) is not None
    assert bench.traffic_for("w5", 8674344960, 256) is not None
