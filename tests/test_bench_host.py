"""The benchmark's host-side bookkeeping, on CPU.

* the clock summary keeps only the samples inside the timed window and
  reports every throttle reason that was active there;
* a traffic figure is reported only while the kernel's sources hash to the
  value recorded with it (an edited kernel reads as null);
* the FFMA and tf32 peaks follow from the unit counts and the clock;
* the per-call launch count follows the plan (copies, GEMM, reduce).
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def sample(sm, mx, hw="Not Active", thermal="Not Active", sw_thermal="Not Active",
           power="Not Active"):
    return f"2026/12/02 10:00:00.000, {sm}, {mx}, 900.0, 0x0, {hw}, {thermal}, {sw_thermal}, {power}"


def test_clock_summary_keeps_the_timed_window_and_its_reasons():
    c = bench.ClockSampler(0)
    c.lines = [(1.0, sample(900, 2070, hw="Active")),          # before t0: ignored
               (2.0, sample(2070, 2070)),
               (2.1, sample(2040, 2070, power="Active")),
               (2.2, sample(2070, 2070)),
               (5.0, sample(300, 2070, thermal="Active"))]     # after t1: ignored
    c.t0, c.t1 = 1.5, 2.3
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    c.t1 = 6.0
    assert c.summary()["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples():
    c = bench.ClockSampler(0)
    c.lines = [(1.0, "garbled line")]
    assert c.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    (tmp_path / "profiles").mkdir()
    import hashlib
    entry = {"bytes_per_launch": 1234, "sources": ["kernel.cu"],
             "sources_sha256": hashlib.sha256(src.read_bytes()).hexdigest()}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k_case": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k_case") == 1234
    assert bench.load_traffic("other_case") is None
    src.write_text("__global__ void k() { /* edited */ }\n")
    assert bench.load_traffic("k_case") is None


def test_committed_traffic_entries_name_existing_sources():
    table = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, entry in table.items():
        assert entry["bytes_per_launch"] > 0, key
        for rel in entry["sources"]:
            assert os.path.exists(os.path.join(ROOT, rel)), (key, rel)


def test_peaks_from_unit_counts_and_clock():
    # 152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz.
    assert bench.ffma_peak_tflops(152, 2070.0) == pytest.approx(80.54784)
    # 152 SMs x 4096 tf32 flop per clock x 2070 MHz.
    assert bench.tf32_clock_peak(152, 2070.0) == pytest.approx(1288.76544)


@pytest.mark.parametrize("plan,want", [
    (dict(variant=0, pack_a=5, split_k=4, workspace_bytes=1), 3),   # copy, GEMM, reduce
    (dict(variant=0, pack_a=4, split_k=1, workspace_bytes=0), 1),   # gathered, no split
    (dict(variant=2, pack_a=0, split_k=1, workspace_bytes=0), 1),   # the one-warp kernel
    (dict(variant=0, pack_a=5, split_k=1, stream_k=456, workspace_bytes=1), 3),  # copy, GEMM, fix-up
    (dict(variant=1, pack_a=1, split_k=1, stream_k=76, workspace_bytes=1), 4),   # packs, GEMM, fix-up
])
def test_launch_count_follows_the_plan(plan, want):
    assert bench.launches_per_call(plan) == want
