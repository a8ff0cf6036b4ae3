"""bench.py's host-side helpers, without a GPU: the clock record taken from
nvidia-smi samples (median SM clock, throttle reasons) and the DRAM traffic
looked up by the kernel's source hash (null once the source has changed)."""
import json
import os

import bench


def test_clock_summary_parses_samples(tmp_path):
    csv = tmp_path / "clocks.csv"
    # clocks.sm, clocks.max.sm, power.draw, active, hw_slowdown, hw_thermal,
    # sw_thermal, sw_power_cap
    csv.write_text("\n".join([
        "2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # skipped
        "short, line",                                                                 # skipped
        "1980, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    ]) + "\n")
    s = bench.ClockSampler(0)
    s.path = str(csv)
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert not csv.exists()                       # the sample file is removed


def test_clock_summary_reports_thermal_reasons(tmp_path):
    csv = tmp_path / "clocks.csv"
    csv.write_text("1500, 2070, 1000, 0x40, Active, Not Active, Active, Not Active\n")
    s = bench.ClockSampler(0)
    s.path = str(csv)
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0)
    out = s.summary()
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "hyper_connection_residual_mhc_gb300" / "csrc"
    src.mkdir(parents=True)
    for f in bench.KERNEL_SRC["mhc_post"]:
        (src / f).write_text(f"// {f} as captured\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.src_hash(bench.KERNEL_SRC["mhc_post"])
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"mhc_post": {"src_sha256_16": h, "dram_bytes_per_launch_full_size": 1234}}))
    assert bench.traffic_for("mhc_post") == 1234
    (src / "post.cu").write_text("// the kernel, changed since\n")
    assert bench.traffic_for("mhc_post") is None
    assert bench.traffic_for("no_such_kernel") is None         # no entry, no file read error
    os.remove(tmp_path / "profiles" / "traffic.json")
    assert bench.traffic_for("mhc_post") is None
