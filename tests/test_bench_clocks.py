"""The bench's clock sampler (host only: a stand-in nvidia-smi on PATH prints
fixed samples).  The bench line's "clocks" key carries the median SM clock
under load, the maximum, and every throttle reason seen active."""
import os
import stat

import bench

# index, clocks.sm, clocks.max.sm, power.draw, active mask, hw_slowdown,
# hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
SAMPLES = [
    "0, 2070, 2070, 850.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 2070, 2070, 1100.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, [N/A], 2070, 900.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "garbage line",
]


def fake_smi(tmp_path, lines):
    exe = tmp_path / "nvidia-smi"
    body = "".join(f"echo '{ln}'\n" for ln in lines)
    exe.write_text("#!/bin/sh\n" + body + "exec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def test_samples_parsed_and_reasons_collected(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", fake_smi(tmp_path, SAMPLES) + os.pathsep + os.environ["PATH"])
    with bench.ClockSampler(0) as clk:
        path = clk.path
    s = clk.summary()
    assert s["samples"] == 3              # the N/A and malformed lines are skipped
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(path)


def test_hw_slowdown_reported(tmp_path, monkeypatch):
    lines = ["0, 1500, 2070, 700.0, 0x08, Active, Not Active, Not Active, Not Active",
             "0, 1400, 2070, 690.0, 0x48, Active, Active, Not Active, Not Active"]
    monkeypatch.setenv("PATH", fake_smi(tmp_path, lines) + os.pathsep + os.environ["PATH"])
    with bench.ClockSampler(0) as clk:
        pass
    s = clk.summary()
    assert s["sm_mhz"] == 1450.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))   # an empty directory: no nvidia-smi
    with bench.ClockSampler(0) as clk:
        path = clk.path
    s = clk.summary()
    assert s["sm_mhz"] is None and s["reasons"] == ["nvidia-smi unavailable"]
    assert not os.path.exists(path)
