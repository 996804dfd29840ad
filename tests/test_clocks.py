"""bench.py's clock record, on CPU: ClockSampler runs `nvidia-smi` in loop
mode during the timed region and reduces its CSV rows to the median SM
clock, the maximum clock and the throttle reasons seen.  A stand-in
`nvidia-smi` on PATH prints known rows."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_smi(tmp_path, rows):
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{r}'" for r in rows)
    script.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def _sample(monkeypatch, tmp_path, rows):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    time.sleep(0.3)
    return s.stop()


def test_median_max_and_reasons(monkeypatch, tmp_path):
    rows = ["2032, 2032, 700.1, Not Active, Not Active, Not Active, Not Active",
            "1980, 2032, 900.5, Not Active, Not Active, Not Active, Active",
            "2010, 2032, 800.0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    clk = _sample(monkeypatch, tmp_path, rows)
    assert clk == {"sm_mhz": 2010.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_slowdown_is_reported(monkeypatch, tmp_path):
    rows = ["1200, 2032, 1000.0, Active, Not Active, Active, Not Active"]
    clk = _sample(monkeypatch, tmp_path, rows)
    assert clk["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_unreadable_clocks_and_missing_tool(monkeypatch, tmp_path):
    clk = _sample(monkeypatch, tmp_path, ["[N/A], [N/A], [N/A], Not Active, Not Active, Not Active, Not Active"])
    assert clk == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 1}
    monkeypatch.setenv("PATH", str(tmp_path / "nowhere"))
    assert bench.ClockSampler(0).stop() is None
