"""The bench's clock sampler on CPU, with a stand-in for nvidia-smi on PATH
that prints one CSV row of the sampler's fields every 20 ms: samples taken
before a pause and after a resume are both kept, none are taken while
paused, the summary reports the median clock and the throttle reasons seen,
and a missing nvidia-smi gives no clock record instead of an error."""
import os
import stat
import time

import pytest


def _fake_smi(tmp_path, sm_mhz, reason_cap):
    script = tmp_path / "nvidia-smi"
    # index, clocks.sm, clocks.max.sm, power.draw, active, hw_slowdown,
    # hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    row = f"0, {sm_mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {reason_cap}"
    script.write_text("#!/bin/sh\nwhile true; do echo '" + row + "'; sleep 0.02; done\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return script


@pytest.fixture
def bench_mod():
    import bench
    return bench


def test_pause_resume_keeps_both_windows(tmp_path, monkeypatch, bench_mod):
    _fake_smi(tmp_path, 1980, "Active")
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench_mod.ClockSampler(0)
    s.start()
    time.sleep(0.2)
    s.pause()
    n_first = len(s.rows)
    assert n_first >= 1
    assert s.proc is None
    time.sleep(0.2)
    assert len(s.rows) == n_first  # nothing is sampled while paused
    s.resume()
    time.sleep(0.2)
    clk = s.stop()
    assert len(s.rows) > n_first
    assert clk["samples"] == len(s.rows)
    assert clk["sm_mhz"] == pytest.approx(1980.0)
    assert clk["sm_max_mhz"] == pytest.approx(2070.0)
    assert clk["reasons"] == ["sw_power_cap"]


def test_start_waits_for_the_first_sample(tmp_path, monkeypatch, bench_mod):
    _fake_smi(tmp_path, 2070, "Not Active")
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench_mod.ClockSampler(0)
    s.start()
    clk = s.stop()  # stopped at once: the first row is already there
    assert clk is not None and clk["samples"] >= 1
    assert clk["reasons"] == []


def test_missing_tool_gives_no_record(tmp_path, monkeypatch, bench_mod):
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi anywhere
    s = bench_mod.ClockSampler(0)
    s.start()
    s.pause()
    s.resume()
    assert s.stop() is None
