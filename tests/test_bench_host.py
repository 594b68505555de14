"""Host-side logic of bench.py that needs no GPU: the clock sampler keeps only
the nvidia-smi samples stamped inside the timed region and reports the
throttle reasons seen there (an nvidia-smi stand-in prints the samples)."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

FAKE_SMI = r'''#!/usr/bin/env python3
import datetime, os, sys, time
# one sample every 20 ms; samples taken while the flag file exists report a
# power cap (the bench must see it only if they fall in its window)
flag = os.environ["FAKE_SMI_FLAG"]
while True:
    ts = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    cap = "Active" if os.path.exists(flag) else "Not Active"
    clk = 1500 if os.path.exists(flag) else 2070
    print(f"{ts}, 0, {clk}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}", flush=True)
    time.sleep(0.02)
'''


def _fake_smi(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE_SMI)
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    flag = tmp_path / "cap"
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    monkeypatch.setenv("FAKE_SMI_FLAG", str(flag))
    return flag


def test_clock_sampler_keeps_only_the_timed_region(tmp_path, monkeypatch):
    flag = _fake_smi(tmp_path, monkeypatch)
    import bench
    flag.write_text("")                 # a power cap before the timed region ...
    c = bench.ClockSampler(0)
    time.sleep(0.3)
    flag.unlink()                       # ... lifted before it starts
    time.sleep(0.1)
    c.start_window()
    time.sleep(0.3)
    c.end_window()
    flag.write_text("")                 # and back after it ends
    time.sleep(0.2)
    r = c.stop()
    assert r is not None and r["samples_in_timed_region"]
    assert r["samples"] >= 5
    assert r["reasons"] == [] and r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0


def test_clock_sampler_reports_a_cap_inside_the_region(tmp_path, monkeypatch):
    flag = _fake_smi(tmp_path, monkeypatch)
    import bench
    c = bench.ClockSampler(0)
    time.sleep(0.1)
    c.start_window()
    flag.write_text("")
    time.sleep(0.3)
    c.end_window()
    r = c.stop()
    assert r is not None and r["samples_in_timed_region"]
    assert "sw_power_cap" in r["reasons"]
    assert r["sm_mhz"] < 2070.0
