"""bench.py's clock sampler on the CPU, against a stand-in for nvidia-smi that
prints the queried fields every 20 ms (no GPU and no real nvidia-smi needed)."""
import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

FAKE = """#!{py}
import sys, time
while True:
    print("0, {sm}, 2070, 900.00, 0x0000000000000000, {hw}, Not Active, Not Active, {pc}", flush=True)
    time.sleep(0.02)
"""


def _fake_smi(tmp_path, monkeypatch, sm=2070, hw="Not Active", pc="Active"):
    path = tmp_path / "nvidia-smi"
    path.write_text(FAKE.format(py=sys.executable, sm=sm, hw=hw, pc=pc))
    path.chmod(path.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")


def _sample(pre=0.2, region=0.2):
    s = bench.ClockSampler(0)
    s.__enter__()
    time.sleep(pre)
    s.mark_start()
    time.sleep(region)
    s.mark_end()
    s.__exit__()
    return s.summary()


def test_samples_reasons_and_timed_window(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    out = _sample()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] >= 5 and 1 <= out["samples_in_timed_region"] < out["samples"]


def test_hardware_slowdown_is_reported(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch, sm=1200, hw="Active", pc="Not Active")
    out = _sample(0.1, 0.1)
    assert out["sm_mhz"] == 1200.0 and out["reasons"] == ["hw_slowdown"]


def test_without_marks_no_window_is_claimed(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    s = bench.ClockSampler(0)
    s.__enter__()
    time.sleep(0.15)
    s.__exit__()
    out = s.summary()
    assert out["samples"] >= 1 and "samples_in_timed_region" not in out


def test_missing_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    out = _sample(0.05, 0.05)
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}


def test_preroll_replays_for_its_duration_and_synchronises():
    calls, syncs = [], []
    t0 = time.perf_counter()
    n = bench.preroll(lambda i: (calls.append(i), time.sleep(0.001)), seconds=0.1, sync=lambda: syncs.append(1))
    dt = time.perf_counter() - t0
    assert 0.1 <= dt < 0.5
    assert n == len(calls) and calls == list(range(n)) and n >= 16
    assert len(syncs) == n // 16 + 1        # every 16 replays, and once at the end
