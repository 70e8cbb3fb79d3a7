"""bench.py's clock sampler on CPU, against a stand-in nvidia-smi that prints fixed samples: the
parsing of clocks and throttle reasons, and a stop that is safe to repeat."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fake_smi(tmp_path, line):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(f'#!/bin/bash\nwhile true; do echo "{line}"; sleep 0.02; done\n')
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def test_samples_are_parsed_and_stop_is_idempotent(tmp_path, monkeypatch):
    d = _fake_smi(tmp_path, "0, 1980, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active")
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ.get("PATH", ""))
    c = bench.ClockSampler(0).__enter__()
    time.sleep(0.15)
    c.__exit__(None, None, None)
    c.__exit__(None, None, None)
    s = c.summary()
    assert s["sm_mhz"] == 1980.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] >= 2


def test_no_nvidia_smi_gives_no_summary(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # an empty directory: the tool is missing
    c = bench.ClockSampler(0).__enter__()
    c.__exit__(None, None, None)
    assert c.summary() is None
