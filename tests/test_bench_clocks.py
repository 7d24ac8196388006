"""bench.py's clock sampler on the CPU, against a stand-in nvidia-smi.

The stand-in prints the sampler's nine CSV fields the way nvidia-smi's
``--format=csv,noheader,nounits`` does, alternating a power-capped sample at
1965 MHz with an unthrottled one at 2070 MHz, plus a malformed line the parser
must skip.  No GPU and no real nvidia-smi are involved.
"""

import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

FAKE = """#!/bin/sh
echo "garbage line"
while true; do
  echo "0, 1965, 2070, 901.20, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
  echo "0, 2070, 2070, 950.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
  sleep 0.02
done
"""


def _fake_path(tmp_path, body):
    d = tmp_path / "bin"
    d.mkdir()
    exe = d / "nvidia-smi"
    exe.write_text(body)
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(d)


def test_sampler_reads_clocks_and_reasons(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _fake_path(tmp_path, FAKE) + os.pathsep + os.environ.get("PATH", ""))
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.3)
    r = s.stop()
    assert r is not None and r["samples"] >= 4
    assert r["sm_max_mhz"] == 2070.0
    assert 1965.0 <= r["sm_mhz"] <= 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(s.path)


def test_sampler_flags_thermal_slowdown(tmp_path, monkeypatch):
    body = FAKE.replace("Not Active, Not Active, Not Active, Active",
                        "Active, Not Active, Active, Not Active")
    monkeypatch.setenv("PATH", _fake_path(tmp_path, body) + os.pathsep + os.environ.get("PATH", ""))
    s = bench.ClockSampler(0)
    s.start()
    time.sleep(0.2)
    r = s.stop()
    assert r["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    empty = tmp_path / "empty"
    empty.mkdir()
    monkeypatch.setenv("PATH", str(empty))
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop() is None
    assert not os.path.exists(s.path)
