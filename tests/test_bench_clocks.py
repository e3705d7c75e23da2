"""The bench's clock sampler on CPU: a stand-in `nvidia-smi` on PATH prints the
CSV rows the real query prints, and the sampler reports the median SM clock,
the maximum clock and every throttle reason it saw, then removes its file."""
import os
import stat
import sys

import bench

ROWS = [
    "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, 2055, 2070, 1210.4, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 2070, 2070, 1190.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "garbled line",
]


def _fake_smi(tmp_path, rows):
    script = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{r}'" for r in rows)
    script.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    script.chmod(script.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def test_clock_sampler_summarises_the_samples(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, ROWS) + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    s.start()
    assert s.proc is not None
    res = s.stop()
    assert res == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(s.path)


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # nothing to run
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop() is None


if sys.platform != "linux":  # the stand-in is a POSIX shell script
    import pytest
    pytestmark = pytest.mark.skip("needs /bin/sh")
