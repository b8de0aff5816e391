"""Host-side helpers of the benchmark (no device work).

The roofline's denominator comes from MEASURED_PEAKS.json when it is present:
top-level or nested, as a number or a {"value": ...} record; anything else
falls back to the stated fallback figure.
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("record,want", [
    (None, (bench.FALLBACK_HBM_GBS, "fallback")),
    ({"hbm_gbs": 7123.5, "bf16_tflops": 1900}, (7123.5, "measured")),
    ({"hbm_gbs": {"value": 7000, "unit": "GB/s"}}, (7000.0, "measured")),
    ({"gb300": {"hbm_gbs": 6950}}, (6950.0, "measured")),
    ({"hbm_gbs": "n/a", "pool": {"hbm_copy_gbs": 7010}}, (7010.0, "measured")),
    ({"bf16_tflops": 1900}, (bench.FALLBACK_HBM_GBS, "fallback")),
    ({"hbm_gbs": 0}, (bench.FALLBACK_HBM_GBS, "fallback")),
    ("not json", (bench.FALLBACK_HBM_GBS, "fallback")),
])
def test_measured_peak_hbm(tmp_path, monkeypatch, record, want):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    if record is not None:
        text = record if isinstance(record, str) else json.dumps(record)
        (tmp_path / "MEASURED_PEAKS.json").write_text(text)
    assert bench.measured_peak_hbm() == want


def _fake_smi(tmp_path, body):
    d = tmp_path / "bin"
    d.mkdir()
    f = d / "nvidia-smi"
    f.write_text("#!/bin/sh\n" + body)
    f.chmod(0o755)
    return str(d)


def test_clock_sampler_reports_the_samples_around_the_timed_region(tmp_path, monkeypatch):
    # three throttled samples at 1000 MHz first (before the timed region), then 2070 MHz, no reason
    body = ("i=0\nwhile true; do\n"
            "  if [ $i -lt 3 ]; then echo '0, 1000, 2070, 900.0, Active, Active, Not Active, Not Active, Not Active';\n"
            "  else echo '0, 2070, 2070, 1100.0, Not Active, Not Active, Not Active, Not Active, Active'; fi\n"
            "  i=$((i+1)); sleep 0.05\ndone\n")
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, body) + os.pathsep + os.environ["PATH"])
    calls = []
    c = bench.ClockSampler(0)
    c.start()
    c.wait_samples(4, lambda: (calls.append(1), __import__("time").sleep(0.01)))
    c.mark()
    c.wait_samples(3, lambda: (calls.append(1), __import__("time").sleep(0.01)))
    info = c.stop()
    assert calls and info["samples"] >= 3
    assert info["sm_mhz"] == 2070.0 and info["sm_max_mhz"] == 2070.0
    assert info["reasons"] == ["sw_power_cap"]             # the earlier hw_slowdown samples are not counted


def test_clock_sampler_bounds(tmp_path, monkeypatch):
    import time
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, "exec sleep 30\n"))     # a sampler that never reports
    c = bench.ClockSampler(0)
    c.start()
    t0 = time.monotonic()
    c.wait_samples(1, lambda: time.sleep(0.01), timeout_s=0.3)
    assert time.monotonic() - t0 < 2.0
    c.wait_samples(1, lambda: 1 / 0, timeout_s=5.0)                    # a failing busy() ends the wait
    assert c.stop()["samples"] == 0
    monkeypatch.setenv("PATH", str(tmp_path / "nowhere"))
    c = bench.ClockSampler(0)
    c.start()
    c.wait_samples(5, lambda: 1 / 0)
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]
