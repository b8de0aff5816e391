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
