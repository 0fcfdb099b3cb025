"""Host-side pieces of the benchmark: algorithmic byte counts per call (the
roofline's numerator) equal the per-row derivation for each workload, and the
JSON helpers behave without a GPU."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_algorithmic_bytes_per_workload():
    # prefill: read x, residual (2H each); write residual, y (2H each), E4M3 (H), scales (4H/128); gamma once
    assert bench.algorithmic_bytes(16384, 7168) == 16384 * 64736 + 14336 == 1060648960
    # decode: no keep_bf16
    assert bench.algorithmic_bytes(64, 7168, True, False) == 64 * 50400 + 14336 == 3239936
    # tiny
    assert bench.algorithmic_bytes(4, 256, True, False) == 7712
    # MLA pair: q_a 1536 and kv_a 512 rows, no residual, no y
    assert bench.qk_bytes(8192, 1536, 512) == 50860032
    # MXFP4: read x, residual; write residual, H/2 codes, H/32 scale bytes
    assert bench.mx_bytes(8192, 7168) == 383531008


def test_traffic_record_requires_current_sources(tmp_path, monkeypatch):
    assert len(bench.kernel_source_digest()) == 16
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("prefill:rows") is None


def test_measured_peak_is_read(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 1234.5}')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (1234.5, "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.measured_peaks()[1] == "fallback"
