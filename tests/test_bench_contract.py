"""Host-side pieces of the benchmark: algorithmic byte counts per call (the
roofline's numerator) equal the per-row derivation for each workload, ncu
traffic records count only while their kernel family's sources are unchanged,
the roofline peaks come from the measured file (else the fallback), and the
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


def _fake_tree(root):
    csrc = root / "mxfp4_activation_quant_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("rmsq_rows.cuh", "rmsq_api.cu", "rmsq_gemm.cu", "rmsq_device.cuh", "notes.txt"):
        (csrc / f).write_text(f"// {f}\n")
    (root / "profiles").mkdir()
    return csrc


def _stamp(root, monkeypatch):
    import json
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec = {"prefill:rows": {"kernel_source_digest": bench.kernel_source_digest("rows"), "dram_bytes_per_launch": 11},
           "consumer:gemm": {"kernel_source_digest": bench.kernel_source_digest("gemm"), "dram_bytes_per_launch": 22}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_traffic_stamps_follow_their_own_sources(tmp_path, monkeypatch):
    """A capture stays valid while the sources of its kernel family are
    unchanged: a GEMM-only file voids the GEMM's record only, a file of the
    norm + quant kernels voids theirs only, a header both include voids both,
    and files that are not sources count for neither."""
    csrc = _fake_tree(tmp_path)
    _stamp(tmp_path, monkeypatch)
    assert bench.recorded_traffic("prefill:rows") == 11 and bench.recorded_traffic("consumer:gemm") == 22
    (csrc / "notes.txt").write_text("changed")
    assert bench.recorded_traffic("prefill:rows") == 11 and bench.recorded_traffic("consumer:gemm") == 22
    (csrc / "rmsq_gemm.cu").write_text("// changed\n")
    assert bench.recorded_traffic("prefill:rows") == 11 and bench.recorded_traffic("consumer:gemm") is None
    _stamp(tmp_path, monkeypatch)
    (csrc / "rmsq_rows.cuh").write_text("// changed\n")
    assert bench.recorded_traffic("prefill:rows") is None and bench.recorded_traffic("consumer:gemm") == 22
    _stamp(tmp_path, monkeypatch)
    (csrc / "rmsq_device.cuh").write_text("// changed\n")
    assert bench.recorded_traffic("prefill:rows") is None and bench.recorded_traffic("consumer:gemm") is None
    assert bench.recorded_traffic("no:such") is None


def test_fp4_peak_is_the_bf16_rate_times_six(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 1.0, "bf16_tflops": 1800.0}')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_fp4_peak()[0] == 10800.0
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    # no measured file: the bf16 GEMM is measured on the device instead
    monkeypatch.setattr(bench, "bf16_gemm_tflops", lambda dev: 1500.0)
    peak, how = bench.measured_fp4_peak("cuda:0")
    assert peak == 9000.0 and "measured here" in how
    assert bench.measured_fp4_peak()[0] is None


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the CPU oracle, timed on the full headline
    workload) prints one JSON line with the headline's metric and unit, its own
    cpu_baseline and an e2e block that moves nothing between host and device."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["metric"] == bench.METRIC and rec["unit"] == "GB/s"
    assert rec["steps"] == 1 and rec["warmup"] == 3 and rec["n_gpus"] == 1 and rec["value"] > 0
    # the headline's own workload, all rows, described exactly as our arm describes it
    assert rec["config"] == bench.workload_config(bench.WORKLOAD, 16384, 1, bench.algorithmic_bytes(16384, 7168))
    cb = rec["cpu_baseline"]
    assert "all 16384 rows" in cb["sample"]
    assert cb["kind"] == "oracle" and cb["value"] == rec["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = rec["e2e"]
    assert e2e["value"] == rec["value"] and e2e["unit"] == rec["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_measured_peak_is_read(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 1234.5}')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (1234.5, "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    # no measured file: the library's own copy kernel is timed on the device;
    # there is no hard-coded figure to fall back to
    monkeypatch.setattr(bench, "copy_peak_gbs", lambda dev: 4321.0)
    peak, how = bench.measured_peaks("cuda:0")
    assert peak == 4321.0 and "copy kernel" in how
    assert bench.measured_peaks()[0] is None
    assert not hasattr(bench, "FALLBACK_HBM_GBS")


def test_restamped_traffic_records_do_not_count(tmp_path, monkeypatch):
    """A record whose digest was re-keyed by hand after the sources changed
    (marked restamped*) is not a capture of the code that runs."""
    import json
    _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"prefill:rows": {"kernel_source_digest": bench.kernel_source_digest("rows"), "dram_bytes_per_launch": 11,
                            "restamped_host_only": "host code changed after the capture"}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("prefill:rows") is None


def test_bench_variants_name_their_layout():
    assert bench.VARIANTS == {"prefill_col": ("prefill", "col"), "prefill_col_pad4": ("prefill", "col_pad4")}
    for name in bench.VARIANTS:
        assert "column-major" in bench.WORKLOAD_TEXT[name]


def test_parity_verdict_applies_the_bar():
    ok = {"rows": 4, "boundary_rows": 0, "codes_differing": 0, "mismatch_fraction": 0.0, "max_code_ulp": 0,
          "codes_bit_exact_outside_boundary": True, "residual_out_bit_exact": True, "scale_max_rel": 0.0,
          "scales_bit_exact_outside_boundary": True}
    assert bench._verdict(ok)["passes"]
    assert not bench._verdict({**ok, "max_code_ulp": 2})["passes"]
    assert not bench._verdict({**ok, "mismatch_fraction": 2e-3})["passes"]
    assert not bench._verdict({**ok, "residual_out_bit_exact": False})["passes"]
    assert not bench._verdict({**ok, "scale_max_rel": 1e-4})["passes"]


def _ncu_csv(path, kernel, launches):
    head = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
            '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')
    rows = ["==PROF== Connected to process 1", head]
    for i, (rd, wr, ns) in enumerate(launches):
        for name, unit, v in (("dram__bytes_read.sum", "Mbyte", rd), ("dram__bytes_write.sum", "byte", wr),
                              ("gpu__time_duration.sum", "ns", ns)):
            rows.append(f'"{i}","1","python3","h","{kernel}","1","7","(224, 1, 1)","(16384, 1, 1)","0","10.3",'
                        f'"Command line profiler metrics","{name}","{unit}","{v}"')
    path.write_text("\n".join(rows) + "\n")


def test_traffic_ingest_takes_the_digest_of_the_run(tmp_path, monkeypatch):
    """A capture is recorded with the digest the captured bench.py run printed,
    and only if that is the digest of the sources here."""
    import json
    import pytest
    _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _ncu_csv(tmp_path / "c.csv", "void rows_kernel<4, 224, 0, 0>(LaunchParams)",
             [(470.5, 590000000, 158000), (471.5, 590000000, 158500)])
    line = {"config": {"workload": "prefill", "bytes_per_step": 1060648960},
            "source_digest": {"rows": bench.kernel_source_digest("rows"), "gemm": "x"}}
    (tmp_path / "b.json").write_text("noise\n" + json.dumps(line) + "\n")
    ent = bench.ingest_traffic("prefill:rows", str(tmp_path / "c.csv"), str(tmp_path / "b.json"), "ncu ...")
    assert ent["dram_bytes_each_launch"] == [1060500000, 1061500000]
    assert ent["dram_bytes_per_launch"] == 1061000000
    assert bench.recorded_traffic("prefill:rows") == 1061000000
    line["source_digest"]["rows"] = "0" * 16
    (tmp_path / "b.json").write_text(json.dumps(line) + "\n")
    with pytest.raises(SystemExit, match="sources"):
        bench.ingest_traffic("prefill:rows", str(tmp_path / "c.csv"), str(tmp_path / "b.json"), "ncu ...")
