#!/usr/bin/env python
"""Benchmark of the fused residual add + RMSNorm + 1x128 FP8 quantisation.

Workload (one "step" = one call of the fused kernel): M=16384 rows, H=7168,
bf16 x and residual, gamma, eps 1e-6, keep_bf16 on; outputs E4M3 codes,
fp32 scales [M, 56], the bf16 residual and the bf16 normalised y. Inputs are
the seeded synthetic prefill workload (DeepSeek-V3/R1 hidden size, 1 % outlier
channels x20, residual N(0,4)); they are 470 MB, larger than the 129 MB L2, so
every step streams from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]

Prints one JSON line. ``value`` is HBM GB/s of algorithmic bytes (every byte
the method must read or write once, gamma counted once per call) over the
device time of K back-to-back launches with inputs resident in HBM; under
torchrun each rank runs its own batch (weak scaling) and the time is the max
over ranks. ``e2e`` is the same metric measured through the public API with
pinned host buffers, the host->device copy of x / residual / gamma and the
device->host copy of every output inside the timed region; the rows are cut
into chunks whose copies and calls are pipelined over three streams (rows are
independent, so this is exact). ``roofline``
relates the kernel's achieved GB/s to the measured HBM copy peak.
``--impl reference`` times the CPU oracle (test infrastructure, plain C)
on the host cores on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HBM GB/s (% of peak) & rows/s, fused add+RMSNorm+1x128 FP8 quant, M=16384 H=7168"
WORKLOAD = "prefill"
# bench-only variants of the prefill workload: the decode config's
# column-major scale layouts at the prefill size
VARIANTS = {"prefill_col": ("prefill", "col"), "prefill_col_pad4": ("prefill", "col_pad4")}


def algorithmic_bytes(M: int, H: int, residual: bool = True, keep_bf16: bool = True) -> int:
    per_row = 2 * H                      # read x
    if residual:
        per_row += 2 * H + 2 * H         # read residual, write residual_out
    if keep_bf16:
        per_row += 2 * H                 # write y
    per_row += H + 4 * (H // 128)        # write E4M3 codes and fp32 scales
    return M * per_row + 2 * H           # gamma once per call


def mx_bytes(M: int, H: int) -> int:
    return M * (2 * H + 2 * H + 2 * H + H // 2 + H // 32) + 2 * H


def qk_bytes(M: int, Hq: int, Hkv: int) -> int:
    return sum(M * (2 * h + h + 4 * (h // 128)) + 2 * h for h in (Hq, Hkv))


def copy_peak_gbs(dev) -> float:
    """Read + write GB/s of the library's own streaming copy kernel (rmsq_copy)
    over 1 GiB, best of 10 (CUDA events): the HBM peak where no separately
    measured one is recorded."""
    import torch
    from mxfp4_activation_quant_gb300 import rmsq
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, device=dev).fill_(1)
    dst = torch.empty_like(src)
    best = float("inf")
    for _ in range(12):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        rmsq.copy_(dst, src)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del src, dst
    return round(2 * n / (best * 1e-3) / 1e9, 1)


def measured_peaks(dev=None) -> tuple[float | None, str]:
    """The HBM peak: the measured copy rate in MEASURED_PEAKS.json, else
    the rate of the library's own copy kernel measured now on `dev`."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        if dev is None:
            return None, "unavailable: no MEASURED_PEAKS.json and no device to measure on"
        return copy_peak_gbs(dev), "measured here: the library's copy kernel, 1 GiB read + written, best of 10"


# Dense FP4 (E2M1) tensor rate over dense bf16 on GB300, from the nominal
# figures (13.5 and 2.25 PFLOP/s); the measured bf16 GEMM rate times this is
# the FP4 roofline.
FP4_OVER_BF16 = 6.0


def bf16_gemm_tflops(dev) -> float:
    """cuBLAS bf16 GEMM rate (torch.matmul, 8192^3, best of 10), as the
    driver measures it, for boxes without MEASURED_PEAKS.json."""
    import torch
    n = 8192
    a = torch.randn((n, n), device=dev).to(torch.bfloat16)
    b = torch.randn((n, n), device=dev).to(torch.bfloat16)
    best = float("inf")
    for _ in range(12):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def measured_fp4_peak(dev=None) -> tuple[float | None, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            bf16 = float(json.load(fh)["bf16_tflops"])
        return bf16 * FP4_OVER_BF16, "measured bf16 burst x nominal fp4/bf16 ratio 6"
    except (OSError, KeyError, ValueError):
        if dev is None:
            return None, "unavailable: no MEASURED_PEAKS.json and no device to measure on"
        return (round(bf16_gemm_tflops(dev) * FP4_OVER_BF16, 1),
                "bf16 GEMM measured here (8192^3, best of 10) x nominal fp4/bf16 ratio 6")


# the GEMM's own files (left out of the norm + quant digest) and the shared headers it also uses
GEMM_ONLY = ("rmsq_gemm.cu", "rmsq_gemm_pair.cu", "rmsq_gemm_common.cuh")
GEMM_SOURCES = GEMM_ONLY + ("rmsq_device.cuh", "rmsq_internal.h")


def kernel_source_digest(kind: str = "rows") -> str:
    """Hash of the sources a kernel family is built from: the GEMM's own
    files for "gemm", everything but the GEMM for the norm + quant kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_activation_quant_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h")):
            continue
        if (kind == "gemm" and f not in GEMM_SOURCES) or (kind == "rows" and f in GEMM_ONLY):
            continue
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_name: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; otherwise None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel_name)
    kind = "gemm" if kernel_name.startswith("consumer") else "rows"
    if not ent or ent.get("kernel_source_digest") != kernel_source_digest(kind):
        return None
    if any(k.startswith("restamped") for k in ent):      # a digest re-keyed by hand is no capture
        return None
    return float(ent["dram_bytes_per_launch"])


_NCU_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
              "ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6, "nsecond": 1}


def ncu_launches(csv_path: str) -> list[dict]:
    """Per-launch DRAM bytes and duration from an ncu --csv metrics log
    (dram__bytes_read.sum, dram__bytes_write.sum, gpu__time_duration.sum)."""
    import csv
    with open(csv_path) as fh:
        lines = [ln for ln in fh if ln.startswith('"')]
    rows = list(csv.reader(lines))
    head, body = rows[0], rows[1:]
    col = {name: i for i, name in enumerate(head)}
    launches: dict[str, dict] = {}
    for r in body:
        ent = launches.setdefault(r[col["ID"]], {"kernel": r[col["Kernel Name"]]})
        value = float(r[col["Metric Value"]].replace(",", "")) * _NCU_UNITS[r[col["Metric Unit"]]]
        ent[r[col["Metric Name"]]] = value
    out = []
    for ident in sorted(launches, key=int):
        e = launches[ident]
        out.append({"kernel": e["kernel"],
                    "dram_bytes": int(e["dram__bytes_read.sum"] + e["dram__bytes_write.sum"]),
                    "ns": e.get("gpu__time_duration.sum")})
    return out


def ingest_traffic(key: str, csv_path: str, bench_log: str, command: str) -> dict:
    """Writes the steady-state DRAM traffic of one kernel into
    profiles/traffic.json from a capture: the ncu metrics log of `command`
    (which ran bench.py) and that bench.py run's own JSON line, whose
    source_digest says which kernel sources ran. Refuses a capture taken on
    sources other than the ones here."""
    kind = "gemm" if key.startswith("consumer") else "rows"
    with open(bench_log) as fh:
        line = json.loads([ln for ln in fh if ln.startswith("{")][-1])
    ran = line["source_digest"][kind]
    if ran != kernel_source_digest(kind):
        raise SystemExit(f"the capture ran {kind} sources {ran}, these are {kernel_source_digest(kind)}")
    launches = ncu_launches(csv_path)
    if not launches:
        raise SystemExit("no launches in the capture")
    per = [ln_["dram_bytes"] for ln_ in launches]
    ent = {"kernel": launches[0]["kernel"], "kernel_source_digest": ran,
           "captured_workload": line["config"]["workload"],
           "dram_bytes_per_launch": int(round(statistics.mean(per))),
           "dram_bytes_each_launch": per,
           "ns_each_launch": [ln_["ns"] for ln_ in launches],
           "algorithmic_bytes_per_launch": line["config"]["bytes_per_step"],
           "command": command,
           "reading": ("launches in their back-to-back state (--cache-control none): the previous launch's "
                       "outputs still dirty in L2 are written back inside this one, as in the timed steps")}
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        rec = {}
    rec["about"] = ("DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch, steady state, from "
                    "ncu metric captures on GB300 with --clock-control none, written by `bench.py "
                    "--ingest-traffic` from the capture's CSV and the captured bench.py run's own line; valid "
                    "only while the kernel family's sources hash to kernel_source_digest")
    rec[key] = ent
    with open(path, "w") as fh:
        json.dump(rec, fh, indent=1)
        fh.write("\n")
    return ent


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", gpu_id], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [ln.split(", ") for ln in self.file.read().strip().splitlines() if ln.count(",") >= 8]
        self.file.close()
        os.unlink(self.file.name)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def gpu_id_for(dev) -> str:
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[dev.index or 0]


# ------------------------------------------------------------ reference arm

def workload_config(name: str, M: int, world: int, bytes_step: int) -> dict:
    """The ``config`` block of a line: what the workload is, nothing about the
    arm that ran it (both arms print the same block for the same workload)."""
    return {"workload": WORKLOAD_TEXT[name].format(M=M), "global_rows": M * world,
            "parallelism": f"rows sharded, {world} independent batch(es)", "bytes_per_step": bytes_step,
            "l2": ("inputs larger than L2 (129 MB); no flush needed" if bytes_step > 400e6 else
                   "inputs smaller than L2: back-to-back steps are partly L2-resident")}


def run_reference(args) -> None:
    """The CPU oracle as it stands, on the host cores, on the full headline
    workload: every step is one pass over all 16384 rows (about 0.1 s on 16
    cores), so the line's config is the headline's own."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from mxfp4_activation_quant_gb300 import synth
    from oracle import oracle

    w = synth.WORKLOADS[WORKLOAD]
    d = synth.make_inputs(w)
    x, r, g = oracle.as_u16(d["x"]), oracle.as_u16(d["residual"]), oracle.as_u16(d["gamma"])
    rows = x.shape[0]
    cores = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.add_rmsnorm_quant_fp8(x, r, g, w.eps, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.add_rmsnorm_quant_fp8(x, r, g, w.eps, nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    b = algorithmic_bytes(rows, w.H)
    value = b / dt / 1e9
    sample = f"all {rows} rows of the prefill workload per step (H={w.H}, keep_bf16)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64/f32", "data": "synthetic",
        "config": workload_config(WORKLOAD, rows, 1, b),
        "timing": "wall clock of K oracle passes on the host cores",
        "rows_per_s": round(rows / dt, 1),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def cpu_baseline(d_cpu, w) -> tuple[dict, dict]:
    """The oracle timed on the host cores on the full prefill workload (3
    passes). Returns the timing and the oracle's outputs of the last pass,
    against which the GPU's outputs of the same inputs are compared."""
    from oracle import oracle
    x, r, g = oracle.as_u16(d_cpu["x"]), oracle.as_u16(d_cpu["residual"]), oracle.as_u16(d_cpu["gamma"])
    cores = oracle.default_threads()
    oracle.add_rmsnorm_quant_fp8(x[:64], r[:64], g, w.eps, nthreads=cores)
    passes = 3
    t0 = time.perf_counter()
    for _ in range(passes):
        ref = oracle.add_rmsnorm_quant_fp8(x, r, g, w.eps, nthreads=cores)
    dt = (time.perf_counter() - t0) / passes
    M = x.shape[0]
    # one thread, on the first 1024 rows (about a second)
    n1 = min(M, 1024)
    t0 = time.perf_counter()
    oracle.add_rmsnorm_quant_fp8(x[:n1], r[:n1], g, w.eps, nthreads=1)
    dt1 = time.perf_counter() - t0
    return ({"value": round(algorithmic_bytes(M, w.H) / dt / 1e9, 3), "unit": "GB/s", "cores": cores,
             "kind": "oracle", "sample": f"all {M} rows of the prefill workload, {passes} passes",
             "rows_per_s": round(M / dt, 1), "ms_per_pass": round(dt * 1e3, 2),
             "one_thread": {"value": round(algorithmic_bytes(n1, w.H) / dt1 / 1e9, 3), "unit": "GB/s",
                            "rows_per_s": round(n1 / dt1, 1), "sample": f"first {n1} rows"}}, ref)


PARITY_RULE = ("residual_out and bf16 y bit-exact; scales within 1e-5 relative; every code within 1 ULP; "
               "at most 0.1 % of codes differing. Rows whose fp64 inv_rms lies within 2^-40 of an fp32 "
               "rounding boundary (boundary_rows) may round the other way; everywhere else every output "
               "must be bit-exact")


def _verdict(st: dict) -> dict:
    """The parity bar applied to one call's figures (tests/parity.py's rule)."""
    ok = (st.get("residual_out_bit_exact", True) and st.get("y_bit_exact_outside_boundary", True)
          and st["max_code_ulp"] <= 1 and st["mismatch_fraction"] <= 1e-3
          and st["codes_bit_exact_outside_boundary"] and st.get("scale_max_rel", 0.0) <= 1e-5
          and st.get("scales_bit_exact_outside_boundary", True) and st.get("scale_max_step", 0) <= 1)
    return {**st, "passes": bool(ok)}


def parity_report(gpu: dict, prefill_ref: dict) -> dict:
    """Part of the CPU-baseline leg: the GPU outputs of every config (0-4)
    against the oracle run on the same inputs, all rows, with the mismatch
    fraction of the codes. ``gpu`` maps a config name to (workload, CPU
    inputs, GPU outputs copied to the host); the prefill oracle outputs come
    from the timed CPU baseline."""
    from oracle import oracle
    from tests import parity
    out = {"rule": PARITY_RULE, "oracle_cores": oracle.default_threads()}
    for name, (w, d, got) in gpu.items():
        t0 = time.perf_counter()
        if name == "prefill":
            out[name] = _verdict(parity.fp8_stats(got, prefill_ref, w.scale_layout))
        elif w.kind == "fp8":
            ref = oracle.add_rmsnorm_quant_fp8(d["x"], d.get("residual"), d["gamma"], w.eps,
                                               layout=w.scale_layout)
            oracle_ms = (time.perf_counter() - t0) * 1e3
            out[name] = _verdict(parity.fp8_stats(got, ref, w.scale_layout))
            out[name]["oracle_ms"] = round(oracle_ms, 3)
        elif w.kind == "qknorm":
            ref = oracle.qknorm_quant_fp8(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], w.eps)
            oracle_ms = (time.perf_counter() - t0) * 1e3
            a = _verdict(parity.fp8_stats(got["q_a"], ref["q"]))
            b = _verdict(parity.fp8_stats(got["kv_a"], ref["kv"]))
            codes = got["q_a"]["q"].numel() + got["kv_a"]["q"].numel()
            out[name] = {"q_a": a, "kv_a": b, "rows": a["rows"],
                         "boundary_rows": a["boundary_rows"] + b["boundary_rows"],
                         "codes_differing": a["codes_differing"] + b["codes_differing"],
                         "mismatch_fraction": (a["codes_differing"] + b["codes_differing"]) / codes,
                         "passes": a["passes"] and b["passes"], "oracle_ms": round(oracle_ms, 3)}
        else:
            ref = oracle.add_rmsnorm_quant_mxfp4(d["x"], d.get("residual"), d["gamma"], w.eps)
            oracle_ms = (time.perf_counter() - t0) * 1e3
            out[name] = _verdict(parity.mx_stats(got, ref))
            out[name]["oracle_ms"] = round(oracle_ms, 3)
    out["all_pass"] = all(v["passes"] for k, v in out.items() if isinstance(v, dict))
    return out


# -------------------------------------------------------------- our arm

def time_launches(fn, steps: int, stream) -> tuple[float, list[float]]:
    """Total ms of `steps` back-to-back calls and each call's ms (events on `stream`)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end), [a.elapsed_time(b) for a, b in evs]


class L2Flush:
    """Evicts L2 between timed calls by reading a 256 MB buffer (twice L2). The
    lines it leaves behind are clean, so the timed call that follows does not
    pay for writing back the flush's own data, as it would after a flush that
    writes (up to 129 MB of dirty lines)."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        self()                      # the fill's dirty lines are written back here, untimed

    def __call__(self):
        import torch
        self.total = self.buf.sum()
        # then keep the GPU busy (~0.1 ms spin) while the host enqueues the
        # timed call, so that the call's events do not measure host latency
        # (torch's private spin kernel; without it, a second read of the
        # buffer does the same)
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(200_000)
        else:
            self.total = self.buf.sum()


def time_launches_cold(fn, steps: int, stream, flush) -> tuple[float, list[float]]:
    """Each of `steps` calls timed alone (events on `stream`) after `flush()`
    has evicted L2 so that no input is L2-resident; returns the sum of the
    calls' ms and each call's ms."""
    import torch
    each = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        each.append(a.elapsed_time(b))
    return sum(each), each


def time_graph(fn, steps: int, stream) -> float:
    """Total ms of `steps` calls captured into one CUDA graph and replayed (the
    host-side cost of each call is paid once, at capture). `fn` must launch on
    `stream`, a non-default stream: capture happens there."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            fn()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g.replay()
        torch.cuda.synchronize()
        start.record(stream)
        g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    # a kernel node costs ~0.5 us of replay; far less per step means the calls
    # launched outside the capture and the graph is empty
    if not ms * 1e3 / steps > 0.1:
        raise RuntimeError("the captured graph ran no work: the calls did not launch on the capture stream")
    return ms


def _cold_us(fn, dev, calls: int = 50) -> float:
    """Median microseconds of `calls` calls, each timed alone (CUDA events)
    after L2 has been evicted by reading 256 MB (L2Flush), so no input is
    L2-resident."""
    import torch
    flush = L2Flush(dev)
    each = []
    for _ in range(calls):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        each.append(e0.elapsed_time(e1) * 1e3)
    del flush
    return statistics.median(each)


def _graph_us(fn, reps: int, timed: int = 7, warm_ms: float = 30.0) -> float:
    """Microseconds per call of fn() replayed from a CUDA graph of `reps` calls
    captured on torch's capture stream (warm L2 across calls): the graph is
    replayed for at least `warm_ms` first (the host-side capture leaves the GPU
    idle long enough for its clocks to drop), then the median of `timed`
    replays, each timed with events on the replay stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    t0 = time.perf_counter()
    while True:
        g.replay()
        torch.cuda.synchronize()
        if (time.perf_counter() - t0) * 1e3 >= warm_ms:
            break
    us = []
    for _ in range(timed):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        us.append(a.elapsed_time(b) * 1e3 / reps)
    return statistics.median(us)


def other_workloads(dev, stream, peak: float) -> tuple[dict, dict]:
    """Decode latency (M=64), the MLA latent pair, MXFP4 throughput and the
    tiny config, reported beside the headline. Returns the report and, per
    config, (workload, CPU inputs, GPU outputs on the host) for the parity
    report of the CPU-baseline leg."""
    import torch
    from mxfp4_activation_quant_gb300 import rmsq, synth

    out, gpu = {}, {}
    # tiny: M=4, H=256, row-major scales
    w = synth.WORKLOADS["tiny"]
    dc = synth.make_inputs(w)
    d = {k: v.to(dev) for k, v in dc.items()}
    (tq, ts), tr = rmsq.add_rmsnorm_quant_fp8(d["x"], d["gamma"], d["residual"], eps=w.eps)
    torch.cuda.synchronize()
    gpu["tiny"] = (w, dc, {"q": tq.cpu(), "scale": ts.cpu(), "residual_out": tr.cpu()})
    tiny_us = _graph_us(lambda: rmsq.add_rmsnorm_quant_fp8_into(d["x"], d["gamma"], d["residual"], tq, ts, tr,
                                                                eps=w.eps), 200)
    out["tiny_m4"] = {"us_per_call_graph_warm_l2": round(tiny_us, 3),
                      "GBps_graph_warm": round(algorithmic_bytes(w.M, w.H, True, False) / tiny_us / 1e3, 3)}

    # decode: M=64, H=7168, column-major scales; launch-free latency via a graph
    w = synth.WORKLOADS["decode"]
    dc = synth.make_inputs(w)
    d = {k: v.to(dev) for k, v in dc.items()}
    M, H = w.M, w.H
    q = torch.empty((M, H), dtype=torch.uint8, device=dev)
    s = torch.empty((H // 128, M), dtype=torch.float32, device=dev)
    ro = torch.empty((M, H), dtype=torch.bfloat16, device=dev)

    def dec():
        rmsq.add_rmsnorm_quant_fp8_into(d["x"], d["gamma"], d["residual"], q, s, ro, None, eps=w.eps,
                                        scale_layout="col")
    for _ in range(10):
        dec()
    torch.cuda.synchronize()
    gpu["decode"] = (w, dc, {"q": q.cpu(), "scale": s.cpu(), "residual_out": ro.cpu()})
    warm_us = _graph_us(dec, 200)
    out["decode_m64"] = {"us_per_call_graph_warm_l2": round(warm_us, 3),
                         "us_per_call_cold_l2_median": round(_cold_us(dec, dev), 3),
                         "GBps_graph_warm": round(algorithmic_bytes(M, H, True, False) / warm_us / 1e3, 1),
                         "form": "latency (one block per SM or fewer)"}

    # MLA q_a / kv_a latents, M=8192
    w = synth.WORKLOADS["qknorm"]
    dc = synth.make_inputs(w)
    d = {k: v.to(dev) for k, v in dc.items()}
    M = w.M
    qq = torch.empty((M, w.Hq), dtype=torch.uint8, device=dev)
    qs = torch.empty((M, w.Hq // 128), dtype=torch.float32, device=dev)
    kq = torch.empty((M, w.Hkv), dtype=torch.uint8, device=dev)
    ks = torch.empty((M, w.Hkv // 128), dtype=torch.float32, device=dev)

    def qk():
        rmsq.qknorm_quant_fp8_into(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], qq, qs, kq, ks, eps=w.eps)
    for _ in range(10):
        qk()
    torch.cuda.synchronize()
    gpu["qknorm"] = (w, dc, {"q_a": {"q": qq.cpu(), "scale": qs.cpu()}, "kv_a": {"q": kq.cpu(), "scale": ks.cpu()}})
    nb = qk_bytes(M, w.Hq, w.Hkv)
    us = _graph_us(qk, 50)
    cold = _cold_us(qk, dev)
    out["qknorm_m8192"] = {"us_per_call_graph": round(us, 3), "GBps": round(nb / us / 1e3, 1),
                           "note": "50.9 MB per call: mostly L2-resident across back-to-back calls",
                           "us_per_call_cold_l2_median": round(cold, 3),
                           "GBps_cold_l2": round(nb / cold / 1e3, 1),
                           "frac_of_hbm_peak_cold_l2": round(nb / cold / 1e3 / peak, 4) if peak else None}

    # the same pair at the decode config's 64 tokens (latency form of the pair)
    Md = synth.WORKLOADS["decode"].M
    dd = {k: v[:Md].contiguous() for k, v in d.items() if k in ("q_a", "kv_a")}
    dq, dqs = qq[:Md].contiguous(), qs[:Md].contiguous()
    dk, dks = kq[:Md].contiguous(), ks[:Md].contiguous()

    def qk_decode():
        rmsq.qknorm_quant_fp8_into(dd["q_a"], dd["kv_a"], d["gamma_q"], d["gamma_kv"], dq, dqs, dk, dks, eps=w.eps)
    for _ in range(10):
        qk_decode()
    torch.cuda.synchronize()
    us = _graph_us(qk_decode, 200)
    out["qknorm_m64"] = {"us_per_call_graph_warm_l2": round(us, 3), "GBps_graph_warm": round(qk_bytes(Md, w.Hq, w.Hkv) / us / 1e3, 1),
                         "form": "latency (one block per SM or fewer)"}

    # MXFP4, M=8192, H=7168
    w = synth.WORKLOADS["mxfp4"]
    dc = synth.make_inputs(w)
    d = {k: v.to(dev) for k, v in dc.items()}
    M, H = w.M, w.H
    mq = torch.empty((M, H // 2), dtype=torch.uint8, device=dev)
    ms = torch.empty((M, H // 32), dtype=torch.uint8, device=dev)
    mr = torch.empty((M, H), dtype=torch.bfloat16, device=dev)

    def mx(st=None):
        rmsq.add_rmsnorm_quant_mxfp4_into(d["x"], d["gamma"], d["residual"], mq, ms, mr, None, eps=w.eps,
                                          stream=st)
    for _ in range(5):
        mx()
    total, each = time_launches(mx, 50, stream)
    gpu["mxfp4"] = (w, dc, {"q": mq.cpu(), "scale": ms.cpu(), "residual_out": mr.cpu()})
    us = statistics.mean(each) * 1e3
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g_us = time_graph(lambda: mx(side.cuda_stream), 200, side) * 1e3 / 200
    stream.wait_stream(side)
    out["mxfp4_m8192"] = {"us_per_call_graph": round(g_us, 2), "GBps_graph": round(mx_bytes(M, H) / g_us / 1e3, 1),
                          "us_per_call_back_to_back": round(us, 2), "GBps_back_to_back": round(mx_bytes(M, H) / us / 1e3, 1)}
    out["quant_placement"] = consumer_placements(dev)
    return out, gpu


# The consumer of the input RMSNorm in the DeepSeek-V3 MLA block: the fused
# q_a + kv_a (+ rope) projection, 7168 -> 1536 + 576 = 2112 outputs.
CONSUMER_N, CONSUMER_K = 2112, 7168


def consumer_setup(dev, M: int):
    """Inputs and outputs of the two placements of the MXFP4 activation quant
    for M tokens: step functions (taking a stream handle) for the fused path,
    the prequant path and the GEMM alone."""
    import torch
    from mxfp4_activation_quant_gb300 import rmsq, synth
    K, N = CONSUMER_K, CONSUMER_N
    w = synth.Workload("consumer", "mxfp4", M=M, H=K, seed=41, group=32, x_dist="student_t3")
    d = {k: v.to(dev) for k, v in synth.make_inputs(w).items()}
    b_q, b_s = synth.mxfp4_weights(42, N, K)
    gb, tb = b_q.to(dev), rmsq.mx_scale_tiles(b_s.to(dev))
    q = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    st = torch.zeros(rmsq.mma_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    ro = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def quant(s):
        rmsq.add_rmsnorm_quant_mxfp4_mma_scales_into(d["x"], d["gamma"], d["residual"], q, st, ro, stream=s)

    def gemm(s):
        rmsq.mxfp4_gemm(q, st, gb, tb, out=D, stream=s)

    def norm(s):
        rmsq.add_rmsnorm(d["x"], d["gamma"], d["residual"], out=y, out_residual=ro, stream=s)

    def pre(s):
        rmsq.a16wfp4_gemm(y, gb, tb, out=D, stream=s)

    return {"fused": lambda s: (quant(s), gemm(s)), "prequant": lambda s: (norm(s), pre(s)),
            "quant": quant, "gemm": gemm, "norm": norm, "prequant_gemm": pre}


def time_on_side_stream(dev, fn, reps: int) -> float:
    """Microseconds per call of fn(stream_handle), replayed from a CUDA graph of
    `reps` calls on a side stream (launch-free, as a serving step would run)."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            fn(side.cuda_stream)
    torch.cuda.synchronize()
    return time_graph(lambda: fn(side.cuda_stream), reps, side) * 1e3 / reps


def consumer_placements(dev, Ms=(4, 64, 8192)) -> dict:
    """Fused norm + MXFP4 quant followed by the block-scaled GEMM, against the
    norm alone followed by the GEMM that quantises its bf16 input itself
    ("prequant"): microseconds per step for each token count, and the GEMM's
    own time and tensor throughput."""
    from mxfp4_activation_quant_gb300 import rmsq
    out = {"shape": f"tokens x 7168 (residual add + RMSNorm) -> MXFP4 -> x [{CONSUMER_N}, {CONSUMER_K}]^T "
                    "MXFP4 weights, bf16 out",
           "timing": "CUDA graph replay, inputs partly L2-resident across calls"}
    for M in Ms:
        f = consumer_setup(dev, M)
        reps = 20 if M >= 4096 else 100
        r = {k: round(time_on_side_stream(dev, fn, reps), 2) for k, fn in f.items()}
        r["gemm_tflops"] = round(2.0 * M * CONSUMER_N * CONSUMER_K / r["gemm"] / 1e6, 1)
        r["faster"] = "fused" if r["fused"] <= r["prequant"] else "prequant"
        out[f"M{M}"] = r
        if rmsq.sync_status(dev) != 0:
            raise RuntimeError("a GEMM kernel reported a timed-out wait")
    return out


def rank_workload(w, rank: int):
    """Each rank draws its own batch of the same workload (seed + 1000 * rank)."""
    from mxfp4_activation_quant_gb300 import synth
    return synth.Workload(**{**w.__dict__, "seed": w.seed + 1000 * rank})


def make_step(name: str, dev, rank: int, rows: int, opts):
    """Inputs, outputs and a launcher of one workload.

    Returns (run, nbytes, M, inputs, outputs, w, d_cpu, chunkable, outs):
    ``run(r0, r1, stream)`` calls the library on rows [r0, r1) on ``stream``;
    inputs and outputs are (device tensor, pinned host tensor, row-indexed)
    triples for the end-to-end leg; ``chunkable`` says whether every per-row
    tensor is row-major (so a row range is a contiguous slice); ``outs`` are
    the device outputs by name."""
    import torch
    from mxfp4_activation_quant_gb300 import rmsq, synth

    if name in VARIANTS:
        base, layout = VARIANTS[name]
        w = synth.Workload(**{**synth.WORKLOADS[base].__dict__, "name": name, "scale_layout": layout})
    else:
        w = synth.WORKLOADS[name]
    if rows:
        w = synth.Workload(**{**w.__dict__, "M": rows})
    wr = rank_workload(w, rank)
    d_cpu = synth.make_inputs(wr)
    d = {k: v.to(dev) for k, v in d_cpu.items()}
    M = w.M
    chunkable = True
    if w.kind == "qknorm":
        outs = {"qq": torch.empty((M, w.Hq), dtype=torch.uint8, device=dev),
                "qs": torch.empty((M, w.Hq // 128), dtype=torch.float32, device=dev),
                "kq": torch.empty((M, w.Hkv), dtype=torch.uint8, device=dev),
                "ks": torch.empty((M, w.Hkv // 128), dtype=torch.float32, device=dev)}

        def run(r0, r1, st):
            o = {k: v[r0:r1] for k, v in outs.items()}
            rmsq.qknorm_quant_fp8_into(d["q_a"][r0:r1], d["kv_a"][r0:r1], d["gamma_q"], d["gamma_kv"],
                                       o["qq"], o["qs"], o["kq"], o["ks"], eps=w.eps, stream=st)
        nbytes = qk_bytes(M, w.Hq, w.Hkv)
    elif w.kind == "mxfp4":
        outs = {"q": torch.empty((M, w.H // 2), dtype=torch.uint8, device=dev),
                "s": torch.empty((M, w.H // 32), dtype=torch.uint8, device=dev),
                "r": torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)}

        def run(r0, r1, st):
            rmsq.add_rmsnorm_quant_mxfp4_into(d["x"][r0:r1], d["gamma"], d["residual"][r0:r1], outs["q"][r0:r1],
                                              outs["s"][r0:r1], outs["r"][r0:r1], None, eps=w.eps, opts=opts,
                                              stream=st)
        nbytes = mx_bytes(M, w.H)
    else:
        col = w.scale_layout != "row"
        chunkable = not col
        outs = {"q": torch.empty((M, w.H), dtype=torch.uint8, device=dev),
                "s": torch.empty(rmsq.scale_shape(M, w.H, 128, rmsq._layout(w.scale_layout)), dtype=torch.float32,
                                 device=dev),
                "r": torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)}
        if w.keep_bf16:
            outs["y"] = torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)

        def run(r0, r1, st):
            sc = outs["s"] if col else outs["s"][r0:r1]
            y = outs["y"][r0:r1] if "y" in outs else None
            rmsq.add_rmsnorm_quant_fp8_into(d["x"][r0:r1], d["gamma"], d["residual"][r0:r1], outs["q"][r0:r1],
                                            sc, outs["r"][r0:r1], y, eps=w.eps, scale_layout=w.scale_layout,
                                            opts=opts, stream=st)
        nbytes = algorithmic_bytes(M, w.H, True, w.keep_bf16)
    inputs = [(d[k], d_cpu[k].pin_memory(), d[k].dim() == 2) for k in d]
    outputs = [(v, torch.empty(v.shape, dtype=v.dtype).pin_memory(), not (col_scales(w) and k == "s"))
               for k, v in outs.items()]
    return run, nbytes, M, inputs, outputs, w, d_cpu, chunkable, outs


def col_scales(w) -> bool:
    return w.kind == "fp8" and w.scale_layout != "row"


def make_e2e_step(run, M: int, inputs, outputs, chunks: int, dev):
    """One end-to-end step: host->device copies, the library call and the
    device->host copies for row chunks spread over three streams, so that
    copies in both directions overlap the kernels of other chunks."""
    import torch
    streams = [torch.cuda.current_stream(dev)] + [torch.cuda.Stream(dev) for _ in range(2)]
    bounds = [(M * i // chunks, M * (i + 1) // chunks) for i in range(chunks)]

    def step():
        s0 = streams[0]
        start = torch.cuda.Event()
        for dv, hv, per_row in inputs:
            if not per_row:
                with torch.cuda.stream(s0):
                    dv.copy_(hv, non_blocking=True)
        start.record(s0)
        for s in streams[1:]:
            s.wait_event(start)
        for c, (r0, r1) in enumerate(bounds):
            s = streams[c % len(streams)]
            with torch.cuda.stream(s):
                for dv, hv, per_row in inputs:
                    if per_row:
                        dv[r0:r1].copy_(hv[r0:r1], non_blocking=True)
                run(r0, r1, s.cuda_stream)
                for dv, hv, per_row in outputs:
                    if per_row:
                        hv[r0:r1].copy_(dv[r0:r1], non_blocking=True)
        for dv, hv, per_row in outputs:
            if not per_row:
                with torch.cuda.stream(streams[(len(bounds) - 1) % len(streams)]):
                    hv.copy_(dv, non_blocking=True)
        for s in streams[1:]:
            e = torch.cuda.Event()
            e.record(s)
            s0.wait_event(e)

    return step


def make_e2e_step_packed(w, d_cpu, M: int, chunks: int, dev):
    """End-to-end step of the FP8 prefill workload with each row chunk's
    inputs (x rows, then residual rows) contiguous in one pinned host buffer
    and its outputs (residual, y, E4M3 codes, scales) contiguous in another, so
    that a chunk moves with one host->device and one device->host copy; chunks
    rotate over three streams so that copies in both directions overlap the
    kernels of other chunks. Returns (step, h2d_bytes, d2h_bytes)."""
    import torch
    from mxfp4_activation_quant_gb300 import rmsq
    H, G = w.H, w.H // 128
    in_row, out_row = 4 * H, 4 * H + H + 4 * G
    bounds = [(M * i // chunks, M * (i + 1) // chunks) for i in range(chunks)]
    host_in = torch.empty(M * in_row, dtype=torch.uint8).pin_memory()
    xb = d_cpu["x"].contiguous().view(torch.uint8).view(M, 2 * H)
    rb = d_cpu["residual"].contiguous().view(torch.uint8).view(M, 2 * H)
    for r0, r1 in bounds:
        seg = host_in[r0 * in_row:r1 * in_row].view(2, r1 - r0, 2 * H)
        seg[0].copy_(xb[r0:r1])
        seg[1].copy_(rb[r0:r1])
    dev_in = torch.empty_like(host_in, device=dev)
    dev_out = torch.empty(M * out_row, dtype=torch.uint8, device=dev)
    host_out = torch.empty(M * out_row, dtype=torch.uint8).pin_memory()
    gamma_h = d_cpu["gamma"].contiguous().pin_memory()
    gamma_d = torch.empty_like(gamma_h, device=dev)
    streams = [torch.cuda.current_stream(dev)] + [torch.cuda.Stream(dev) for _ in range(2)]

    def views(r0, r1):
        n = r1 - r0
        i = dev_in[r0 * in_row:r1 * in_row]
        o = dev_out[r0 * out_row:r1 * out_row]
        bf = lambda t: t.view(torch.bfloat16).view(n, H)
        x, res = bf(i[:2 * H * n]), bf(i[2 * H * n:])
        ro, y = bf(o[:2 * H * n]), bf(o[2 * H * n:4 * H * n])
        q = o[4 * H * n:5 * H * n].view(n, H)
        sc = o[5 * H * n:].view(torch.float32).view(n, G)
        return x, res, ro, y, q, sc
    chunk_views = [views(r0, r1) for r0, r1 in bounds]

    def step():
        s0 = streams[0]
        with torch.cuda.stream(s0):
            gamma_d.copy_(gamma_h, non_blocking=True)
        start = torch.cuda.Event()
        start.record(s0)
        for s in streams[1:]:
            s.wait_event(start)
        for c, (r0, r1) in enumerate(bounds):
            s = streams[c % len(streams)]
            x, res, ro, y, q, sc = chunk_views[c]
            with torch.cuda.stream(s):
                dev_in[r0 * in_row:r1 * in_row].copy_(host_in[r0 * in_row:r1 * in_row], non_blocking=True)
                rmsq.add_rmsnorm_quant_fp8_into(x, gamma_d, res, q, sc, ro, y, eps=w.eps, stream=s.cuda_stream)
                host_out[r0 * out_row:r1 * out_row].copy_(dev_out[r0 * out_row:r1 * out_row], non_blocking=True)
        for s in streams[1:]:
            e = torch.cuda.Event()
            e.record(s)
            s0.wait_event(e)

    return step, host_in.numel() + gamma_h.numel() * 2, host_out.numel()


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    from mxfp4_activation_quant_gb300 import build as lib_build
    from mxfp4_activation_quant_gb300 import rmsq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib_build.build()
    rmsq.lib()

    kernel = {"auto": rmsq.KERNEL_AUTO, "rows": rmsq.KERNEL_ROWS, "persistent": rmsq.KERNEL_PERSISTENT}[args.kernel]
    opts = rmsq.LaunchOpts(kernel=kernel) if kernel != rmsq.KERNEL_AUTO else None
    run, bytes_step, M, io_in, io_out, w, d_cpu, chunkable, outs = make_step(args.workload, dev, rank, args.rows,
                                                                             opts)
    stream = torch.cuda.current_stream(dev)

    def step():
        run(0, M, stream.cuda_stream)

    peak, peak_kind = measured_peaks(dev)
    sampler = ClockSampler(gpu_id_for(dev)) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # The K steps are replayed from one CUDA graph: the steps' host-side calls
    # and the events between them stay out of the timed region (a graph of K
    # launches runs the same kernels). --graph off times K back-to-back calls
    # with events around each instead; those numbers are also reported.
    use_graph = args.graph in ("on", "auto")
    back_to_back = None
    if use_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        total_ms = time_graph(lambda: run(0, M, side.cuda_stream), args.steps, side)
        stream.wait_stream(side)
        each_ms = [total_ms / args.steps]
        if args.workload not in ("decode", "qknorm"):      # launch-dominated steps have no meaningful per-call time
            k = min(args.steps, 500)
            b2b_ms, b2b_each = time_launches(step, k, stream)
            back_to_back = {"steps": k, "ms_per_step": round(b2b_ms / k, 5),
                            "value": round(world * bytes_step * k / (b2b_ms * 1e-3) / 1e9, 1),
                            "achieved_per_launch": round(bytes_step / (statistics.mean(b2b_each) * 1e-3) / 1e9, 1),
                            "timing": "K back-to-back calls, CUDA events around each"}
    else:
        total_ms, each_ms = time_launches(step, args.steps, stream)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    max_ms = max_over_ranks(total_ms, world, dev)
    value = world * bytes_step * args.steps / (max_ms * 1e-3) / 1e9
    launch_ms = statistics.mean(each_ms)
    achieved = bytes_step / (launch_ms * 1e-3) / 1e9

    # end to end through the public API: pinned host buffers, copies inside the
    # timed region, row chunks pipelined over three streams
    chunks = args.e2e_chunks if chunkable else 1
    packed = w.kind == "fp8" and w.scale_layout == "row" and w.keep_bf16 and w.residual and chunkable
    plain_step = make_e2e_step(run, M, io_in, io_out, chunks, dev)
    if packed:      # the headline workload: one copy each way per chunk
        e2e_step, h2d_packed, d2h_packed = make_e2e_step_packed(rank_workload(w, rank), d_cpu, M, chunks, dev)
    else:
        e2e_step = plain_step
    h2d = sum(hv.numel() * hv.element_size() for _, hv, _ in io_in)
    d2h = sum(hv.numel() * hv.element_size() for _, hv, _ in io_out)

    def time_e2e(fn):
        n = max(3, min(20, args.steps))
        for _ in range(2):
            fn()
        if world > 1:
            dist.barrier()
        ms, _ = time_launches(fn, n, stream)
        return round(world * bytes_step * n / (max_over_ranks(ms, world, dev) * 1e-3) / 1e9, 1)
    e2e = {"value": None, "unit": "GB/s", "h2d_bytes_per_step": h2d_packed if packed else h2d,
           "d2h_bytes_per_step": d2h_packed if packed else d2h, "row_chunks": chunks, "streams": 3}
    if not args.no_e2e:
        e2e["value"] = time_e2e(e2e_step)
    if packed:
        e2e["copies"] = "one each way per chunk"
        e2e["host_layout"] = ("chunk-packed pinned buffers: each chunk's x then residual rows in one buffer, its "
                              "outputs in another, arranged once before the timed region")
        e2e["plain"] = {"value": None if args.no_e2e else time_e2e(plain_step), "unit": "GB/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "copies": "one per tensor and chunk",
                        "host_layout": "plain [M, H] pinned tensors, as a caller holds them"}
    else:
        e2e["copies"] = "one per tensor and chunk"
        e2e["host_layout"] = "plain pinned tensors, as a caller holds them"

    headline = args.workload == WORKLOAD and not args.rows
    extra, gpu_out = (other_workloads(dev, stream, peak) if (rank == 0 and headline and not args.no_extra)
                      else (None, {}))
    cpu, parity = None, None
    if rank == 0 and world == 1 and headline and not args.no_cpu:
        # the CPU-baseline leg: the oracle timed on the host cores, and the
        # GPU's outputs of the timed steps compared with the oracle's
        cpu, ref = cpu_baseline(d_cpu, w)
        torch.cuda.synchronize()
        gpu_out["prefill"] = (w, d_cpu, {"q": outs["q"].cpu(), "scale": outs["s"].cpu(),
                                         "residual_out": outs["r"].cpu(), "y": outs["y"].cpu()})
        parity = parity_report({k: gpu_out[k] for k in ("tiny", "decode", "prefill", "qknorm", "mxfp4")
                                if k in gpu_out}, ref)
        del ref
    if world > 1:
        dist.barrier()
    if rank == 0:
        kernel_name = f"{args.workload}:{'bulk' if kernel == rmsq.KERNEL_PERSISTENT else 'rows'}"
        traffic = recorded_traffic(kernel_name)
        text_key = w.kind if w.kind != "fp8" else args.workload
        line = {
            "metric": METRIC if headline else f"HBM GB/s & rows/s, {args.workload} workload",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": workload_config(text_key, M, world, bytes_step),
            "kernel": args.kernel,
            "timing": "CUDA graph of the K steps" if use_graph else "K back-to-back calls",
            "rows_per_s": round(world * M * args.steps / (max_ms * 1e-3), 1),
            "pct_of_peak": round(100 * value / world / peak, 2) if peak else None,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4) if peak else None, "traffic": traffic,
                         "peak_kind": f"{peak_kind} HBM copy"},
            "mismatch_fraction": parity["prefill"]["mismatch_fraction"] if parity else None,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "parity": parity,
            "back_to_back": back_to_back,
            "other_workloads": extra,
            "source_digest": {"rows": kernel_source_digest("rows"), "gemm": kernel_source_digest("gemm")},
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_consumer(args) -> None:
    """--workload consumer: the block-scaled MXFP4 GEMM that consumes the fused
    quant's output, timed alone at M=8192 tokens (tensor roofline), with both
    placements of the quant reported beside it."""
    import torch

    from mxfp4_activation_quant_gb300 import build as lib_build
    from mxfp4_activation_quant_gb300 import rmsq, synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib_build.build()
    M, N, K = args.rows or 8192, CONSUMER_N, CONSUMER_K
    f = consumer_setup(dev, M)
    stream = torch.cuda.current_stream(dev)
    f["quant"](stream.cuda_stream)
    step = lambda: f["gemm"](stream.cuda_stream)
    sampler = ClockSampler(gpu_id_for(dev))
    time.sleep(0.25)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # The operands (37 MB) fit in L2: each timed call starts with L2 evicted
    # (256 MB read between calls, outside the events).
    flush = L2Flush(dev)
    total_ms, each = time_launches_cold(step, args.steps, stream, flush)
    del flush
    clocks = sampler.stop()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    warm_ms = time_graph(lambda: f["gemm"](side.cuda_stream), 200, side)
    stream.wait_stream(side)
    if rmsq.sync_status(dev) != 0:
        raise RuntimeError("the GEMM reported a timed-out wait")
    flops = 2.0 * M * N * K
    value = flops * args.steps / (total_ms * 1e-3) / 1e12
    achieved = flops / (statistics.mean(each) * 1e-3) / 1e12
    peak, peak_kind = measured_fp4_peak(dev)
    # end to end: A codes + scale tiles in from pinned host memory, D out
    a_q = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    a_t = torch.empty(rmsq.mma_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    (q, t), _ = rmsq.add_rmsnorm_quant_mxfp4_mma_scales(*[synth.make_inputs(synth.Workload(
        "consumer", "mxfp4", M=M, H=K, seed=41, group=32, x_dist="student_t3"))[k].to(dev)
        for k in ("x", "gamma", "residual")])
    hq, ht = q.cpu().pin_memory(), t.cpu().pin_memory()
    b_q, b_s = synth.mxfp4_weights(42, N, K)
    gb, tb = b_q.to(dev), rmsq.mx_scale_tiles(b_s.to(dev))
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    hD = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

    def e2e():
        a_q.copy_(hq, non_blocking=True)
        a_t.copy_(ht, non_blocking=True)
        rmsq.mxfp4_gemm(a_q, a_t, gb, tb, out=D)
        hD.copy_(D, non_blocking=True)
    for _ in range(2):
        e2e()
    e2e_steps = max(3, min(20, args.steps))
    e2e_ms, _ = time_launches(e2e, e2e_steps, stream)
    cpu = None
    if not args.no_cpu:
        from oracle import oracle
        rows = 8
        s_q, s_s = synth.mxfp4_weights(43, rows, K, 124, 131)     # activation-like MXFP4 rows
        t0 = time.perf_counter()
        oracle.mxfp4_gemm(s_q.numpy(), s_s.numpy(), b_q.numpy(), b_s.numpy())
        dt = time.perf_counter() - t0
        cpu = {"value": round(2.0 * rows * N * K / dt / 1e12, 6), "unit": "TFLOP/s",
               "cores": oracle.default_threads(), "kind": "oracle",
               "sample": f"{rows} of the {M} token rows x all {N} outputs (exact fp64 sums)"}
    line = {
        "metric": "block-scaled MXFP4 GEMM TFLOP/s (consumer of the fused quant)", "value": round(value, 1),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "source_digest": {"rows": kernel_source_digest("rows"), "gemm": kernel_source_digest("gemm")},
        "config": {"workload": f"D[{M},{N}] = A[{M},{K}] B[{N},{K}]^T, A and B MXFP4 (E2M1, E8M0 per 32), "
                               "bf16 out; A from the fused norm + quant", "M": M, "N": N, "K": K,
                   "bytes_per_step": (M + N) * K // 2 + rmsq.mma_scale_bytes(M, K) + rmsq.mma_scale_bytes(N, K)
                   + 2 * M * N,
                   "l2": "L2 evicted before each timed call by reading 256 MB (clean lines)",
                   "timing": "K calls, CUDA events around each, L2 evicted in between"},
        "warm_l2_graph": {"steps": 200, "ms_per_step": round(warm_ms / 200, 5),
                          "value": round(flops * 200 / (warm_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                          "timing": "CUDA graph of 200 calls, operands L2-resident"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("consumer:gemm"), "peak_kind": peak_kind},
        "e2e": {"value": round(flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": hq.numel() + ht.numel(), "d2h_bytes_per_step": hD.numel() * 2},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "quant_placement": None if args.no_extra else consumer_placements(dev),
    }
    print(json.dumps(line))


WORKLOAD_TEXT = {
    "prefill": "prefill input RMSNorm: M={M} H=7168 bf16, residual add, FP8 E4M3 1x128 groups, "
               "fp32 scales [M,56], keep_bf16 y",
    "prefill_col": "prefill input RMSNorm: M={M} H=7168 bf16, residual add, FP8 E4M3 1x128 groups, "
                   "fp32 scales column-major [56,M], keep_bf16 y",
    "prefill_col_pad4": "prefill input RMSNorm: M={M} H=7168 bf16, residual add, FP8 E4M3 1x128 groups, "
                        "fp32 scales column-major [56,M rounded up to 4], keep_bf16 y",
    "decode": "decode input RMSNorm: M={M} H=7168 bf16, residual add, FP8 E4M3 1x128, column-major scales",
    "qknorm": "MLA latents: q_a [M,1536] + kv_a [M,512], no residual, FP8 E4M3 1x128, one launch",
    "mxfp4": "input RMSNorm M={M} H=7168, residual add, MXFP4 (E8M0 per 32, E2M1 packed)",
}


def max_over_ranks(ms: float, world: int, dev) -> float:
    """The slowest rank's time (all ranks call this)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", choices=["auto", "rows", "persistent"], default="auto")
    ap.add_argument("--workload", choices=["prefill", "decode", "qknorm", "mxfp4", "consumer", *VARIANTS],
                    default=WORKLOAD,
                    help="the timed step (the headline line is prefill; consumer: the MXFP4 GEMM; prefill_col, "
                         "prefill_col_pad4: the prefill step with column-major scales)")
    ap.add_argument("--no-extra", action="store_true", help="skip the decode / qknorm / MXFP4 lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--e2e-chunks", type=int, default=24, help="row chunks pipelined in the e2e leg")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="replay the K timed steps from a CUDA graph (auto = on; off: back-to-back calls)")
    ap.add_argument("--rows", type=int, default=0,
                    help="rows of the batch (profiler captures only; the benchmark is M=16384)")
    ap.add_argument("--ingest-traffic", nargs=4, metavar=("KEY", "NCU_CSV", "BENCH_LOG", "COMMAND"),
                    help="record a steady-state DRAM traffic capture in profiles/traffic.json (no GPU needed)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.ingest_traffic:
        key, csv_path, log_path, command = args.ingest_traffic
        print(json.dumps(ingest_traffic(key, csv_path, log_path, command)))
    elif args.impl == "reference":
        run_reference(args)
    elif args.workload == "consumer":
        run_consumer(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
