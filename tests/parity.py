"""Comparison rules between the CUDA path and the CPU oracle.

The bar (per output of a call):
  * residual_out and the bf16 y: bit-exact;
  * scales: within 1e-5 relative;
  * codes: every code within 1 ULP of the oracle's (ordered magnitude, +0 and
    -0 equal) and at most 0.1 % of codes differing.

Rows whose fp64 inv_rms lies within 2^-40 (relative) of an fp32 rounding
boundary ("boundary rows", reported by the oracle's margin) are the only
place where a correct implementation may round inv_rms the other way; there
y may differ by one bf16 step and the codes and scale follow it. Everywhere
else the design is bit-exact, and the checks below assert exactly that.
"""

from __future__ import annotations

import numpy as np
import torch

BOUNDARY = 2.0 ** -40


def u8(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        return t.numpy()
    return np.asarray(t, dtype=np.uint8)


def u16(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.asarray(t, dtype=np.uint16)


def e4m3_ordinal(c: np.ndarray) -> np.ndarray:
    mag = (c & 0x7F).astype(np.int32)
    return np.where(c & 0x80, -mag, mag)


def e2m1_ordinal(c: np.ndarray) -> np.ndarray:
    mag = (c & 0x7).astype(np.int32)
    return np.where(c & 0x8, -mag, mag)


def bf16_ordinal(b: np.ndarray) -> np.ndarray:
    mag = (b & 0x7FFF).astype(np.int32)
    return np.where(b & 0x8000, -mag, mag)


def unpack_e2m1(q: np.ndarray) -> np.ndarray:
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def _boundary_rows(ref: dict, what: str) -> np.ndarray:
    """Rows the oracle flags as within 2^-40 of an fp32 rounding boundary of
    inv_rms. Such rows are rare (about 2^-16 of random rows); a comparison
    that would exempt more than a few is refused, so that a broken margin
    cannot weaken the checks."""
    boundary = ref["margin"] < BOUNDARY
    assert boundary.sum() <= max(2, len(boundary) // 1000), f"{what}: {boundary.sum()} boundary rows"
    return boundary


def _scale_array(s) -> np.ndarray:
    return s.detach().cpu().numpy() if isinstance(s, torch.Tensor) else np.asarray(s)


def fp8_stats(got: dict, ref: dict, scale_layout: str = "row") -> dict:
    """Every figure of the parity bar for an FP8 call, without judging it.

    got/ref: dicts with q (codes [M,H]), scale, optional y, residual_out (bf16
    bits). Returns the rows, boundary rows, codes differing and their
    fraction, the largest code distance in ULPs, the largest relative scale
    error, and whether residual_out, y, codes and scales are bit-exact
    outside boundary rows."""
    boundary = ref["margin"] < BOUNDARY
    ok_rows = ~boundary
    st = {"rows": int(len(boundary)), "boundary_rows": int(boundary.sum())}
    if "residual_out" in ref and got.get("residual_out") is not None:
        st["residual_out_bit_exact"] = bool(np.array_equal(u16(got["residual_out"]), ref["residual_out"]))
    if got.get("y") is not None:
        gy, ry = u16(got["y"]), ref["y"]
        st["y_bit_exact_outside_boundary"] = bool(np.array_equal(gy[ok_rows], ry[ok_rows]))
        st["y_max_step"] = int(np.abs(bf16_ordinal(gy) - bf16_ordinal(ry)).max(initial=0))
    gq, rq = u8(got["q"]), ref["q"]
    st["codes_differing"] = int((gq != rq).sum())
    st["mismatch_fraction"] = st["codes_differing"] / max(1, gq.size)
    st["max_code_ulp"] = int(np.abs(e4m3_ordinal(gq) - e4m3_ordinal(rq)).max(initial=0))
    st["codes_bit_exact_outside_boundary"] = bool(np.array_equal(gq[ok_rows], rq[ok_rows]))
    gs, rs = _scale_array(got["scale"]), ref["scale"]
    st["scale_shape_ok"] = gs.shape == rs.shape
    if st["scale_shape_ok"]:
        rel = np.abs(gs.astype(np.float64) - rs) / np.maximum(np.abs(rs.astype(np.float64)), 1e-30)
        st["scale_max_rel"] = float(rel.max(initial=0))
        gs_rows = gs if scale_layout == "row" else gs.T
        rs_rows = rs if scale_layout == "row" else rs.T
        st["scales_bit_exact_outside_boundary"] = bool(
            np.array_equal(gs_rows[ok_rows].view(np.uint32), rs_rows[ok_rows].view(np.uint32)))
    return st


def compare_fp8(got: dict, ref: dict, scale_layout: str = "row", what: str = "") -> dict:
    """got/ref: dicts with q (codes [M,H]), scale, optional y, residual_out (bf16 bits)."""
    _boundary_rows(ref, what)
    assert "residual_out" not in ref or got.get("residual_out") is not None, f"{what}: no residual_out"
    st = fp8_stats(got, ref, scale_layout)
    assert st.get("residual_out_bit_exact", True), f"{what}: residual_out differs"
    assert st.get("y_bit_exact_outside_boundary", True), f"{what}: bf16 y differs outside boundary rows"
    assert st.get("y_max_step", 0) <= 1, f"{what}: bf16 y off by > 1 step"
    assert st["max_code_ulp"] <= 1, f"{what}: a code is more than 1 ULP from the oracle"
    assert st["mismatch_fraction"] <= 1e-3, f"{what}: {st['mismatch_fraction']:.2e} of codes differ"
    assert st["codes_bit_exact_outside_boundary"], f"{what}: codes differ outside boundary rows"
    assert st["scale_shape_ok"], f"{what}: scale shape differs"
    assert st["scale_max_rel"] <= 1e-5, f"{what}: scale relative error {st['scale_max_rel']:.3e}"
    assert st["scales_bit_exact_outside_boundary"], f"{what}: scales differ outside boundary rows"
    return st


def mx_stats(got: dict, ref: dict) -> dict:
    """Every figure of the parity bar for an MXFP4 call, without judging it
    (codes compared per 4-bit element, E8M0 scales in exponent steps)."""
    boundary = ref["margin"] < BOUNDARY
    ok_rows = ~boundary
    st = {"rows": int(len(boundary)), "boundary_rows": int(boundary.sum())}
    if "residual_out" in ref and got.get("residual_out") is not None:
        st["residual_out_bit_exact"] = bool(np.array_equal(u16(got["residual_out"]), ref["residual_out"]))
    if got.get("y") is not None:
        st["y_bit_exact_outside_boundary"] = bool(np.array_equal(u16(got["y"])[ok_rows], ref["y"][ok_rows]))
    gq, rq = unpack_e2m1(u8(got["q"])), unpack_e2m1(ref["q"])
    st["codes_differing"] = int((gq != rq).sum())
    st["mismatch_fraction"] = st["codes_differing"] / max(1, gq.size)
    st["max_code_ulp"] = int(np.abs(e2m1_ordinal(gq) - e2m1_ordinal(rq)).max(initial=0))
    st["codes_bit_exact_outside_boundary"] = bool(np.array_equal(gq[ok_rows], rq[ok_rows]))
    gs, rs = u8(got["scale"]), ref["scale"]
    st["scales_bit_exact_outside_boundary"] = bool(np.array_equal(gs[ok_rows], rs[ok_rows]))
    st["scale_max_step"] = int(np.abs(gs.astype(np.int32) - rs.astype(np.int32)).max(initial=0))
    return st


def compare_mx(got: dict, ref: dict, what: str = "") -> dict:
    _boundary_rows(ref, what)
    assert "residual_out" not in ref or got.get("residual_out") is not None, f"{what}: no residual_out"
    st = mx_stats(got, ref)
    assert st.get("residual_out_bit_exact", True), f"{what}: residual_out differs"
    assert st.get("y_bit_exact_outside_boundary", True), f"{what}: bf16 y differs outside boundary rows"
    assert st["max_code_ulp"] <= 1, f"{what}: an E2M1 code is more than 1 ULP from the oracle"
    assert st["mismatch_fraction"] <= 1e-3, f"{what}: {st['mismatch_fraction']:.2e} of codes differ"
    assert st["codes_bit_exact_outside_boundary"], f"{what}: codes differ outside boundary rows"
    assert st["scales_bit_exact_outside_boundary"], f"{what}: E8M0 scales differ outside boundary rows"
    assert st["scale_max_step"] <= 1, f"{what}: E8M0 off by > 1"
    return st


def compare_gemm(got, ref: dict, K: int, what: str = "") -> dict:
    """GEMM output (bf16 [M, N]) against the oracle's exact sum.

    Bound per element: the tensor core adds K/64 MMA results into an fp32
    accumulator, each rounding at most 2^-24 of the magnitude sum of the terms
    so far, so the accumulation error is at most (K/64) * 2^-24 * sum|term|
    (taken here with a factor-2 margin, plus two roundings); the bf16 output
    rounding adds at most 2^-8 of the value. Also reports the fraction of
    outputs bit-equal to the oracle's bf16(f32(exact sum)), which is near one
    for data without heavy cancellation."""
    g = u16(got)
    d = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d64, mag = ref["d64"], ref["abs"]
    acc = (K / 64 + 2) * 2.0 ** -23 * mag
    bound = acc * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(d64) + 2.0 ** -133
    err = np.abs(d - d64)
    assert np.all(np.isfinite(d)), f"{what}: non-finite outputs"
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} outputs beyond the bound, worst excess {np.max(err / bound):.3g}"
    exact = float(np.mean(g == ref["d"]))
    return {"outputs": int(g.size), "bit_equal_fraction": exact,
            "max_err_over_bound": float(np.max(err / bound, initial=0.0))}
