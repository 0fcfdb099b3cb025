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


def compare_fp8(got: dict, ref: dict, scale_layout: str = "row", what: str = "") -> dict:
    """got/ref: dicts with q (codes [M,H]), scale, optional y, residual_out (bf16 bits)."""
    boundary = _boundary_rows(ref, what)
    stats = {"rows": int(len(boundary)), "boundary_rows": int(boundary.sum())}
    ok_rows = ~boundary
    if "residual_out" in ref:
        assert np.array_equal(u16(got["residual_out"]), ref["residual_out"]), f"{what}: residual_out differs"
    if got.get("y") is not None:
        gy, ry = u16(got["y"]), ref["y"]
        assert np.array_equal(gy[ok_rows], ry[ok_rows]), f"{what}: bf16 y differs outside boundary rows"
        assert np.all(np.abs(bf16_ordinal(gy) - bf16_ordinal(ry)) <= 1), f"{what}: bf16 y off by > 1 step"
    gq, rq = u8(got["q"]), ref["q"]
    dist = np.abs(e4m3_ordinal(gq) - e4m3_ordinal(rq))
    stats["codes_differing"] = int((gq != rq).sum())
    stats["mismatch_fraction"] = stats["codes_differing"] / max(1, gq.size)
    assert dist.max(initial=0) <= 1, f"{what}: a code is more than 1 ULP from the oracle"
    assert stats["mismatch_fraction"] <= 1e-3, f"{what}: {stats['mismatch_fraction']:.2e} of codes differ"
    assert np.array_equal(gq[ok_rows], rq[ok_rows]), f"{what}: codes differ outside boundary rows"
    gs = got["scale"].detach().cpu().numpy() if isinstance(got["scale"], torch.Tensor) else got["scale"]
    rs = ref["scale"]
    assert gs.shape == rs.shape, f"{what}: scale shape {gs.shape} vs {rs.shape}"
    rel = np.abs(gs.astype(np.float64) - rs) / np.maximum(np.abs(rs.astype(np.float64)), 1e-30)
    assert rel.max(initial=0) <= 1e-5, f"{what}: scale relative error {rel.max():.3e}"
    row_axis = 0 if scale_layout == "row" else 1
    gs_rows = gs if row_axis == 0 else gs.T
    rs_rows = rs if row_axis == 0 else rs.T
    assert np.array_equal(gs_rows[ok_rows].view(np.uint32), rs_rows[ok_rows].view(np.uint32)), \
        f"{what}: scales differ outside boundary rows"
    return stats


def compare_mx(got: dict, ref: dict, what: str = "") -> dict:
    boundary = _boundary_rows(ref, what)
    stats = {"rows": int(len(boundary)), "boundary_rows": int(boundary.sum())}
    ok_rows = ~boundary
    if "residual_out" in ref:
        assert np.array_equal(u16(got["residual_out"]), ref["residual_out"]), f"{what}: residual_out differs"
    if got.get("y") is not None:
        gy, ry = u16(got["y"]), ref["y"]
        assert np.array_equal(gy[ok_rows], ry[ok_rows]), f"{what}: bf16 y differs outside boundary rows"
    gq, rq = unpack_e2m1(u8(got["q"])), unpack_e2m1(ref["q"])
    dist = np.abs(e2m1_ordinal(gq) - e2m1_ordinal(rq))
    stats["codes_differing"] = int((gq != rq).sum())
    stats["mismatch_fraction"] = stats["codes_differing"] / max(1, gq.size)
    assert dist.max(initial=0) <= 1, f"{what}: an E2M1 code is more than 1 ULP from the oracle"
    assert stats["mismatch_fraction"] <= 1e-3, f"{what}: {stats['mismatch_fraction']:.2e} of codes differ"
    assert np.array_equal(gq[ok_rows], rq[ok_rows]), f"{what}: codes differ outside boundary rows"
    gs, rs = u8(got["scale"]), ref["scale"]
    assert np.array_equal(gs[ok_rows], rs[ok_rows]), f"{what}: E8M0 scales differ outside boundary rows"
    assert np.all(np.abs(gs.astype(np.int32) - rs.astype(np.int32)) <= 1), f"{what}: E8M0 off by > 1"
    return stats


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
