"""Pins the oracle's add, RMSNorm and group-quant steps to library routines and
to invariants the definition implies.

* add: torch's CPU bf16 addition (fp32 sum, one rounding to bf16);
* RMSNorm: torch.nn.functional.rms_norm in float64 -- the bf16 y must be the
  nearest bf16 of the fp64 result, up to the fp32 roundings the definition
  makes; inv_rms equals the fp32 rounding of numpy's fp64 1/sqrt(mean+eps)
  wherever that value is not within 1e-12 of an fp32 rounding boundary;
* FP8 quant: the amax element encodes to +-448, every code dequantises to
  within half an E4M3 step (plus the fp32 quotient's rounding), the scale is
  the IEEE fp32 quotient amax/448 (numpy's float32 division), the
  column-major layout is the transpose of the row-major one;
* MXFP4: amax * 2^-X in [4, 8), each nibble dequantises to within half an
  E2M1 step of its own element (so a swapped nibble order fails), saturation
  only above 6;
* structure: qknorm halves equal single-tensor calls; results do not depend
  on the thread count or on the row's position in the batch.
"""

import numpy as np
import pytest
import torch

from mxfp4_activation_quant_gb300 import synth


def _f(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def batch():
    w = synth.WORKLOADS["decode"]
    d = synth.make_inputs(w, M=48)
    return {k: _bits(v) for k, v in d.items()}


def test_add_matches_library_bf16_add(oracle_mod):
    rng = np.random.default_rng(11)
    n = 400_000
    a = rng.standard_normal(n).astype(np.float32)
    b = (rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))).astype(np.float32)
    b[::7] = -a[::7]                                     # exact cancellation
    b[1::7] = a[1::7] * np.float32(2.0 ** -8)            # ties at the bf16 position
    ta = torch.from_numpy(a).to(torch.bfloat16)
    tb = torch.from_numpy(b).to(torch.bfloat16)
    want = _bits(ta + tb)
    got = oracle_mod.add_residual(_bits(ta)[None, :], _bits(tb)[None, :])[0]
    np.testing.assert_array_equal(got, want)


def test_rmsnorm_matches_library_fp64(oracle_mod, batch):
    r = oracle_mod.add_residual(batch["x"], batch["residual"])
    y, inv, margin = oracle_mod.rmsnorm(r, batch["gamma"], 1e-6)
    r64 = torch.from_numpy(_f(r).astype(np.float64))
    g64 = torch.from_numpy(_f(batch["gamma"]).astype(np.float64))
    y64 = torch.nn.functional.rms_norm(r64, (r.shape[1],), weight=g64, eps=1e-6).numpy()
    yo = _f(y).astype(np.float64)
    # one bf16 step at |y64| (normal range), and the three fp32 roundings
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y64), 2.0 ** -126))) - 7)
    assert np.all(np.abs(yo - y64) <= 0.5 * ulp + np.abs(y64) * 2.0 ** -21)
    # inv_rms: fp32 rounding of the fp64 closed form
    ms = np.mean(_f(r).astype(np.float64) ** 2, axis=1)
    t = 1.0 / np.sqrt(ms + np.float64(np.float32(1e-6)))
    clear = margin > 1e-12
    assert clear.sum() > 40
    np.testing.assert_array_equal(inv[clear], t[clear].astype(np.float32))
    assert np.all(np.abs(inv.astype(np.float64) - t) <= t * 2.0 ** -23)


def test_rmsnorm_scale_invariance(oracle_mod, batch):
    r = batch["x"][:8]
    r2 = oracle_mod.bf16_round(_f(r) * 2.0).reshape(r.shape)    # exact doubling
    y1, inv1, _ = oracle_mod.rmsnorm(r, batch["gamma"], 0.0)
    y2, inv2, _ = oracle_mod.rmsnorm(r2, batch["gamma"], 0.0)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(inv1, inv2 * 2)


def test_rmsnorm_order_invariance(oracle_mod, batch):
    r = np.ascontiguousarray(batch["x"][:16])
    rng = np.random.default_rng(3)
    perm = rng.permutation(r.shape[1])
    y1, inv1, m1 = oracle_mod.rmsnorm(r, batch["gamma"], 1e-6)
    y2, inv2, _ = oracle_mod.rmsnorm(np.ascontiguousarray(r[:, perm]),
                                     np.ascontiguousarray(batch["gamma"][perm]), 1e-6)
    ok = m1 > 1e-12
    np.testing.assert_array_equal(inv1[ok], inv2[ok])
    np.testing.assert_array_equal(y1[ok][:, perm], y2[ok])


def _e4m3_values():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def test_fp8_quant_invariants(oracle_mod, batch):
    out = oracle_mod.add_rmsnorm_quant_fp8(batch["x"], batch["residual"], batch["gamma"], 1e-6)
    y = _f(out["y"])
    M, H = y.shape
    G = 128
    yg = y.reshape(M, H // G, G)
    amax = np.abs(yg).max(axis=2)
    np.testing.assert_array_equal(out["scale"], amax / np.float32(448.0))
    q = out["q"].reshape(M, H // G, G)
    arg = np.abs(yg).argmax(axis=2)
    qa = np.take_along_axis(q, arg[..., None], axis=2)[..., 0]
    assert np.all((qa & 0x7F) == 0x7E)
    dec = _e4m3_values()[q].astype(np.float64)
    s = out["scale"].astype(np.float64)[..., None]
    v = np.abs(yg.astype(np.float64)) / s
    step = np.where(v < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3))
    err = np.abs(dec * s - yg)
    assert np.all(err <= (0.5 * step + v * 2.0 ** -22) * s)
    assert np.all(np.signbit(dec) == np.signbit(yg))


def test_fp8_column_major_is_transpose(oracle_mod, batch):
    a = oracle_mod.add_rmsnorm_quant_fp8(batch["x"], batch["residual"], batch["gamma"], 1e-6, layout="row")
    b = oracle_mod.add_rmsnorm_quant_fp8(batch["x"], batch["residual"], batch["gamma"], 1e-6, layout="col")
    np.testing.assert_array_equal(a["scale"].T, b["scale"])
    np.testing.assert_array_equal(a["q"], b["q"])


def test_mxfp4_invariants(oracle_mod):
    w = synth.WORKLOADS["mxfp4"]
    d = {k: _bits(v) for k, v in synth.make_inputs(w, M=32).items()}
    out = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], 1e-6)
    y = _f(out["y"]).astype(np.float64)
    M, H = y.shape
    yg = y.reshape(M, H // 32, 32)
    amax = np.abs(yg).max(axis=2)
    X = out["scale"].astype(np.int64) - 127
    ratio = amax * np.exp2(-X.astype(np.float64))
    assert np.all((ratio >= 4) & (ratio < 8))
    lo = out["q"] & 0xF
    hi = out["q"] >> 4
    codes = np.empty((M, H), dtype=np.uint8)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    dec = np.where(codes & 8, -1.0, 1.0) * mag[codes & 7]
    v = np.abs(y) * np.exp2(-np.repeat(X, 32, axis=1))
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    sat = v > 6
    err = np.abs(dec - y * np.exp2(-np.repeat(X, 32, axis=1)))
    assert np.all(err[~sat] <= 0.5 * step[~sat])
    assert np.all((codes[sat] & 7) == 7) and np.all(err[sat] < 2.0)


def test_qknorm_halves_equal_single_calls(oracle_mod):
    w = synth.WORKLOADS["qknorm"]
    d = {k: _bits(v) for k, v in synth.make_inputs(w, M=24).items()}
    both = oracle_mod.qknorm_quant_fp8(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], 1e-6)
    one = oracle_mod.add_rmsnorm_quant_fp8(d["kv_a"], None, d["gamma_kv"], 1e-6)
    for k in ("q", "scale", "y"):
        np.testing.assert_array_equal(both["kv"][k], one[k])
    assert both["q"]["q"].shape == (24, 1536) and both["q"]["scale"].shape == (24, 12)


def test_thread_count_and_row_position_do_not_matter(oracle_mod, batch):
    a = oracle_mod.add_rmsnorm_quant_fp8(batch["x"], batch["residual"], batch["gamma"], 1e-6, nthreads=1)
    b = oracle_mod.add_rmsnorm_quant_fp8(batch["x"], batch["residual"], batch["gamma"], 1e-6, nthreads=7)
    c = oracle_mod.add_rmsnorm_quant_fp8(batch["x"][5:9], batch["residual"][5:9], batch["gamma"], 1e-6)
    for k in ("q", "scale", "y", "residual_out", "inv"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(a["q"][5:9], c["q"])
    np.testing.assert_array_equal(a["scale"][5:9], c["scale"])


def test_strided_input_rows(oracle_mod, batch):
    wide = np.zeros((8, 7168 + 64), dtype=np.uint16)
    wide[:, 32:32 + 7168] = batch["x"][:8]
    view = wide[:, 32:32 + 7168]
    a = oracle_mod.add_rmsnorm_quant_fp8(view, None, batch["gamma"], 1e-6)
    b = oracle_mod.add_rmsnorm_quant_fp8(np.ascontiguousarray(batch["x"][:8]), None, batch["gamma"], 1e-6)
    np.testing.assert_array_equal(a["q"], b["q"])
    np.testing.assert_array_equal(a["y"], b["y"])


def test_mxfp4_qknorm_halves_equal_single_calls(oracle_mod):
    w = synth.WORKLOADS["qknorm"]
    d = {k: _bits(v) for k, v in synth.make_inputs(w, M=16).items()}
    both = oracle_mod.qknorm_quant_mxfp4(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], 1e-6)
    one = oracle_mod.add_rmsnorm_quant_mxfp4(d["q_a"], None, d["gamma_q"], 1e-6)
    for k in ("q", "scale", "y"):
        np.testing.assert_array_equal(both["q"][k], one[k])
    assert both["kv"]["q"].shape == (16, 256) and both["kv"]["scale"].shape == (16, 16)


def test_margin_is_the_distance_to_the_fp32_rounding_boundary(oracle_mod, batch):
    """The per-row margin (which decides the rows where parity may differ by
    one bf16 step) equals the relative distance of numpy's fp64 inv_rms from
    the nearest point where its fp32 rounding changes."""
    r = oracle_mod.add_residual(batch["x"], batch["residual"])
    _, inv, margin = oracle_mod.rmsnorm(r, batch["gamma"], 1e-6)
    t = 1.0 / np.sqrt(np.mean(_f(r).astype(np.float64) ** 2, axis=1) + np.float64(np.float32(1e-6)))
    f = t.astype(np.float32)
    up = np.nextafter(f, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(f, np.float32(0)).astype(np.float64)
    want = np.minimum(np.abs(t - (f + up) / 2), np.abs(t - (f + dn) / 2)) / t
    # the oracle's S and numpy's mean differ in the last bits only
    np.testing.assert_allclose(margin, want, rtol=0, atol=2.0 ** -50)
    assert margin.max() < 2.0 ** -23 and np.median(margin) > 2.0 ** -30
