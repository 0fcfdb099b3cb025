"""Pins the oracle's encoders to brute force over the formats' code points.

* E4M3: the value of every code comes from torch's float8_e4m3fn storage type
  (a library decode, independent of the oracle); each input is encoded by
  locating it between two neighbouring code values and comparing with their
  exact midpoint, ties going to the even code, saturation above 448.
* E2M1: the eight magnitudes of the OCP MX v1.0 element format
  (0, 0.5, 1, 1.5, 2, 3, 4, 6), the same search, saturation at 6.
* E8M0 exponent: the defining property amax * 2^-X in [4, 8).
* bf16 rounding: torch's float32 -> bfloat16 cast.
"""

import numpy as np
import pytest
import torch

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_table() -> np.ndarray:
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def _nearest_code(a: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Brute-force round-to-nearest-even onto the increasing code values ``values``
    (code k has value values[k]); inputs above the last value saturate."""
    a = a.astype(np.float64)
    top = len(values) - 1
    hi = np.searchsorted(values, a, side="left")          # values[hi-1] < a <= values[hi]
    hi = np.clip(hi, 1, top)
    lo = hi - 1
    exact_hi = values[hi] == a
    mid = (values[lo] + values[hi]) / 2.0                  # exact in float64
    pick = np.where(a < mid, lo, np.where(a > mid, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(exact_hi, hi, pick)
    pick = np.where(a == 0.0, 0, pick)
    pick = np.where(a > values[top], top, pick)
    return pick


def _probe_values(values: np.ndarray, rng, n_random: int, lo_exp: int, hi_exp: int) -> np.ndarray:
    pts = [values, (values[:-1] + values[1:]) / 2.0]
    base = np.concatenate(pts).astype(np.float32)
    near = [base]
    up, dn = base, base
    for _ in range(3):                                     # 1, 2 and 3 fp32 ulps either side
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(0))
        near += [up, dn]
    mags = np.exp2(rng.uniform(lo_exp, hi_exp, n_random)).astype(np.float32)
    special = np.array([0.0, 1e-45, 1e-40, 1.17549435e-38, 1e30, 3.4e38, np.inf], dtype=np.float32)
    allv = np.concatenate(near + [mags, special]).astype(np.float32)
    allv = allv[np.isfinite(allv) | np.isinf(allv)]
    return np.concatenate([allv, -allv])


def test_e4m3_decode_matches_library_table(oracle_mod):
    table = e4m3_table()
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(table)
    assert np.array_equal(np.isnan(dec), nan)
    np.testing.assert_array_equal(dec[~nan], table[~nan])
    assert list(np.flatnonzero(nan)) == [0x7F, 0xFF]


def test_e4m3_encode_brute_force(oracle_mod):
    table = e4m3_table().astype(np.float64)
    values = table[:0x7F]                                  # codes 0x00..0x7E, increasing
    assert np.all(np.diff(values) > 0) and values[-1] == 448.0
    rng = np.random.default_rng(1234)
    v = _probe_values(values, rng, 2_000_000, -16, 10)
    got = oracle_mod.e4m3_encode(v)
    want = _nearest_code(np.abs(v), values).astype(np.uint8)
    want |= np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} mismatches, e.g. v={v[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def test_e4m3_all_codes_round_trip(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3_table()[codes]
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(vals), codes)


def test_e4m3_matches_library_cast_in_range(oracle_mod):
    rng = np.random.default_rng(7)
    v = (np.exp2(rng.uniform(-12, np.log2(448.0), 500_000)) *
         rng.choice([-1.0, 1.0], 500_000)).astype(np.float32)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(v), lib)


def test_e4m3_listed_cases(oracle_mod):
    cases = {1.0625: 0x38, 1.1875: 0x3A, 464.0: 0x7E, 1e9: 0x7E, float("inf"): 0x7E,
             2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02, -0.0: 0x80, 448.0: 0x7E, -448.0: 0xFE,
             2.0 ** -9: 0x01, 2.0 ** -6: 0x08}
    v = np.array(list(cases), dtype=np.float32)
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(v), np.array(list(cases.values()), np.uint8))
    assert oracle_mod.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_e2m1_decode_is_the_format_table(oracle_mod):
    dec = oracle_mod.e2m1_decode(np.arange(16, dtype=np.uint8)).astype(np.float64)
    np.testing.assert_array_equal(dec[:8], E2M1_VALUES)
    np.testing.assert_array_equal(dec[8:], -E2M1_VALUES)
    assert np.signbit(dec[8])


def test_e2m1_encode_brute_force(oracle_mod):
    rng = np.random.default_rng(99)
    v = _probe_values(E2M1_VALUES, rng, 1_000_000, -6, 4)
    got = oracle_mod.e2m1_encode(v)
    want = _nearest_code(np.abs(v), E2M1_VALUES).astype(np.uint8)
    want |= np.where(np.signbit(v), 0x8, 0).astype(np.uint8)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} mismatches, e.g. v={v[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def test_e2m1_listed_ties(oracle_mod):
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7, 6.5: 7, -0.0: 8}
    v = np.array(list(cases), dtype=np.float32)
    np.testing.assert_array_equal(oracle_mod.e2m1_encode(v), np.array(list(cases.values()), np.uint8))


def test_mx_exponent_defining_property(oracle_mod):
    rng = np.random.default_rng(5)
    bits = rng.integers(1, 0x7F800000, 1_000_000, dtype=np.uint32)   # every positive finite fp32
    amax = bits.view(np.float32)
    X = oracle_mod.mx_exponent(amax).astype(np.int64)
    ratio = np.ldexp(amax.astype(np.float64), -X)
    free = X > -127                                   # not clamped from below
    assert np.all((ratio[free] >= 4.0) & (ratio[free] < 8.0))
    # clamped ones: the exponent the property asks for is below -127
    assert np.all(np.ldexp(amax[~free].astype(np.float64), 127) < 8.0)
    assert np.all(X <= 127) and np.all(X >= -127)
    assert oracle_mod.mx_exponent(np.array([0.0], np.float32))[0] == -127


@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_rounding_matches_library_cast(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 0x7F800000, 2_000_000, dtype=np.uint32)
    # force exact ties and near-ties at the bf16 rounding position
    bits[::4] = (bits[::4] & 0xFFFF0000) | 0x8000
    bits[1::4] = (bits[1::4] & 0xFFFF0000) | 0x7FFF
    bits[2::8] |= 0x80000000
    v = bits.view(np.float32)
    lib = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle_mod.bf16_round(v), lib)
