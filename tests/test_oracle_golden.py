"""Pins the CPU oracle to rows worked out by hand (tests/golden/handworked_rows.json).

Each row's expected values were derived on paper from the definition (the
derivation and citation travel with the row in the fixture); none comes from
running any implementation.
"""

import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handworked_rows.json")


def _vec(spec, H, dtype):
    v = np.full(H, spec["fill"], dtype=np.float64)
    for i, val in spec["set"]:
        v[i] = val
    return v.astype(dtype)


def _bf16_bits(vals: np.ndarray) -> np.ndarray:
    """Exact bf16 values -> bit patterns (asserts exactness)."""
    f = vals.astype(np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "fixture value is not an exact bf16"
    return (bits >> 16).astype(np.uint16)


def _rows():
    with open(GOLDEN) as fh:
        return json.load(fh)["rows"]


@pytest.mark.parametrize("row", _rows(), ids=lambda r: r["name"])
def test_handworked_row(row, oracle_mod):
    O = oracle_mod
    H = row["H"]
    x = _bf16_bits(_vec(row["x"], H, np.float64))[None, :]
    res = None if row["residual"] is None else _bf16_bits(_vec(row["residual"], H, np.float64))[None, :]
    gamma = _bf16_bits(_vec(row["gamma"], H, np.float64))
    exp = row["expect"]
    if row["kind"] == "fp8":
        out = O.add_rmsnorm_quant_fp8(x, res, gamma, eps=row["eps"], group=128)
    else:
        out = O.add_rmsnorm_quant_mxfp4(x, res, gamma, eps=row["eps"])

    assert out["inv"][0] == np.float32(exp["inv"])
    if "residual_out" in exp:
        np.testing.assert_array_equal(out["residual_out"][0],
                                      _bf16_bits(_vec(exp["residual_out"], H, np.float64)))
    if "y" in exp:
        np.testing.assert_array_equal(O.bf16_to_f32(out["y"][0]), _vec(exp["y"], H, np.float32))
    if row["kind"] == "fp8":
        amax = np.array(exp["amax"], dtype=np.float32)
        if "scale" in exp:
            want_scale = np.array(exp["scale"], dtype=np.float32)
        else:
            # the IEEE fp32 quotient amax/448, formed by numpy
            want_scale = amax / np.float32(448.0)
        np.testing.assert_array_equal(out["scale"][0], want_scale)
        np.testing.assert_array_equal(out["q"][0], _vec(exp["q"], H, np.int64).astype(np.uint8))
    else:
        np.testing.assert_array_equal(out["scale"][0], np.array(exp["mx_scale"], dtype=np.uint8))
        codes = _vec(exp["codes"], H, np.int64).astype(np.uint8)
        packed = codes[0::2] | (codes[1::2] << 4)
        np.testing.assert_array_equal(out["q"][0], packed)


def test_golden_rows_cover_both_variants():
    kinds = {r["kind"] for r in _rows()}
    assert kinds == {"fp8", "mxfp4"}
