"""Pins of the oracle's GEMM-ready scale layouts: hand-evaluated positions of
the block-scaled MMA tile layout (tests/golden/mx_scale_tiles.json), the
layout being a bijection onto the non-padding bytes, padding bytes holding the
requested fill, and the padded column-major FP8 scales equalling the plain
column-major ones."""

import json
import os

import numpy as np

from mxfp4_activation_quant_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_scale_tiles.json")


def test_mx_scale_tiles_hand_positions(oracle_mod):
    spec = json.load(open(GOLDEN))
    M, G = spec["M"], spec["G"]
    # a distinct value per (m, g) modulo 251, so every position is identifiable
    ids = (np.arange(M * G, dtype=np.int64) % 251 + 1).astype(np.uint8).reshape(M, G)
    out = oracle_mod.mx_scale_tiles(ids, fill=0)
    assert out.size == spec["size"]
    for p in spec["positions"]:
        assert out[p["byte"]] == ids[p["m"], p["g"]], p


def test_mx_scale_tiles_is_a_bijection(oracle_mod):
    for M, G in ((300, 224), (128, 4), (1, 1), (129, 7)):
        idx = np.arange(M * G, dtype=np.int64)
        # the index of every entry, one byte at a time, through the layout
        planes = [oracle_mod.mx_scale_tiles(((idx >> (8 * i)) & 255).astype(np.uint8).reshape(M, G),
                                            fill=0).astype(np.int64) for i in range(3)]
        mark = oracle_mod.mx_scale_tiles(np.ones((M, G), np.uint8), fill=0)
        assert int(mark.sum()) == M * G                       # every entry lands on its own byte
        got = np.sort((planes[0] + (planes[1] << 8) + (planes[2] << 16))[mark == 1])
        np.testing.assert_array_equal(got, idx)


def test_mx_scale_tiles_padding_is_fill(oracle_mod):
    """Bytes of the padded tiles that hold no entry (rows past M, groups past
    G) carry the requested fill; the entries keep their values."""
    for M, G, fill in ((130, 5, 0xAB), (1, 1, 7), (128, 4, 255)):
        data = np.full((M, G), 3, np.uint8)                   # no entry equals the fill
        out = oracle_mod.mx_scale_tiles(data, fill=fill)
        assert out.size == -(-M // 128) * -(-G // 4) * 512
        assert int((out == 3).sum()) == M * G
        assert int((out == fill).sum()) == out.size - M * G


def test_fp8_padded_column_major(oracle_mod):
    d = synth.make_inputs(synth.WORKLOADS["decode"], M=37)
    a = oracle_mod.add_rmsnorm_quant_fp8(d["x"], d["residual"], d["gamma"], 1e-6, layout="col")
    b = oracle_mod.add_rmsnorm_quant_fp8(d["x"], d["residual"], d["gamma"], 1e-6, layout="col_pad4")
    assert b["scale"].shape == (56, 40)
    np.testing.assert_array_equal(a["scale"], b["scale"][:, :37])
    assert np.all(np.isnan(b["scale"][:, 37:]))
