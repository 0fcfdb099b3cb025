"""Pins of the oracle's consumer GEMM (D = A B^T on MXFP4 operands).

Each check rests on something other than the oracle's own code: a product
worked out by hand (tests/golden/mxfp4_gemm_hand.json), the E2M1 value
table of the OCP Microscaling spec written out here, exact fp64 matrix
products of the dequantised operands (numpy), and the algebra of the
definition (transposition, one-hot extraction, linearity in each group's
scale)."""

import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp4_gemm_hand.json")

# OCP Microscaling Formats v1.0, E2M1: codes 0..7 (bit 3 is the sign)
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _value(code):
    code = np.asarray(code)
    v = E2M1_VALUES[code & 7]
    return np.where(code & 8, -v, v)


def _dequant(q, s):
    """[R, K/2] packed codes + [R, K/32] scale bytes -> fp64 [R, K]."""
    codes = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    return _value(codes) * np.exp2(np.repeat(s.astype(np.int64) - 127, 32, axis=1))


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _operand(rows, K):
    codes = np.zeros((len(rows), K), dtype=np.uint8)
    scales = np.zeros((len(rows), K // 32), dtype=np.uint8)
    for r, groups in enumerate(rows):
        for g, spec in enumerate(groups):
            codes[r, g * 32:(g + 1) * 32] = spec["fill"]
            for k, c in spec["set"]:
                codes[r, g * 32 + k] = c
            scales[r, g] = spec["scale"]
    return _pack(codes), scales


def _random_operand(rng, R, K, lo=122, hi=132):
    q = rng.integers(0, 256, (R, K // 2), dtype=np.uint8)
    s = rng.integers(lo, hi, (R, K // 32), dtype=np.uint8)
    return q, s


def test_hand_worked_product(oracle_mod):
    g = json.load(open(GOLDEN))
    a_q, a_s = _operand(g["a"], g["K"])
    b_q, b_s = _operand(g["b"], g["K"])
    out = oracle_mod.mxfp4_gemm(a_q, a_s, b_q, b_s)
    for e in g["expect"]:
        m, n = e["m"], e["n"]
        assert out["d64"][m, n] == e["d"], e
        assert out["abs"][m, n] == e["abs"], e
        assert int(out["d"][m, n]) == int(e["d_bf16"], 16), e


def test_one_hot_weights_extract_the_activation(oracle_mod):
    """B[n, k] = 1.0 exactly when k == n: column n of D is element n of A."""
    rng = np.random.default_rng(11)
    M, K = 5, 128
    a_q, a_s = _random_operand(rng, M, K)
    codes = np.zeros((K, K), dtype=np.uint8)
    codes[np.arange(K), np.arange(K)] = 2          # E2M1 1.0
    b_q, b_s = _pack(codes), np.full((K, K // 32), 127, dtype=np.uint8)
    out = oracle_mod.mxfp4_gemm(a_q, a_s, b_q, b_s)
    assert np.array_equal(out["d64"], _dequant(a_q, a_s))


def test_swapping_operands_transposes(oracle_mod):
    rng = np.random.default_rng(12)
    a_q, a_s = _random_operand(rng, 7, 96)
    b_q, b_s = _random_operand(rng, 9, 96)
    ab = oracle_mod.mxfp4_gemm(a_q, a_s, b_q, b_s)
    ba = oracle_mod.mxfp4_gemm(b_q, b_s, a_q, a_s)
    assert np.array_equal(ab["d64"], ba["d64"].T)
    assert np.array_equal(ab["d"], ba["d"].T)


def test_exact_fp64_matrix_product(oracle_mod):
    """Scale bytes in a narrow band keep every partial sum exact in fp64, so
    numpy's fp64 product of the dequantised operands is the exact result."""
    rng = np.random.default_rng(13)
    a_q, a_s = _random_operand(rng, 33, 256)
    b_q, b_s = _random_operand(rng, 40, 256)
    out = oracle_mod.mxfp4_gemm(a_q, a_s, b_q, b_s)
    A, B = _dequant(a_q, a_s), _dequant(b_q, b_s)
    assert np.array_equal(out["d64"], A @ B.T)
    assert np.array_equal(out["abs"], np.abs(A) @ np.abs(B).T)
    # bf16 output: the fp32 rounding of the sum, rounded to bf16 (checked
    # against torch's round-to-nearest-even fp32 -> bf16 cast)
    import torch
    ref = torch.from_numpy(out["d64"].astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(out["d"], ref.view(torch.int16).numpy().view(np.uint16))


def test_scale_byte_scales_its_group_only(oracle_mod):
    """Raising one A scale byte by one doubles that group's contribution to
    its row and leaves every other row unchanged."""
    rng = np.random.default_rng(14)
    M, N, K = 4, 6, 128
    a_q, a_s = _random_operand(rng, M, K)
    b_q, b_s = _random_operand(rng, N, K)
    base = oracle_mod.mxfp4_gemm(a_q, a_s, b_q, b_s)["d64"]
    m, g = 2, 1
    only = np.zeros_like(a_q)
    only[m, g * 16:(g + 1) * 16] = a_q[m, g * 16:(g + 1) * 16]
    contrib = oracle_mod.mxfp4_gemm(only, a_s, b_q, b_s)["d64"][m]
    bumped_s = a_s.copy()
    bumped_s[m, g] += 1
    bumped = oracle_mod.mxfp4_gemm(a_q, bumped_s, b_q, b_s)["d64"]
    assert np.array_equal(bumped[m], base[m] + contrib)
    keep = np.arange(M) != m
    assert np.array_equal(bumped[keep], base[keep])


def test_prequant_is_quant_then_gemm(oracle_mod):
    """The prequant placement quantises with the same group-32 rule as the
    fused kernel (step 3b), so both placements feed the GEMM the same codes."""
    import torch
    from mxfp4_activation_quant_gb300 import synth
    y = synth.random_bf16(15, (3, 128)).view(torch.int16).numpy().view(np.uint16)
    rng = np.random.default_rng(15)
    b_q, b_s = _random_operand(rng, 5, 128)
    pre = oracle_mod.a16wfp4_gemm(y, b_q, b_s)
    q, s = oracle_mod.group_quant_mxfp4(y)
    assert np.array_equal(pre["a_q"], q) and np.array_equal(pre["a_scale"], s)
    assert np.array_equal(pre["d"], oracle_mod.mxfp4_gemm(q, s, b_q, b_s)["d"])


def test_rejects_bad_shapes(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.mxfp4_gemm(np.zeros((2, 16), np.uint8), np.zeros((2, 1), np.uint8),
                              np.zeros((3, 8), np.uint8), np.zeros((3, 1), np.uint8))


def test_cancellation_keeps_small_terms(oracle_mod):
    """+2^60 + 1 - 2^60 along K: the exact sum is 1, which a plain fp64
    running sum would lose."""
    K = 96
    a = np.zeros((1, K), dtype=np.uint8)
    b = np.zeros((1, K), dtype=np.uint8)
    a[0, 0], a[0, 32], a[0, 64] = 2, 2, 10          # +1, +1, -1
    b[0, 0], b[0, 32], b[0, 64] = 2, 2, 2
    a_s = np.array([[127 + 60, 127, 127 + 60]], dtype=np.uint8)
    b_s = np.full((1, 3), 127, dtype=np.uint8)
    out = oracle_mod.mxfp4_gemm(_pack(a), a_s, _pack(b), b_s)
    assert out["d64"][0, 0] == 1.0
    assert out["abs"][0, 0] == 2.0 ** 61 + 1
