"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (compiled on
the CPU and swapped in for the real oracle) or of its numpy layer (loaded over
the real C library), and runs the pins (hand-worked rows, encoder brute force,
library cross-checks, invariants, structural identities): at least one of them
must fail. Nothing here touches the GPU or the real oracle build.
"""

import importlib.util
import os
import shutil

import numpy as np
import pytest

from oracle import build as oracle_build
from oracle import oracle as O

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "rmsq_oracle.c")
PY_SRC = os.path.join(os.path.dirname(SRC), "oracle.py")

MUTANTS = {
    "drop_eps": ("sqrt(S / (double)c->H + (double)c->eps)", "sqrt(S / (double)c->H)"),
    "mean_over_H_minus_1": ("S / (double)c->H + (double)c->eps", "S / (double)(c->H - 1) + (double)c->eps"),
    "gamma_index_reversed": ("bf16_to_f32(c->gamma[i])", "bf16_to_f32(c->gamma[c->H - 1 - i])"),
    "fnuz_max_240": ("float scale = amax / 448.0f;", "float scale = amax / 240.0f;"),
    "scale_by_reciprocal": ("float scale = amax / 448.0f;", "float scale = amax * (1.0f / 448.0f);"),
    "e4m3_round_half_up": ("double n = nearbyint(ldexp(a, 3 - e));", "double n = floor(ldexp(a, 3 - e) + 0.5);"),
    "e4m3_no_saturation": [("if (a > 448.0) /* saturate", "if (a > 3.0e38) /* saturate"),
                           ("    if (code > 0x7e)\n        code = 0x7e;\n    return (uint8_t)(sign | code);",
                            "    return (uint8_t)(sign | code);")],
    "e4m3_subnormal_step": ("code = (int)nearbyint(a * 512.0);", "code = (int)nearbyint(a * 256.0);"),
    "e4m3_sign_dropped": ("    if (code > 0x7e)\n        code = 0x7e;\n    return (uint8_t)(sign | code);",
                          "    if (code > 0x7e)\n        code = 0x7e;\n    return (uint8_t)(code);"),
    "e2m1_round_half_up": ("code = (int)nearbyint(2.0 * a);", "code = (int)floor(2.0 * a + 0.5);"),
    "mx_exponent_off_by_one": ("int X = (e2 - 1) - 2;", "int X = (e2 - 1) - 3;"),
    "mx_no_lower_clamp": ("    if (X < -127)\n        X = -127;\n", ""),
    "mx_nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "bf16_round_half_up": ("u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    "residual_not_added": ("float s = bf16_to_f32(c->x[m * c->ldx + i]) + bf16_to_f32(c->res[m * c->ldres + i]);",
                           "float s = bf16_to_f32(c->x[m * c->ldx + i]);"),
    "col_major_as_row_major": ("c->scale[g * c->M + m] = scale;", "c->scale[m * ngroups + g] = scale;"),
    "quantise_unnormalised": ("float v = bf16_to_f32(row[i]);\n                float quot", "float v = bf16_to_f32(row[i]) * 2.0f;\n                float quot"),
    "mx_tiles_rows_transposed": ("out[tile * 512 + (r % 32) * 16 + (r / 32) * 4 + c]",
                                 "out[tile * 512 + (r / 32) * 16 + (r % 32) * 4 + c]"),
    "col_pad4_unpadded": ("c->scale[g * ((c->M + 3) / 4 * 4) + m] = scale;", "c->scale[g * c->M + m] = scale;"),
    # swapping the nibble order of BOTH operands leaves every sum unchanged;
    # a mismatch between the two is the mistake that matters
    "gemm_a_nibbles_swapped": ("mx_element(arow, asc, k)", "mx_element(arow, asc, k ^ 1)"),
    "gemm_scale_bias_128": ("(int)s[k / 32] - 127", "(int)s[k / 32] - 128"),
    "gemm_b_scales_by_a_row": ("*bsc = c->sb + n * (K / 32)", "*bsc = c->sb + m * (K / 32)"),
    "gemm_plain_running_sum": ("double d = sum + comp;", "double d = sum;"),
    "gemm_output_truncated": ("c->dbf16[o] = f32_to_bf16_rne((float)d);",
                              "c->dbf16[o] = (uint16_t)(*(uint32_t *)&(float){(float)d} >> 16);"),
    "gemm_b_nibbles_swapped": ("mx_element(brow, bsc, k)", "mx_element(brow, bsc, k ^ 1)"),
    "gemm_magnitude_signed": ("mag += fabs(term);", "mag += term;"),
    "gemm_last_group_dropped": ("for (int64_t k = 0; k < K; ++k) {\n                double term",
                                "for (int64_t k = 0; k < K - 32; ++k) {\n                double term"),
    "zero_group_nan": ("float quot = (amax == 0.0f) ? v : v / scale;", "float quot = v / scale;"),
    "margin_to_the_far_boundary": ("fmin(fabs(t64 - mid_up), fabs(t64 - mid_dn))",
                                   "fmax(fabs(t64 - mid_up), fabs(t64 - mid_dn))"),
}

# Mistakes in the numpy layer that chains the C steps (oracle/oracle.py).
PY_MUTANTS = {
    "residual_skipped": ("        r = add_residual(x, residual, nthreads)\n    else:\n        r = x",
                         "        r = x\n    else:\n        r = x"),
    "scale_layout_ignored": ("q, scale = group_quant_fp8(y, group, _layout_code(layout), nthreads)",
                             "q, scale = group_quant_fp8(y, group, SCALE_ROW_MAJOR, nthreads)"),
    "kv_half_is_the_q_half": ('    return {"q": a, "kv": b}', '    return {"q": a, "kv": a}'),
    "prequant_drops_activation_scales": ("    out = mxfp4_gemm(q, s, b_q, b_scale, nthreads)",
                                         "    out = mxfp4_gemm(q, np.full_like(s, 127), b_q, b_scale, nthreads)"),
    "tile_padding_fill_ignored": ("out = np.full(((M + 127) // 128) * ((G + 3) // 4) * 512, fill, dtype=np.uint8)",
                                  "out = np.full(((M + 127) // 128) * ((G + 3) // 4) * 512, 0, dtype=np.uint8)"),
}


def _pins(oracle_mod):
    """The oracle's pins, run against whatever library oracle_mod has loaded."""
    from tests import test_oracle_encoders as enc
    from tests import test_oracle_golden as gold
    from tests import test_oracle_norm as norm

    for row in gold._rows():
        yield f"golden:{row['name']}", lambda r=row: gold.test_handworked_row(r, oracle_mod)
    yield "enc:e4m3_listed", lambda: enc.test_e4m3_listed_cases(oracle_mod)
    yield "enc:e4m3_brute", lambda: enc.test_e4m3_encode_brute_force(oracle_mod)
    yield "enc:e2m1_listed", lambda: enc.test_e2m1_listed_ties(oracle_mod)
    yield "enc:e2m1_brute", lambda: enc.test_e2m1_encode_brute_force(oracle_mod)
    yield "enc:mx_exponent", lambda: enc.test_mx_exponent_defining_property(oracle_mod)
    yield "enc:bf16", lambda: enc.test_bf16_rounding_matches_library_cast(oracle_mod, 0)
    yield "norm:add", lambda: norm.test_add_matches_library_bf16_add(oracle_mod)
    b = _batch()
    yield "norm:rms_norm", lambda: norm.test_rmsnorm_matches_library_fp64(oracle_mod, b)
    yield "norm:fp8_invariants", lambda: norm.test_fp8_quant_invariants(oracle_mod, b)
    yield "norm:col_major", lambda: norm.test_fp8_column_major_is_transpose(oracle_mod, b)
    yield "norm:mxfp4_invariants", lambda: norm.test_mxfp4_invariants(oracle_mod)
    yield "norm:margin", lambda: norm.test_margin_is_the_distance_to_the_fp32_rounding_boundary(oracle_mod, b)
    yield "norm:qknorm_halves", lambda: norm.test_qknorm_halves_equal_single_calls(oracle_mod)
    yield "norm:mxfp4_qknorm_halves", lambda: norm.test_mxfp4_qknorm_halves_equal_single_calls(oracle_mod)
    from tests import test_oracle_layouts as lay
    yield "layout:mx_tiles", lambda: lay.test_mx_scale_tiles_hand_positions(oracle_mod)
    yield "layout:mx_tiles_fill", lambda: lay.test_mx_scale_tiles_padding_is_fill(oracle_mod)
    yield "layout:col_pad4", lambda: lay.test_fp8_padded_column_major(oracle_mod)
    from tests import test_oracle_gemm as gemm
    yield "gemm:hand", lambda: gemm.test_hand_worked_product(oracle_mod)
    yield "gemm:one_hot", lambda: gemm.test_one_hot_weights_extract_the_activation(oracle_mod)
    yield "gemm:transpose", lambda: gemm.test_swapping_operands_transposes(oracle_mod)
    yield "gemm:numpy_fp64", lambda: gemm.test_exact_fp64_matrix_product(oracle_mod)
    yield "gemm:scale_group", lambda: gemm.test_scale_byte_scales_its_group_only(oracle_mod)
    yield "gemm:cancellation", lambda: gemm.test_cancellation_keeps_small_terms(oracle_mod)
    yield "gemm:prequant", lambda: gemm.test_prequant_is_quant_then_gemm(oracle_mod)


def _batch():
    import torch
    from mxfp4_activation_quant_gb300 import synth
    d = synth.make_inputs(synth.WORKLOADS["decode"], M=48)
    return {k: v.contiguous().view(torch.int16).numpy().view(np.uint16) for k, v in d.items()}


def test_real_oracle_passes_every_pin(oracle_mod):
    for name, run in _pins(oracle_mod):
        run()


def _first_failing_pin(oracle_mod):
    for name, run in _pins(oracle_mod):
        try:
            run()
        except AssertionError:
            return name
    return None


@pytest.mark.parametrize("mutant", sorted(PY_MUTANTS))
def test_planted_mistake_in_the_composition_is_caught(mutant, tmp_path):
    """The same for the numpy layer: a copy of oracle.py with one mistake,
    loaded as a module of the oracle package over the real C library."""
    find, repl = PY_MUTANTS[mutant]
    src = open(PY_SRC).read()
    assert src.count(find) == 1, f"mutation site for {mutant} not found exactly once"
    path = tmp_path / "oracle_mutant.py"
    path.write_text(src.replace(find, repl))
    spec = importlib.util.spec_from_file_location("oracle.oracle_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._lib = O.lib()
    assert _first_failing_pin(mod), f"no pin caught the planted mistake {mutant!r}"


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path, monkeypatch):
    edits = MUTANTS[mutant]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for find, repl in edits:
        assert src.count(find) == 1, f"mutation site for {mutant} not found exactly once"
        src = src.replace(find, repl)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle_build.compile_source(str(path), str(tmp_path / "libmutant.so"))
    monkeypatch.setattr(O, "_lib", O.load_library(lib))
    assert _first_failing_pin(O), f"no pin caught the planted mistake {mutant!r}"
