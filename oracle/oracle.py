"""numpy wrapper around the plain-C oracle (``rmsq_oracle.c``).

TEST INFRASTRUCTURE: loaded only by the tests, the smoke check and the
benchmark's CPU-baseline leg. bf16 tensors travel as ``uint16`` bit patterns;
the composite functions chain the separate steps exactly as the C file's
header states (add -> RMSNorm -> group quant), which is the unfused sequence
the fusion replaces (sglang PR "[AMD] Add fused all-reduce RMSNorm per-group
quant for Qwen3.5 FP8", Fallback order, item 2).

Parity of every function here is pinned by ``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None
_i64 = ctypes.c_int64
_p = ctypes.c_void_p

SCALE_ROW_MAJOR = 0
SCALE_COL_MAJOR = 1
SCALE_COL_MAJOR_PAD4 = 2


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Loads a compiled oracle and declares its signatures."""
    L = ctypes.CDLL(path)
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_mx_exponent.argtypes = [ctypes.c_float]
    L.oracle_mx_exponent.restype = ctypes.c_int
    for name in ("oracle_e4m3_encode_array", "oracle_e4m3_decode_array",
                 "oracle_e2m1_encode_array", "oracle_e2m1_decode_array",
                 "oracle_mx_exponent_array", "oracle_bf16_round_array"):
        getattr(L, name).argtypes = [_p, _i64, _p]
        getattr(L, name).restype = None
    L.oracle_add_residual.argtypes = [_p, _i64, _p, _i64, _i64, _i64, _p, _i64, ctypes.c_int]
    L.oracle_add_residual.restype = ctypes.c_int
    L.oracle_rmsnorm.argtypes = [_p, _i64, _p, ctypes.c_float, _i64, _i64, _p, _i64, _p, _p,
                                 ctypes.c_int]
    L.oracle_rmsnorm.restype = ctypes.c_int
    L.oracle_group_quant_fp8.argtypes = [_p, _i64, _i64, _i64, _i64, ctypes.c_int, _p, _i64, _p,
                                         ctypes.c_int]
    L.oracle_group_quant_fp8.restype = ctypes.c_int
    L.oracle_group_quant_mxfp4.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _i64, ctypes.c_int]
    L.oracle_group_quant_mxfp4.restype = ctypes.c_int
    L.oracle_mx_scale_tiles.argtypes = [_p, _i64, _i64, _p]
    L.oracle_mx_scale_tiles.restype = ctypes.c_int
    L.oracle_mxfp4_gemm.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _p, ctypes.c_int]
    L.oracle_mxfp4_gemm.restype = ctypes.c_int
    return L


# ------------------------------------------------------------ conversions

def as_u16(a) -> np.ndarray:
    """bf16 bit patterns as a numpy uint16 array (accepts torch bf16 tensors)."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bits as uint16, got {a.dtype}")
    return a


def _rows(a: np.ndarray):
    """(pointer, leading dimension in elements) of a 2-D array with unit inner stride."""
    if a.ndim != 2 or a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        raise ValueError("expected a 2-D row-major array with contiguous rows")
    return a.ctypes.data, a.strides[0] // a.itemsize


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (as_u16(u16).astype(np.uint32) << 16).view(np.float32)


def _elementwise(name, src, src_dtype, out_dtype):
    src = np.ascontiguousarray(src, dtype=src_dtype)
    out = np.empty(src.shape, dtype=out_dtype)
    getattr(lib(), name)(src.ctypes.data, src.size, out.ctypes.data)
    return out


def e4m3_encode(v) -> np.ndarray:
    return _elementwise("oracle_e4m3_encode_array", v, np.float32, np.uint8)


def e4m3_decode(c) -> np.ndarray:
    return _elementwise("oracle_e4m3_decode_array", c, np.uint8, np.float32)


def e2m1_encode(v) -> np.ndarray:
    return _elementwise("oracle_e2m1_encode_array", v, np.float32, np.uint8)


def e2m1_decode(c) -> np.ndarray:
    return _elementwise("oracle_e2m1_decode_array", c, np.uint8, np.float32)


def mx_exponent(amax) -> np.ndarray:
    return _elementwise("oracle_mx_exponent_array", amax, np.float32, np.int32)


def bf16_round(v) -> np.ndarray:
    return _elementwise("oracle_bf16_round_array", v, np.float32, np.uint16)


# ------------------------------------------------------------------ steps

def add_residual(x, res, nthreads: int | None = None) -> np.ndarray:
    x, res = as_u16(x), as_u16(res)
    if x.shape != res.shape:
        raise ValueError("x and residual shapes differ")
    M, H = x.shape
    r = np.empty((M, H), dtype=np.uint16)
    px, ldx = _rows(x)
    pr, ldr = _rows(res)
    rc = lib().oracle_add_residual(px, ldx, pr, ldr, M, H, r.ctypes.data, H,
                                   nthreads or default_threads())
    if rc:
        raise ValueError("oracle_add_residual rejected its arguments")
    return r


def rmsnorm(r, gamma, eps: float, nthreads: int | None = None):
    """Returns (y bf16 bits [M,H], inv_rms fp32 [M], margin fp64 [M])."""
    r = as_u16(r)
    gamma = np.ascontiguousarray(as_u16(gamma))
    M, H = r.shape
    if gamma.shape != (H,):
        raise ValueError("gamma must have shape [H]")
    y = np.empty((M, H), dtype=np.uint16)
    inv = np.empty(M, dtype=np.float32)
    margin = np.empty(M, dtype=np.float64)
    pr, ldr = _rows(r)
    rc = lib().oracle_rmsnorm(pr, ldr, gamma.ctypes.data, ctypes.c_float(eps), M, H,
                              y.ctypes.data, H, inv.ctypes.data, margin.ctypes.data,
                              nthreads or default_threads())
    if rc:
        raise ValueError("oracle_rmsnorm rejected its arguments")
    return y, inv, margin


def group_quant_fp8(y, group: int = 128, layout: int = SCALE_ROW_MAJOR,
                    nthreads: int | None = None):
    """Returns (q e4m3 codes [M,H] uint8, scale fp32 [M,H/G] or [H/G,M])."""
    y = as_u16(y)
    M, H = y.shape
    if H % group:
        raise ValueError("H must be a multiple of the group size")
    q = np.empty((M, H), dtype=np.uint8)
    if layout == SCALE_ROW_MAJOR:
        shape = (M, H // group)
    elif layout == SCALE_COL_MAJOR:
        shape = (H // group, M)
    else:
        shape = (H // group, (M + 3) // 4 * 4)
    scale = np.full(shape, np.nan, dtype=np.float32)     # padding stays NaN
    py, ldy = _rows(y)
    rc = lib().oracle_group_quant_fp8(py, ldy, M, H, group, layout, q.ctypes.data, H,
                                      scale.ctypes.data, nthreads or default_threads())
    if rc:
        raise ValueError("oracle_group_quant_fp8 rejected its arguments")
    return q, scale


def group_quant_mxfp4(y, nthreads: int | None = None):
    """Returns (q packed e2m1 [M,H/2] uint8, E8M0 scale bytes [M,H/32])."""
    y = as_u16(y)
    M, H = y.shape
    if H % 32:
        raise ValueError("H must be a multiple of 32")
    q = np.empty((M, H // 2), dtype=np.uint8)
    scale = np.empty((M, H // 32), dtype=np.uint8)
    py, ldy = _rows(y)
    rc = lib().oracle_group_quant_mxfp4(py, ldy, M, H, q.ctypes.data, H // 2, scale.ctypes.data,
                                        H // 32, nthreads or default_threads())
    if rc:
        raise ValueError("oracle_group_quant_mxfp4 rejected its arguments")
    return q, scale


# ------------------------------------------------------------- composites

def _layout_code(layout) -> int:
    if layout in ("row", SCALE_ROW_MAJOR):
        return SCALE_ROW_MAJOR
    if layout in ("col", SCALE_COL_MAJOR):
        return SCALE_COL_MAJOR
    if layout in ("col_pad4", SCALE_COL_MAJOR_PAD4):
        return SCALE_COL_MAJOR_PAD4
    raise ValueError(f"unknown scale layout {layout!r}")


def mx_scale_tiles(scale, fill: int = 0) -> np.ndarray:
    """Row-major [M, G] E8M0 bytes -> the block-scaled MMA tile layout
    (ceil(M/128) * ceil(G/4) * 512 bytes; padding bytes are ``fill``)."""
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    M, G = scale.shape
    out = np.full(((M + 127) // 128) * ((G + 3) // 4) * 512, fill, dtype=np.uint8)
    if lib().oracle_mx_scale_tiles(scale.ctypes.data, M, G, out.ctypes.data):
        raise ValueError("oracle_mx_scale_tiles rejected its arguments")
    return out


def add_rmsnorm_quant_fp8(x, residual, gamma, eps: float = 1e-6, group: int = 128,
                          layout="row", nthreads: int | None = None) -> dict:
    """add, then RMSNorm, then FP8 quantisation by groups: each step a separate oracle call."""
    x = as_u16(x)
    if residual is not None:
        r = add_residual(x, residual, nthreads)
    else:
        r = x
    y, inv, margin = rmsnorm(r, gamma, eps, nthreads)
    q, scale = group_quant_fp8(y, group, _layout_code(layout), nthreads)
    out = {"q": q, "scale": scale, "y": y, "inv": inv, "margin": margin}
    if residual is not None:
        out["residual_out"] = r
    return out


def qknorm_quant_fp8(q_a, kv_a, gamma_q, gamma_kv, eps: float = 1e-6, group: int = 128,
                     layout="row", nthreads: int | None = None) -> dict:
    """Each latent normalised with its own gamma and quantised separately."""
    a = add_rmsnorm_quant_fp8(q_a, None, gamma_q, eps, group, layout, nthreads)
    b = add_rmsnorm_quant_fp8(kv_a, None, gamma_kv, eps, group, layout, nthreads)
    return {"q": a, "kv": b}


def add_rmsnorm_quant_mxfp4(x, residual, gamma, eps: float = 1e-6,
                            nthreads: int | None = None) -> dict:
    x = as_u16(x)
    r = add_residual(x, residual, nthreads) if residual is not None else x
    y, inv, margin = rmsnorm(r, gamma, eps, nthreads)
    q, scale = group_quant_mxfp4(y, nthreads)
    out = {"q": q, "scale": scale, "y": y, "inv": inv, "margin": margin}
    if residual is not None:
        out["residual_out"] = r
    return out


def qknorm_quant_mxfp4(q_a, kv_a, gamma_q, gamma_kv, eps: float = 1e-6,
                       nthreads: int | None = None) -> dict:
    """Each latent normalised with its own gamma and MXFP4-quantised separately."""
    return {"q": add_rmsnorm_quant_mxfp4(q_a, None, gamma_q, eps, nthreads),
            "kv": add_rmsnorm_quant_mxfp4(kv_a, None, gamma_kv, eps, nthreads)}


# ------------------------------------------------------- consumer GEMM

def mxfp4_gemm(a_q, a_scale, b_q, b_scale, nthreads: int | None = None) -> dict:
    """D = A B^T on MXFP4 operands: a_q [M, K/2], a_scale [M, K/32], b_q
    [N, K/2], b_scale [N, K/32] (packed codes and row-major E8M0 bytes).
    Returns {"d64": exact fp64 [M,N], "abs": sum |term| [M,N], "d": bf16 bits
    [M,N] = bf16(f32(d64))}."""
    a_q, a_scale = np.ascontiguousarray(a_q, np.uint8), np.ascontiguousarray(a_scale, np.uint8)
    b_q, b_scale = np.ascontiguousarray(b_q, np.uint8), np.ascontiguousarray(b_scale, np.uint8)
    M, K = a_q.shape[0], a_q.shape[1] * 2
    N = b_q.shape[0]
    if b_q.shape != (N, K // 2) or a_scale.shape != (M, K // 32) or b_scale.shape != (N, K // 32):
        raise ValueError("operand shapes do not agree")
    d64 = np.empty((M, N), dtype=np.float64)
    mag = np.empty((M, N), dtype=np.float64)
    d = np.empty((M, N), dtype=np.uint16)
    rc = lib().oracle_mxfp4_gemm(a_q.ctypes.data, a_scale.ctypes.data, b_q.ctypes.data,
                                 b_scale.ctypes.data, M, N, K, d64.ctypes.data, mag.ctypes.data,
                                 d.ctypes.data, nthreads or default_threads())
    if rc:
        raise ValueError("oracle_mxfp4_gemm rejected its arguments")
    return {"d64": d64, "abs": mag, "d": d}


def a16wfp4_gemm(a_bf16, b_q, b_scale, nthreads: int | None = None) -> dict:
    """The "prequant" placement: the bf16 activation is MXFP4-quantised (the
    same group quant as step 3b) and then multiplied; returns mxfp4_gemm's
    dict plus the activation codes and scales."""
    q, s = group_quant_mxfp4(a_bf16, nthreads)
    out = mxfp4_gemm(q, s, b_q, b_scale, nthreads)
    out["a_q"], out["a_scale"] = q, s
    return out
