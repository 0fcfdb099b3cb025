"""Python binding of librmsq (include/rmsq.h): argument marshalling only.

torch supplies device memory and the current stream; every step of the
computation runs in the library's CUDA kernels. The shared library must have
been built (``python -m mxfp4_activation_quant_gb300.build``); without it
every call raises -- there is no other implementation to fall back to.

Return values follow the tuple forms of sglang PR "[AMD] Add fused
all-reduce RMSNorm per-group quant for Qwen3.5 FP8" (Modifications):
``((q, scale), residual)`` or, with ``keep_bf16``, ``((y, q, scale), residual)``.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# RMSQ_DEBUG=1 selects the bounds-checking debug build (tests only)
LIB_PATH = os.path.join(HERE, "_build",
                        "librmsq_debug.so" if os.environ.get("RMSQ_DEBUG") == "1" else "librmsq.so")

RMSQ_OK = 0
STATUS_NAMES = {0: "RMSQ_OK", 1: "RMSQ_ERR_INVALID_ARG", 2: "RMSQ_ERR_MISALIGNED",
                3: "RMSQ_ERR_UNSUPPORTED", 4: "RMSQ_ERR_CUDA", 5: "RMSQ_ERR_TIMEOUT", 6: "RMSQ_ERR_BOUNDS"}
KERNEL_AUTO, KERNEL_ROWS, KERNEL_PERSISTENT = 0, 1, 2
FORM_AUTO, FORM_THROUGHPUT, FORM_LATENCY = 0, 1, 2
SCALE_ROW_MAJOR, SCALE_COL_MAJOR, SCALE_COL_MAJOR_PAD4 = 0, 1, 2

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f = ctypes.c_float


class LaunchOpts(ctypes.Structure):
    """Mirror of ``rmsq_launch_opts``."""
    _fields_ = [("kernel", _i32), ("vpt", _i32), ("rows_per_block", _i32), ("grid", _i32),
                ("debug_skip_row", _i64), ("wait_limit_ns", _i64), ("form", _i32), ("split", _i32)]

    def __init__(self, kernel=KERNEL_AUTO, vpt=0, rows_per_block=0, grid=0, debug_skip_row=-1,
                 wait_limit_ns=0, form=FORM_AUTO, split=0):
        super().__init__(kernel, vpt, rows_per_block, grid, debug_skip_row, wait_limit_ns, form, split)


class GemmOpts(ctypes.Structure):
    """Mirror of ``rmsq_gemm_opts``."""
    _fields_ = [("bn", _i32), ("ksplit", _i32), ("wait_limit_ns", _i64), ("debug_stall_stage", _i32),
                ("schedule", _i32)]

    def __init__(self, bn=0, ksplit=0, wait_limit_ns=0, debug_stall_stage=0, schedule=0):
        super().__init__(bn, ksplit, wait_limit_ns, debug_stall_stage, schedule)


class GemmPlan(ctypes.Structure):
    """Mirror of ``rmsq_gemm_plan``."""
    _fields_ = [("bn", _i32), ("ksplit", _i32), ("schedule", _i32), ("persistent_ctas", _i32)]


class RmsqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None

_SIGNATURES = {
    "rmsq_add_rmsnorm_quant_group_fp8": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _i32, _p, _p, _i32, _p, _p, _p],
    "rmsq_add_rmsnorm_quant_group_fp8_ex": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _i32, _p, _p, _i32, _p, _p, _p, _p],
    "rmsq_qknorm_quant_fp8": [_p, _i64, _p, _i64, _p, _p, _f, _i64, _i64, _i64, _i32, _p, _p, _p, _p, _i32, _p, _p, _p],
    "rmsq_add_rmsnorm_quant_mxfp4": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _p, _p, _p, _p, _p],
    "rmsq_add_rmsnorm_quant_mxfp4_ex": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _p, _p, _p, _p, _p, _p],
    "rmsq_qknorm_quant_mxfp4": [_p, _i64, _p, _i64, _p, _p, _f, _i64, _i64, _i64, _p, _p, _p, _p, _p, _p, _p],
    "rmsq_add_rmsnorm_quant_mxfp4_mma_scales": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _p, _p, _p, _p, _p],
    "rmsq_add_rmsnorm": [_p, _i64, _p, _i64, _p, _f, _i64, _i64, _p, _p, _p],
    "rmsq_mxfp4_gemm": [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p],
    "rmsq_mxfp4_gemm_ex": [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p, _p],
    "rmsq_a16wfp4_gemm": [_p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p],
    "rmsq_a16wfp4_gemm_ex": [_p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p, _p],
    "rmsq_gemm_plan_for": [_i32, _i64, _i64, _i64, _p, _i32, _i32, _i32, _p],
    "rmsq_mx_scale_tiles": [_p, _i64, _i64, _i64, _p, ctypes.c_uint8, _p],
    "rmsq_sync_status": [_p],
    "rmsq_copy": [_p, _p, _i64, _p],
    "rmsq_encode_e4m3": [_p, _p, _i64, _p],
    "rmsq_encode_e2m1": [_p, _p, _i64, _p],
    "rmsq_check_group_division": [_p, _p],
    "rmsq_debug_bounds_selftest": [_p],
}


def lib() -> ctypes.CDLL:
    """The loaded librmsq; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librmsq is not built ({LIB_PATH} missing); run "
                               "`python -m mxfp4_activation_quant_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.rmsq_status_string.argtypes = [ctypes.c_int]
        L.rmsq_status_string.restype = ctypes.c_char_p
        L.rmsq_last_error.argtypes = []
        L.rmsq_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != RMSQ_OK:
        raise RmsqError(status, lib().rmsq_last_error().decode())


def _current_index() -> int:
    return torch.cuda.current_device()


def _device_guard(index: int):
    """Makes GPU `index` current for the library call (the C library launches
    on the calling thread's current device); a no-op when it already is."""
    if index == _current_index():
        return contextlib.nullcontext()
    return torch.cuda.device(index)


def _device_index(*tensors) -> int:
    """The one GPU all tensor arguments live on. Tensors on different GPUs are
    refused: a kernel (or a TMA tensor map) given another GPU's address would
    fault without peer access."""
    found = sorted({t.device.index if t.device.index is not None else _current_index()
                    for t in tensors if t is not None and getattr(t, "is_cuda", False)})
    if len(found) > 1:
        raise ValueError(f"all tensor arguments must be on the same GPU (got cuda:{found})")
    return found[0] if found else _current_index()


def _call(tensors, name: str, *args) -> None:
    """Calls library entry point `name` on the GPU that holds `tensors`."""
    with _device_guard(_device_index(*tensors)):
        _check(getattr(lib(), name)(*args))


def _ptr(t):
    """Device address of a tensor argument (None for an absent optional one).
    Host tensors are refused here: a kernel given a host address would fault."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors (got a CPU tensor)")
    return t.data_ptr()


# dtypes a buffer may have, by what the kernels store in it
BF16 = (torch.bfloat16,)
F32 = (torch.float32,)
E4M3_CODES = (torch.uint8, torch.float8_e4m3fn)
BYTES = (torch.uint8,) + tuple(getattr(torch, n) for n in ("float8_e8m0fnu",) if hasattr(torch, n))
E2M1_CODES = (torch.uint8,) + tuple(getattr(torch, n) for n in ("float4_e2m1fn_x2",) if hasattr(torch, n))


def _buf(t, name: str, nbytes: int, dtypes: tuple):
    """Address of a buffer the library addresses without a pitch (gamma, the
    outputs, scale tiles): a contiguous CUDA tensor of one of `dtypes`
    holding at least nbytes bytes, or None when absent. The C calls see only
    pointers, so dtypes and sizes are checked here (an fp32 gamma, say, would
    be read as pairs of bf16 halves)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes; this call needs {nbytes}")
    return t.data_ptr()


def _scale_bytes(M: int, H: int, group: int, layout: int) -> int:
    r, c = scale_shape(M, H, group, layout)
    return 4 * r * c


def _like_x(t, name: str, M: int, H: int) -> int:
    """A second [M, H] bf16 input (the residual); returns its leading dimension."""
    ld = _rows_view(t, name)
    if tuple(t.shape) != (M, H):
        raise ValueError(f"{name} must have the shape of x, [{M}, {H}]")
    return ld


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _rows_view(t: torch.Tensor, name: str) -> int:
    """Checks a bf16 CUDA matrix with unit inner stride; returns its leading dimension."""
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D bf16 CUDA tensor")
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} must have contiguous rows")
    return t.stride(0)


def _layout(scale_layout) -> int:
    return {"row": SCALE_ROW_MAJOR, "col": SCALE_COL_MAJOR, "col_pad4": SCALE_COL_MAJOR_PAD4,
            SCALE_ROW_MAJOR: SCALE_ROW_MAJOR, SCALE_COL_MAJOR: SCALE_COL_MAJOR,
            SCALE_COL_MAJOR_PAD4: SCALE_COL_MAJOR_PAD4}[scale_layout]


def scale_shape(M: int, H: int, group: int, layout: int) -> tuple:
    """Shape of the fp32 scale tensor for a layout (column-major padded: [H/G, M rounded up to 4])."""
    G = H // group if group > 0 else 0
    if layout == SCALE_ROW_MAJOR:
        return (M, G)
    if layout == SCALE_COL_MAJOR:
        return (G, M)
    return (G, (M + 3) // 4 * 4)


def mma_scale_bytes(M: int, H: int) -> int:
    """Bytes of MXFP4 scales in the block-scaled MMA tile layout."""
    return (M + 127) // 128 * ((H // 32 + 3) // 4) * 512


def add_rmsnorm_quant_fp8(x: torch.Tensor, gamma: torch.Tensor, residual: torch.Tensor | None = None,
                          eps: float = 1e-6, group: int = 128, scale_layout="row",
                          keep_bf16: bool = False, out_residual: torch.Tensor | None = None,
                          opts: LaunchOpts | None = None):
    """Residual add + RMSNorm + 1x128 FP8 quant.

    Returns ``((q, scale), residual_out)``, or ``((y, q, scale), residual_out)``
    when ``keep_bf16``; ``residual_out`` is None without a residual. Pass
    ``out_residual=residual`` for the in-place residual update.
    """
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    dev = x.device
    layout = _layout(scale_layout)
    q = torch.empty((M, H), dtype=torch.float8_e4m3fn, device=dev)
    scale = torch.empty(scale_shape(M, H, group, layout), dtype=torch.float32, device=dev)
    res_out = None
    if residual is not None:
        res_out = out_residual if out_residual is not None else torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if keep_bf16 else None
    args = (_ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H, group, _ptr(q),
            _ptr(scale), layout, _buf(res_out, "out_residual", 2 * M * H, BF16), _ptr(y), _stream(dev))
    if opts is None:
        _call((x, gamma, residual, out_residual), "rmsq_add_rmsnorm_quant_group_fp8", *args)
    else:
        _call((x, gamma, residual, out_residual), "rmsq_add_rmsnorm_quant_group_fp8_ex", *args, ctypes.byref(opts))
    return ((y, q, scale) if keep_bf16 else (q, scale)), res_out


def add_rmsnorm_quant_fp8_into(x, gamma, residual, q, scale, res_out=None, y=None, eps: float = 1e-6,
                               group: int = 128, scale_layout="row", opts: LaunchOpts | None = None,
                               stream: int | None = None) -> None:
    """As add_rmsnorm_quant_fp8, writing into caller-allocated outputs (no allocation)."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    st = _stream(x.device) if stream is None else stream
    layout = _layout(scale_layout)
    args = (_ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H, group,
            _buf(q, "q", M * H, E4M3_CODES), _buf(scale, "scale", _scale_bytes(M, H, group, layout), F32), layout,
            _buf(res_out, "res_out", 2 * M * H, BF16), _buf(y, "y", 2 * M * H, BF16), st)
    if opts is None:
        _call((x, gamma, residual, q, scale, res_out, y), "rmsq_add_rmsnorm_quant_group_fp8", *args)
    else:
        _call((x, gamma, residual, q, scale, res_out, y), "rmsq_add_rmsnorm_quant_group_fp8_ex", *args, ctypes.byref(opts))


def add_rmsnorm_quant_mxfp4_into(x, gamma, residual, q, scale, res_out=None, y=None, eps: float = 1e-6,
                                 opts: LaunchOpts | None = None, stream: int | None = None) -> None:
    """As add_rmsnorm_quant_mxfp4, writing into caller-allocated outputs."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    st = _stream(x.device) if stream is None else stream
    args = (_ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H,
            _buf(q, "q", M * (H // 2), E2M1_CODES), _buf(scale, "scale", M * (H // 32), BYTES), _buf(res_out, "res_out", 2 * M * H, BF16),
            _buf(y, "y", 2 * M * H, BF16), st)
    if opts is None:
        _call((x, gamma, residual, q, scale, res_out, y), "rmsq_add_rmsnorm_quant_mxfp4", *args)
    else:
        _call((x, gamma, residual, q, scale, res_out, y), "rmsq_add_rmsnorm_quant_mxfp4_ex", *args, ctypes.byref(opts))


def qknorm_quant_fp8_into(q_a, kv_a, gamma_q, gamma_kv, qq, qs, kq, ks, qy=None, ky=None,
                          eps: float = 1e-6, group: int = 128, scale_layout="row",
                          stream: int | None = None) -> None:
    """As qknorm_quant_fp8, writing into caller-allocated outputs."""
    ldq = _rows_view(q_a, "q_a")
    ldk = _rows_view(kv_a, "kv_a")
    M, Hq = q_a.shape
    Mk, Hkv = kv_a.shape
    if Mk != M:
        raise ValueError("q_a and kv_a must have the same number of rows")
    st = _stream(q_a.device) if stream is None else stream
    layout = _layout(scale_layout)
    _call((q_a, kv_a, gamma_q, gamma_kv, qq, qs, kq, ks, qy, ky), "rmsq_qknorm_quant_fp8",
        _ptr(q_a), ldq, _ptr(kv_a), ldk, _buf(gamma_q, "gamma_q", 2 * Hq, BF16), _buf(gamma_kv, "gamma_kv", 2 * Hkv, BF16),
        eps, M, Hq, Hkv, group, _buf(qq, "qq", M * Hq, E4M3_CODES), _buf(qs, "qs", _scale_bytes(M, Hq, group, layout), F32),
        _buf(kq, "kq", M * Hkv, E4M3_CODES), _buf(ks, "ks", _scale_bytes(M, Hkv, group, layout), F32), layout,
        _buf(qy, "qy", 2 * M * Hq, BF16), _buf(ky, "ky", 2 * M * Hkv, BF16), st)


def qknorm_quant_fp8(q_a: torch.Tensor, kv_a: torch.Tensor, gamma_q: torch.Tensor,
                     gamma_kv: torch.Tensor, eps: float = 1e-6, group: int = 128,
                     scale_layout="row", keep_bf16: bool = False):
    """One launch for the MLA q_a / kv_a latents. Returns ``(q_tuple, kv_tuple)``,
    each ``(q, scale)`` or ``(y, q, scale)``."""
    ldq = _rows_view(q_a, "q_a")
    ldk = _rows_view(kv_a, "kv_a")
    M, Hq = q_a.shape
    Mk, Hkv = kv_a.shape
    if Mk != M:
        raise ValueError("q_a and kv_a must have the same number of rows")
    dev = q_a.device
    layout = _layout(scale_layout)

    def outs(H):
        q = torch.empty((M, H), dtype=torch.float8_e4m3fn, device=dev)
        G = H // group if group > 0 else 0
        s = torch.empty((M, G) if layout == SCALE_ROW_MAJOR else (G, M), dtype=torch.float32, device=dev)
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if keep_bf16 else None
        return q, s, y

    qq, qs, qy = outs(Hq)
    kq, ks, ky = outs(Hkv)
    _call((q_a, kv_a, gamma_q, gamma_kv), "rmsq_qknorm_quant_fp8", _ptr(q_a), ldq, _ptr(kv_a), ldk, _buf(gamma_q, "gamma_q", 2 * Hq, BF16),
                                       _buf(gamma_kv, "gamma_kv", 2 * Hkv, BF16), eps, M, Hq, Hkv, group, _ptr(qq), _ptr(qs), _ptr(kq), _ptr(ks),
                                       layout, _ptr(qy), _ptr(ky), _stream(dev))
    if keep_bf16:
        return (qy, qq, qs), (ky, kq, ks)
    return (qq, qs), (kq, ks)


def qknorm_quant_mxfp4(q_a: torch.Tensor, kv_a: torch.Tensor, gamma_q: torch.Tensor,
                       gamma_kv: torch.Tensor, eps: float = 1e-6, keep_bf16: bool = False):
    """One launch for the MLA latents, MXFP4: ``(q_tuple, kv_tuple)``, each
    ``(q, scale)`` or ``(y, q, scale)`` with q [M, H/2] uint8 and E8M0 scales [M, H/32]."""
    ldq = _rows_view(q_a, "q_a")
    ldk = _rows_view(kv_a, "kv_a")
    M, Hq = q_a.shape
    Mk, Hkv = kv_a.shape
    if Mk != M:
        raise ValueError("q_a and kv_a must have the same number of rows")
    dev = q_a.device

    def outs(H):
        q = torch.empty((M, H // 2), dtype=torch.uint8, device=dev)
        s = torch.empty((M, H // 32), dtype=torch.uint8, device=dev)
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if keep_bf16 else None
        return q, s, y

    qq, qs, qy = outs(Hq)
    kq, ks, ky = outs(Hkv)
    _call((q_a, kv_a, gamma_q, gamma_kv), "rmsq_qknorm_quant_mxfp4", _ptr(q_a), ldq, _ptr(kv_a), ldk, _buf(gamma_q, "gamma_q", 2 * Hq, BF16),
                                         _buf(gamma_kv, "gamma_kv", 2 * Hkv, BF16), eps,
                                         M, Hq, Hkv, _ptr(qq), _ptr(qs), _ptr(kq), _ptr(ks), _ptr(qy),
                                         _ptr(ky), _stream(dev))
    if keep_bf16:
        return (qy, qq, qs), (ky, kq, ks)
    return (qq, qs), (kq, ks)


def qknorm_quant_mxfp4_into(q_a, kv_a, gamma_q, gamma_kv, qq, qs, kq, ks, qy=None, ky=None,
                            eps: float = 1e-6, stream: int | None = None) -> None:
    """As qknorm_quant_mxfp4, writing into caller-allocated outputs: codes
    [M, H/2] uint8 and E8M0 scales [M, H/32] uint8 per latent."""
    ldq = _rows_view(q_a, "q_a")
    ldk = _rows_view(kv_a, "kv_a")
    M, Hq = q_a.shape
    Mk, Hkv = kv_a.shape
    if Mk != M:
        raise ValueError("q_a and kv_a must have the same number of rows")
    st = _stream(q_a.device) if stream is None else stream
    _call((q_a, kv_a, gamma_q, gamma_kv, qq, qs, kq, ks, qy, ky), "rmsq_qknorm_quant_mxfp4",
        _ptr(q_a), ldq, _ptr(kv_a), ldk, _buf(gamma_q, "gamma_q", 2 * Hq, BF16), _buf(gamma_kv, "gamma_kv", 2 * Hkv, BF16),
        eps, M, Hq, Hkv, _buf(qq, "qq", M * (Hq // 2), E2M1_CODES), _buf(qs, "qs", M * (Hq // 32), BYTES),
        _buf(kq, "kq", M * (Hkv // 2), E2M1_CODES), _buf(ks, "ks", M * (Hkv // 32), BYTES), _buf(qy, "qy", 2 * M * Hq, BF16),
        _buf(ky, "ky", 2 * M * Hkv, BF16), st)


def add_rmsnorm_quant_mxfp4(x: torch.Tensor, gamma: torch.Tensor, residual: torch.Tensor | None = None,
                            eps: float = 1e-6, keep_bf16: bool = False,
                            out_residual: torch.Tensor | None = None, opts: LaunchOpts | None = None):
    """Residual add + RMSNorm + MXFP4 quant: q [M, H/2] uint8 (element 2k in
    the low nibble), E8M0 scales [M, H/32] uint8. Same tuple forms as the FP8 call."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    dev = x.device
    q = torch.empty((M, H // 2), dtype=torch.uint8, device=dev)
    scale = torch.empty((M, H // 32), dtype=torch.uint8, device=dev)
    res_out = None
    if residual is not None:
        res_out = out_residual if out_residual is not None else torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if keep_bf16 else None
    args = (_ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H, _ptr(q), _ptr(scale),
            _buf(res_out, "out_residual", 2 * M * H, BF16), _ptr(y), _stream(dev))
    if opts is None:
        _call((x, gamma, residual, out_residual), "rmsq_add_rmsnorm_quant_mxfp4", *args)
    else:
        _call((x, gamma, residual, out_residual), "rmsq_add_rmsnorm_quant_mxfp4_ex", *args, ctypes.byref(opts))
    return ((y, q, scale) if keep_bf16 else (q, scale)), res_out


def add_rmsnorm_quant_mxfp4_mma_scales(x: torch.Tensor, gamma: torch.Tensor,
                                       residual: torch.Tensor | None = None, eps: float = 1e-6,
                                       keep_bf16: bool = False, scale_out: torch.Tensor | None = None):
    """MXFP4 with the E8M0 scales in the block-scaled MMA tile layout (a flat
    uint8 tensor of ``mma_scale_bytes(M, H)``; padding bytes are left as they
    are in ``scale_out``, zero-filled when it is allocated here)."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    dev = x.device
    q = torch.empty((M, H // 2), dtype=torch.uint8, device=dev)
    scale = scale_out if scale_out is not None else torch.zeros(mma_scale_bytes(M, H), dtype=torch.uint8,
                                                                device=dev)
    res_out = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if residual is not None else None
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev) if keep_bf16 else None
    _call((x, gamma, residual, scale_out), "rmsq_add_rmsnorm_quant_mxfp4_mma_scales", _ptr(x), ldx, _ptr(residual), ldr,
                                                         _buf(gamma, "gamma", 2 * H, BF16), eps, M, H, _ptr(q),
                                                         _buf(scale, "scale_out", mma_scale_bytes(M, H), BYTES),
                                                         _ptr(res_out), _ptr(y), _stream(dev))
    return ((y, q, scale) if keep_bf16 else (q, scale)), res_out


def add_rmsnorm(x: torch.Tensor, gamma: torch.Tensor, residual: torch.Tensor | None = None,
                eps: float = 1e-6, out: torch.Tensor | None = None, out_residual: torch.Tensor | None = None,
                stream: int | None = None):
    """Residual add + RMSNorm without quantisation: returns ``(y, residual_out)``
    (``residual_out`` None without a residual). H must be a multiple of 32."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    dev = x.device
    y = out if out is not None else torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    res_out = None
    if residual is not None:
        res_out = out_residual if out_residual is not None else torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    st = _stream(dev) if stream is None else stream
    _call((x, gamma, residual, out, out_residual), "rmsq_add_rmsnorm", _ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H,
                                  _buf(res_out, "out_residual", 2 * M * H, BF16), _buf(y, "out", 2 * M * H, BF16), st)
    return y, res_out


def mx_scale_tiles(scale: torch.Tensor, fill: int = 0, stream: int | None = None) -> torch.Tensor:
    """Row-major [R, G] E8M0 bytes (uint8 CUDA) -> the block-scaled MMA tile
    layout (flat uint8, ceil(R/128) * ceil(G/4) * 512 bytes, padding = fill)."""
    if not scale.is_cuda or scale.dtype != torch.uint8 or scale.dim() != 2 or scale.stride(1) != 1:
        raise ValueError("scale must be a 2-D uint8 CUDA tensor with contiguous rows")
    R, G = scale.shape
    out = torch.empty((R + 127) // 128 * ((G + 3) // 4) * 512, dtype=torch.uint8, device=scale.device)
    st = _stream(scale.device) if stream is None else stream
    _call((scale,), "rmsq_mx_scale_tiles", _ptr(scale), scale.stride(0), R, G, _ptr(out), fill, st)
    return out


def _codes_view(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError(f"{name} must be a 2-D uint8 CUDA tensor with contiguous rows")
    return t.stride(0)


def _gemm_out(M, N, dev, out):
    if out is None:
        return torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if out.dtype != torch.bfloat16 or out.dim() != 2 or out.shape[0] != M or out.shape[1] != N or out.stride(1) != 1:
        raise ValueError("out must be a [M, N] bf16 tensor with contiguous rows")
    return out


def _gemm_check(check: bool, device) -> None:
    """check=True: wait for the GEMM and raise if one of its bounded waits
    gave up (D is then incomplete); otherwise the caller checks sync_status."""
    if check:
        with _device_guard(torch.device(device).index):
            st = lib().rmsq_sync_status(_stream(device))
        _check(st)


def mxfp4_gemm(a_q: torch.Tensor, a_scale_tiles: torch.Tensor, b_q: torch.Tensor, b_scale_tiles: torch.Tensor,
               out: torch.Tensor | None = None, opts: GemmOpts | None = None, stream: int | None = None,
               check: bool = False):
    """D = A B^T (bf16 [M, N]) on the block-scaled tensor cores, A and B MXFP4:
    codes [rows, K/2] uint8, scales in the MMA tile layout (flat uint8).
    With ``check`` the call waits for the GEMM and raises RmsqError if a
    bounded wait inside it ran out (D incomplete); without it, call
    ``sync_status`` before trusting D when the GPU may have been stalled."""
    lda, ldb = _codes_view(a_q, "a_q"), _codes_view(b_q, "b_q")
    M, K = a_q.shape[0], a_q.shape[1] * 2
    N = b_q.shape[0]
    if b_q.shape[1] * 2 != K:
        raise ValueError("A and B have different K")
    d = _gemm_out(M, N, a_q.device, out)
    st = _stream(a_q.device) if stream is None else stream
    args = (_ptr(a_q), lda, _buf(a_scale_tiles, "a_scale_tiles", mma_scale_bytes(M, K), BYTES), _ptr(b_q), ldb,
            _buf(b_scale_tiles, "b_scale_tiles", mma_scale_bytes(N, K), BYTES), _ptr(d), d.stride(0),
            M, N, K, st)
    if opts is None:
        _call((a_q, a_scale_tiles, b_q, b_scale_tiles, out), "rmsq_mxfp4_gemm", *args)
    else:
        _call((a_q, a_scale_tiles, b_q, b_scale_tiles, out), "rmsq_mxfp4_gemm_ex", *args, ctypes.byref(opts))
    _gemm_check(check, a_q.device)
    return d


def a16wfp4_gemm(a: torch.Tensor, b_q: torch.Tensor, b_scale_tiles: torch.Tensor,
                 out: torch.Tensor | None = None, opts: GemmOpts | None = None, stream: int | None = None,
                 check: bool = False):
    """The prequant placement: A bf16 [M, K] is MXFP4-quantised inside the
    GEMM (same rule as add_rmsnorm_quant_mxfp4), then D = A B^T (bf16 [M, N]).
    ``check`` as for mxfp4_gemm."""
    lda = _rows_view(a, "a")
    ldb = _codes_view(b_q, "b_q")
    M, K = a.shape
    N = b_q.shape[0]
    if b_q.shape[1] * 2 != K:
        raise ValueError("A and B have different K")
    d = _gemm_out(M, N, a.device, out)
    st = _stream(a.device) if stream is None else stream
    args = (_ptr(a), lda, _ptr(b_q), ldb, _buf(b_scale_tiles, "b_scale_tiles", mma_scale_bytes(N, K), BYTES), _ptr(d),
            d.stride(0), M, N, K, st)
    if opts is None:
        _call((a, b_q, b_scale_tiles, out), "rmsq_a16wfp4_gemm", *args)
    else:
        _call((a, b_q, b_scale_tiles, out), "rmsq_a16wfp4_gemm_ex", *args, ctypes.byref(opts))
    _gemm_check(check, a.device)
    return d


def gemm_plan(M: int, N: int, K: int, *, sms: int, pairs_256: int, pairs_192: int, prequant: bool = False,
              opts: GemmOpts | None = None) -> GemmPlan:
    """The launch mxfp4_gemm (or, with prequant, a16wfp4_gemm) makes for an
    M x N x K product on a device with ``sms`` SMs that holds ``pairs_256`` /
    ``pairs_192`` CTA pairs at once: B-tile width, K split, schedule (1 one
    tile per CTA, 2 persistent, 3 CTA pairs) and persistent grid size. Host
    arithmetic only (rmsq_gemm_plan_for); raises on the arguments the GEMM
    calls reject."""
    plan = GemmPlan()
    o = ctypes.byref(opts) if opts is not None else None
    _check(lib().rmsq_gemm_plan_for(1 if prequant else 0, M, N, K, o, sms, pairs_256, pairs_192,
                                    ctypes.byref(plan)))
    return plan


def add_rmsnorm_quant_mxfp4_mma_scales_into(x, gamma, residual, q, scale_tiles, res_out=None, y=None,
                                            eps: float = 1e-6, stream: int | None = None) -> None:
    """As add_rmsnorm_quant_mxfp4_mma_scales, writing into caller-allocated outputs."""
    ldx = _rows_view(x, "x")
    M, H = x.shape
    ldr = _like_x(residual, "residual", M, H) if residual is not None else 0
    st = _stream(x.device) if stream is None else stream
    _call((x, gamma, residual, q, scale_tiles, res_out, y), "rmsq_add_rmsnorm_quant_mxfp4_mma_scales",
        _ptr(x), ldx, _ptr(residual), ldr, _buf(gamma, "gamma", 2 * H, BF16), eps, M, H, _buf(q, "q", M * (H // 2), E2M1_CODES),
        _buf(scale_tiles, "scale_tiles", mma_scale_bytes(M, H), BYTES), _buf(res_out, "res_out", 2 * M * H, BF16),
        _buf(y, "y", 2 * M * H, BF16), st)


def copy_(dst: torch.Tensor, src: torch.Tensor, stream: int | None = None) -> None:
    """dst <- src with the library's streaming copy kernel (both contiguous
    CUDA tensors of the same byte size, a multiple of 16)."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must have the same size in bytes")
    for t, name in ((src, "src"), (dst, "dst")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    st = _stream(src.device) if stream is None else stream
    _call((src, dst), "rmsq_copy", _ptr(src), _ptr(dst), nbytes, st)


def sync_status(device=None) -> int:
    """Synchronises the device's current stream and returns the verdict of
    the library's status word on that device (process-wide: it covers the
    library's kernels on every stream of the device)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    index = dev.index if dev.index is not None else _current_index()
    with _device_guard(index):
        return lib().rmsq_sync_status(_stream(dev))


def encode_e4m3(v: torch.Tensor) -> torch.Tensor:
    """The kernels' E4M3 conversion applied elementwise (fp32 CUDA tensor -> uint8)."""
    if v.dtype != torch.float32:
        raise ValueError("v must be float32")
    v = v.contiguous()
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _call((v,), "rmsq_encode_e4m3", _ptr(v), _ptr(out), v.numel(), _stream(v.device))
    return out


def encode_e2m1(v: torch.Tensor) -> torch.Tensor:
    """The kernels' E2M1 conversion applied elementwise (one code per byte)."""
    if v.dtype != torch.float32:
        raise ValueError("v must be float32")
    v = v.contiguous()
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _call((v,), "rmsq_encode_e2m1", _ptr(v), _ptr(out), v.numel(), _stream(v.device))
    return out


def check_group_division(device=None) -> dict:
    """Runs the library's exhaustive division self-check; returns its counters."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    counts = torch.zeros(5, dtype=torch.int64, device=dev)
    _check(lib().rmsq_check_group_division(_ptr(counts), _stream(dev)))
    c = counts.cpu().tolist()
    return {"code_mismatches": c[0], "quotient_mismatches": c[1], "pairs": c[2], "scale_mismatches": c[3],
            "quotient_mismatches_y_ge_2m100": c[4]}
