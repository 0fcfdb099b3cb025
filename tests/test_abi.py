"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments before launching anything (these
calls never reach the GPU, so they run on machines without one)."""

import ctypes
import os
import re

import pytest

from mxfp4_activation_quant_gb300 import build as lib_build
from mxfp4_activation_quant_gb300 import rmsq

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "rmsq.h")


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return rmsq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rmsq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    fns = declared_functions()
    for name in ("rmsq_add_rmsnorm_quant_group_fp8", "rmsq_qknorm_quant_fp8",
                 "rmsq_add_rmsnorm_quant_mxfp4"):
        assert name in fns


def test_every_declared_symbol_is_exported(L):
    missing = [f for f in declared_functions() if not hasattr(L, f)]
    assert not missing, missing


def _kind_of_c(param: str) -> str:
    if "*" in param:
        return "ptr"
    base = param.split()[-2] if len(param.split()) > 1 else param
    return {"int64_t": "i64", "int32_t": "i32", "int": "i32", "float": "f32", "uint8_t": "u8"}[base]


def _kind_of_ctypes(t) -> str:
    return {ctypes.c_void_p: "ptr", ctypes.c_char_p: "ptr", ctypes.c_int64: "i64", ctypes.c_int32: "i32",
            ctypes.c_float: "f32", ctypes.c_uint8: "u8"}[t]


def test_binding_signatures_match_the_header():
    """Every function the header declares has a ctypes signature in the
    binding (the two error-reporting calls aside), with the same number of
    arguments and the same kind (pointer, int64, int32, float, byte) at every
    position, so no call passes its arguments in the wrong registers."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"\b(rmsq_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text)
    checked = 0
    for name, params in decls:
        if name in ("rmsq_status_string", "rmsq_last_error"):
            continue
        assert name in rmsq._SIGNATURES, f"{name} has no ctypes signature"
        want = [_kind_of_c(p.strip()) for p in params.split(",")] if params.strip() not in ("", "void") else []
        got = [_kind_of_ctypes(t) for t in rmsq._SIGNATURES[name]]
        assert got == want, (name, want, got)
        checked += 1
    assert checked == len(rmsq._SIGNATURES)


def test_binding_structs_match_the_header():
    """Each struct the header defines has a ctypes mirror with the same
    fields, in the same order, of the same widths."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    structs = dict(re.findall(r"typedef struct (rmsq_[a-z_]+) \{([^}]*)\}", text))
    mirrors = {"rmsq_launch_opts": rmsq.LaunchOpts, "rmsq_gemm_opts": rmsq.GemmOpts, "rmsq_gemm_plan": rmsq.GemmPlan}
    assert set(structs) == set(mirrors)
    for name, body in structs.items():
        want = [(f.split()[1], _kind_of_c(f)) for f in (x.strip() for x in body.split(";")) if f]
        got = [(fname, _kind_of_ctypes(t)) for fname, t in mirrors[name]._fields_]
        assert got == want, (name, want, got)


def test_status_strings(L):
    for s in range(7):
        assert L.rmsq_status_string(s)
    assert L.rmsq_status_string(99) == b"unknown status"


# Fake, well-aligned device addresses: every call below must be rejected by
# the host checks, so nothing is ever dereferenced or launched.
BASE = 1 << 40
X, RES, G, Q, S, RO, Y = (BASE + i * (1 << 32) for i in range(7))


def fp8(L, **kw):
    a = dict(x=X, ldx=256, res=RES, ldr=256, gamma=G, eps=1e-6, M=4, H=256, group=128, q=Q, scale=S,
             layout=0, res_out=RO, y=Y)
    a.update(kw)
    return L.rmsq_add_rmsnorm_quant_group_fp8(a["x"], a["ldx"], a["res"], a["ldr"], a["gamma"], a["eps"],
                                              a["M"], a["H"], a["group"], a["q"], a["scale"], a["layout"],
                                              a["res_out"], a["y"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), 1),
    (dict(gamma=None), 1),
    (dict(H=200), 1),                      # not a multiple of 128
    (dict(group=64), 3),                   # FP8 groups other than 128 are not implemented
    (dict(group=0), 1),
    (dict(layout=7), 1),
    (dict(eps=-1.0), 1),
    (dict(eps=float("nan")), 1),
    (dict(M=-1), 1),
    (dict(H=0), 1),
    (dict(res_out=None), 1),               # residual without its output
    (dict(res=None), 1),                   # output without a residual
    (dict(x=X + 2), 2),                    # misaligned base
    (dict(ldx=260), 2),                    # leading dimension not a multiple of 8
    (dict(ldx=128), 1),                    # leading dimension < H
    (dict(q=X + 64), 1),                   # output overlaps x
    (dict(y=Q + 512), 1),                  # two outputs overlap
    (dict(res_out=RES, ldr=264), 1),       # in-place residual needs ld_res == H
    (dict(H=1 << 20), 3),                  # row longer than the kernels handle
])
def test_fp8_rejects_bad_arguments(L, kw, status):
    assert fp8(L, **kw) == status
    assert L.rmsq_last_error()


def test_m_zero_is_a_no_op(L):
    assert fp8(L, M=0) == 0
    assert L.rmsq_add_rmsnorm_quant_mxfp4(X, 256, RES, 256, G, 1e-6, 0, 256, Q, S, RO, Y, None) == 0


def test_mxfp4_rejects_bad_arguments(L):
    call = L.rmsq_add_rmsnorm_quant_mxfp4
    assert call(X, 256, RES, 256, G, 1e-6, 4, 48, Q, S, RO, Y, None) == 1         # H % 32
    assert call(X, 256, RES, 256, None, 1e-6, 4, 256, Q, S, RO, Y, None) == 1     # no gamma
    assert call(X + 8, 256, RES, 256, G, 1e-6, 4, 256, Q, S, RO, Y, None) == 2    # misaligned


def test_qknorm_rejects_bad_arguments(L):
    call = L.rmsq_qknorm_quant_fp8
    args = [X, 1536, RES, 512, G, G + 4096, 1e-6, 8, 1536, 512, 128, Q, S, RO, Y, 0, None, None, None]
    bad = list(args)
    bad[9] = 500                           # Hkv not a multiple of 128
    assert call(*bad) == 1
    bad = list(args)
    bad[13] = Q + 128                      # kv codes overlap q codes
    assert call(*bad) == 1
    bad = list(args)
    bad[10] = 32
    assert call(*bad) == 3


def test_launch_opts_layout_matches_header():
    # int32 kernel, vpt, rows_per_block, grid; int64 debug_skip_row, wait_limit_ns; int32 form, split
    assert ctypes.sizeof(rmsq.LaunchOpts) == 40
    assert rmsq.LaunchOpts.debug_skip_row.offset == 16
    assert rmsq.LaunchOpts.form.offset == 32
    assert rmsq.LaunchOpts.split.offset == 36


def test_host_tensors_are_refused():
    """The binding never hands a kernel the address of host memory."""
    import torch
    with pytest.raises(ValueError, match="CUDA tensors"):
        rmsq._ptr(torch.zeros(4))
    assert rmsq._ptr(None) is None


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(rmsq, "_lib", None)
    monkeypatch.setattr(rmsq, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        rmsq.lib()


def test_gemm_opts_layout_matches_header():
    # int32 bn, ksplit; int64 wait_limit_ns; int32 debug_stall_stage, schedule
    assert ctypes.sizeof(rmsq.GemmOpts) == 24
    assert rmsq.GemmOpts.wait_limit_ns.offset == 8
    assert rmsq.GemmOpts.debug_stall_stage.offset == 16
    assert rmsq.GemmOpts.schedule.offset == 20
    # zero-initialised options are the defaults (the hook is off)
    assert bytes(rmsq.GemmOpts()) == bytes(24)


A_Q, A_S, B_Q, B_S, D = (BASE + i * (1 << 32) for i in range(5))


def gemm(L, pre=False, **kw):
    a = dict(a=A_Q, lda=2048 if pre else 512, a_s=A_S, b=B_Q, ldb=512, b_s=B_S, d=D, ldd=256,
             M=64, N=256, K=1024)
    a.update(kw)
    if pre:
        return L.rmsq_a16wfp4_gemm(a["a"], a["lda"], a["b"], a["ldb"], a["b_s"], a["d"], a["ldd"],
                                   a["M"], a["N"], a["K"], None)
    return L.rmsq_mxfp4_gemm(a["a"], a["lda"], a["a_s"], a["b"], a["ldb"], a["b_s"], a["d"], a["ldd"],
                             a["M"], a["N"], a["K"], None)


@pytest.mark.parametrize("pre", [False, True])
@pytest.mark.parametrize("kw,status", [
    (dict(K=1000), 3),                     # K not a multiple of 256
    (dict(K=0), 1),
    (dict(N=260), 3),                      # N not a multiple of 8
    (dict(M=-1), 1),
    (dict(b=None), 1),
    (dict(b_s=None), 1),
    (dict(d=None), 1),
    (dict(ldb=256), 1),                    # B rows are K/2 = 512 bytes
    (dict(ldd=128), 1),                    # ld_d < N
    (dict(b=B_Q + 8), 2),                  # misaligned
    (dict(ldd=260), 2),                    # ld_d not a multiple of 8
    (dict(d=B_Q + 1024), 1),               # D overlaps B
])
def test_gemm_rejects_bad_arguments(L, pre, kw, status):
    assert gemm(L, pre, **kw) == status
    assert L.rmsq_last_error()


def test_gemm_specific_checks(L):
    assert gemm(L, False, a_s=None) == 1                     # quantised A needs its scales
    assert gemm(L, False, lda=256) == 1                      # A rows are K/2 bytes
    assert gemm(L, True, lda=1000) == 1                      # bf16 A rows are K elements
    assert gemm(L, True, lda=1028) == 2                      # bf16 leading dimension % 8
    assert gemm(L, False, M=0) == 0 and gemm(L, True, N=0) == 0
    for opts in (rmsq.GemmOpts(bn=96), rmsq.GemmOpts(schedule=4), rmsq.GemmOpts(schedule=-1)):
        assert L.rmsq_mxfp4_gemm_ex(A_Q, 512, A_S, B_Q, 512, B_S, D, 256, 64, 256, 1024, None,
                                    ctypes.byref(opts)) == 1


def test_norm_only_and_tiles_reject_bad_arguments(L):
    call = L.rmsq_add_rmsnorm
    assert call(X, 256, RES, 256, G, 1e-6, 4, 256, RO, None, None) == 1    # out_bf16 required
    assert call(X, 256, RES, 256, G, 1e-6, 4, 48, RO, Y, None) == 1        # H % 32
    assert call(X, 256, None, 0, G, 1e-6, 4, 256, RO, Y, None) == 1        # residual output without input
    assert call(X, 256, RES, 256, G, 1e-6, 4, 256, RO, X + 64, None) == 1  # y overlaps x
    assert call(X, 256, RES, 256, G, 1e-6, 0, 256, RO, Y, None) == 0
    tiles = L.rmsq_mx_scale_tiles
    assert tiles(A_S, 4, 10, 8, B_S, 0, None) == 1                         # ld < G
    assert tiles(None, 8, 10, 8, B_S, 0, None) == 1
    assert tiles(A_S, 8, 1000, 8, A_S + 512, 0, None) == 1                 # out overlaps the input
    assert tiles(A_S, 8, 0, 8, B_S, 0, None) == 0


def test_bounds_selftest_needs_the_debug_build(L):
    if os.environ.get("RMSQ_DEBUG") == "1":
        pytest.skip("release-build behaviour")
    assert L.rmsq_debug_bounds_selftest(None) == 3         # RMSQ_ERR_UNSUPPORTED, nothing launched
