"""The Python binding's argument marshalling, without a GPU: duck-typed
stand-ins for CUDA tensors go in, a recording stand-in for the C library
takes the call. Buffers sized exactly as the calls need them reach the
library in the declared argument order; a buffer one element short, a
non-contiguous output, a residual of another shape or a kv_a with other rows
is refused before the library is called (a kernel given it would read or
write out of bounds)."""

import math

import pytest
import torch

from mxfp4_activation_quant_gb300 import rmsq

BF16, U8, F32, F8 = torch.bfloat16, torch.uint8, torch.float32, torch.float8_e4m3fn


class FakeCuda:
    """What the binding reads of a CUDA tensor: shape, dtype, strides, size,
    address, device."""
    is_cuda = True
    _next = 1 << 32

    def __init__(self, shape, dtype, strides=None, device=0):
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device("cuda", device)
        dense, acc = [], 1
        for n in reversed(self.shape):
            dense.insert(0, acc)
            acc *= n
        self._dense = tuple(dense)
        self._strides = tuple(strides) if strides is not None else self._dense
        FakeCuda._next += 1 << 24
        self.addr = FakeCuda._next

    def dim(self):
        return len(self.shape)

    def stride(self, i=None):
        return self._strides if i is None else self._strides[i]

    def is_contiguous(self):
        return self._strides == self._dense

    def numel(self):
        return math.prod(self.shape)

    def element_size(self):
        return torch.empty((), dtype=self.dtype).element_size()

    def data_ptr(self):
        return self.addr


class FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


class FakeGuard:
    """Records which GPU the binding makes current around a library call."""
    def __init__(self, lib, index):
        self.lib, self.index = lib, index

    def __enter__(self):
        self.lib.devices.append(self.index)

    def __exit__(self, *exc):
        return False


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    lib.devices = []
    monkeypatch.setattr(rmsq, "lib", lambda: lib)
    monkeypatch.setattr(rmsq, "_current_index", lambda: 0)
    monkeypatch.setattr(rmsq, "_device_guard", lambda index: FakeGuard(lib, index))
    return lib


M, H, HQ, HKV, N, K = 5, 256, 1536, 512, 64, 512


def fp8_into_args():
    return dict(x=FakeCuda((M, H), BF16), gamma=FakeCuda((H,), BF16), residual=FakeCuda((M, H), BF16),
                q=FakeCuda((M, H), F8), scale=FakeCuda((M, H // 128), F32), res_out=FakeCuda((M, H), BF16),
                y=FakeCuda((M, H), BF16))


def mx_into_args():
    return dict(x=FakeCuda((M, H), BF16), gamma=FakeCuda((H,), BF16), residual=FakeCuda((M, H), BF16),
                q=FakeCuda((M, H // 2), U8), scale=FakeCuda((M, H // 32), U8), res_out=FakeCuda((M, H), BF16),
                y=FakeCuda((M, H), BF16))


def mma_into_args():
    return dict(x=FakeCuda((M, H), BF16), gamma=FakeCuda((H,), BF16), residual=FakeCuda((M, H), BF16),
                q=FakeCuda((M, H // 2), U8), scale_tiles=FakeCuda((rmsq.mma_scale_bytes(M, H),), U8),
                res_out=FakeCuda((M, H), BF16), y=FakeCuda((M, H), BF16))


def qk_into_args():
    return dict(q_a=FakeCuda((M, HQ), BF16), kv_a=FakeCuda((M, HKV), BF16), gamma_q=FakeCuda((HQ,), BF16),
                gamma_kv=FakeCuda((HKV,), BF16), qq=FakeCuda((M, HQ), F8), qs=FakeCuda((HQ // 128, M), F32),
                kq=FakeCuda((M, HKV), F8), ks=FakeCuda((HKV // 128, M), F32), qy=FakeCuda((M, HQ), BF16),
                ky=FakeCuda((M, HKV), BF16))


def qk_mx_into_args():
    return dict(q_a=FakeCuda((M, HQ), BF16), kv_a=FakeCuda((M, HKV), BF16), gamma_q=FakeCuda((HQ,), BF16),
                gamma_kv=FakeCuda((HKV,), BF16), qq=FakeCuda((M, HQ // 2), U8), qs=FakeCuda((M, HQ // 32), U8),
                kq=FakeCuda((M, HKV // 2), U8), ks=FakeCuda((M, HKV // 32), U8), qy=FakeCuda((M, HQ), BF16),
                ky=FakeCuda((M, HKV), BF16))


def norm_args():
    return dict(x=FakeCuda((M, H), BF16), gamma=FakeCuda((H,), BF16), residual=FakeCuda((M, H), BF16),
                out=FakeCuda((M, H), BF16), out_residual=FakeCuda((M, H), BF16))


def gemm_args():
    return dict(a_q=FakeCuda((M, K // 2), U8), a_scale_tiles=FakeCuda((rmsq.mma_scale_bytes(M, K),), U8),
                b_q=FakeCuda((N, K // 2), U8), b_scale_tiles=FakeCuda((rmsq.mma_scale_bytes(N, K),), U8),
                out=FakeCuda((M, N), BF16))


def pre_args():
    return dict(a=FakeCuda((M, K), BF16), b_q=FakeCuda((N, K // 2), U8),
                b_scale_tiles=FakeCuda((rmsq.mma_scale_bytes(N, K),), U8), out=FakeCuda((M, N), BF16))


CALLS = {
    "fp8": (lambda a: rmsq.add_rmsnorm_quant_fp8_into(**a, stream=0), fp8_into_args),
    "fp8_col": (lambda a: rmsq.add_rmsnorm_quant_fp8_into(**a, scale_layout="col", stream=0),
                lambda: {**fp8_into_args(), "scale": FakeCuda((H // 128, M), F32)}),
    "fp8_col_pad4": (lambda a: rmsq.add_rmsnorm_quant_fp8_into(**a, scale_layout="col_pad4", stream=0),
                     lambda: {**fp8_into_args(), "scale": FakeCuda((H // 128, 8), F32)}),
    "mxfp4": (lambda a: rmsq.add_rmsnorm_quant_mxfp4_into(**a, stream=0), mx_into_args),
    "mma_scales": (lambda a: rmsq.add_rmsnorm_quant_mxfp4_mma_scales_into(**a, stream=0), mma_into_args),
    "qknorm": (lambda a: rmsq.qknorm_quant_fp8_into(**a, scale_layout="col", stream=0), qk_into_args),
    "qknorm_mx": (lambda a: rmsq.qknorm_quant_mxfp4_into(**a, stream=0), qk_mx_into_args),
    "norm": (lambda a: rmsq.add_rmsnorm(**a, stream=0), norm_args),
    "gemm": (lambda a: rmsq.mxfp4_gemm(**a, stream=0), gemm_args),
    "prequant": (lambda a: rmsq.a16wfp4_gemm(**a, stream=0), pre_args),
}

INPUTS_WITH_A_PITCH = {"x", "residual", "q_a", "kv_a", "a_q", "b_q", "a", "out"}


@pytest.mark.parametrize("call", sorted(CALLS))
def test_exact_buffers_reach_the_library(fake, call):
    run, make = CALLS[call]
    args = make()
    run(args)
    assert len(fake.calls) == 1
    name, passed = fake.calls[0]
    # every tensor's address is passed, each exactly once
    for key, t in args.items():
        assert list(passed).count(t.addr) == 1, (call, key)


@pytest.mark.parametrize("call,arg", [(c, a) for c in sorted(CALLS) for a in sorted(CALLS[c][1]())
                                      if a not in INPUTS_WITH_A_PITCH])
def test_short_buffers_are_refused(fake, call, arg):
    run, make = CALLS[call]
    args = make()
    t = args[arg]
    shape = list(t.shape)
    shape[0] -= 1
    args[arg] = FakeCuda(shape, t.dtype)
    with pytest.raises(ValueError, match=arg):
        run(args)
    assert not fake.calls


@pytest.mark.parametrize("call,arg", [("fp8", "q"), ("fp8", "y"), ("mxfp4", "scale"), ("qknorm", "ky"),
                                      ("norm", "out_residual")])
def test_non_contiguous_outputs_are_refused(fake, call, arg):
    run, make = CALLS[call]
    args = make()
    t = args[arg]
    args[arg] = FakeCuda(t.shape, t.dtype, strides=(t.shape[1] + 8, 1))
    with pytest.raises(ValueError, match="contiguous"):
        run(args)
    assert not fake.calls


@pytest.mark.parametrize("call", ["fp8", "mxfp4", "mma_scales", "norm"])
def test_residual_must_have_the_shape_of_x(fake, call):
    run, make = CALLS[call]
    args = make()
    args["residual"] = FakeCuda((M - 1, H), BF16)
    with pytest.raises(ValueError, match="shape of x"):
        run(args)
    assert not fake.calls


@pytest.mark.parametrize("call", ["qknorm", "qknorm_mx"])
def test_kv_rows_must_match_q_rows(fake, call):
    run, make = CALLS[call]
    args = make()
    args["kv_a"] = FakeCuda((M - 1, HKV), BF16)
    with pytest.raises(ValueError, match="same number of rows"):
        run(args)
    assert not fake.calls


def test_declared_argument_order(fake):
    """Spot checks of positions against include/rmsq.h: sizes and pitches
    where the header puts them."""
    a = fp8_into_args()
    rmsq.add_rmsnorm_quant_fp8_into(**a, scale_layout="col", stream=7)
    _, p = fake.calls[-1]
    assert p[:9] == (a["x"].addr, H, a["residual"].addr, H, a["gamma"].addr, 1e-6, M, H, 128)
    assert p[9:] == (a["q"].addr, a["scale"].addr, rmsq.SCALE_COL_MAJOR, a["res_out"].addr, a["y"].addr, 7)
    k = qk_mx_into_args()
    rmsq.qknorm_quant_mxfp4_into(**k, eps=1e-5, stream=3)
    _, p = fake.calls[-1]
    assert p == (k["q_a"].addr, HQ, k["kv_a"].addr, HKV, k["gamma_q"].addr, k["gamma_kv"].addr, 1e-5, M, HQ, HKV,
                 k["qq"].addr, k["qs"].addr, k["kq"].addr, k["ks"].addr, k["qy"].addr, k["ky"].addr, 3)
    g = gemm_args()
    rmsq.mxfp4_gemm(**g, stream=9)
    _, p = fake.calls[-1]
    assert p == (g["a_q"].addr, K // 2, g["a_scale_tiles"].addr, g["b_q"].addr, K // 2, g["b_scale_tiles"].addr,
                 g["out"].addr, N, M, N, K, 9)


def test_encoders_want_float32(fake):
    with pytest.raises(ValueError, match="float32"):
        rmsq.encode_e4m3(FakeCuda((4,), BF16))
    with pytest.raises(ValueError, match="float32"):
        rmsq.encode_e2m1(FakeCuda((4,), torch.float16))


@pytest.mark.parametrize("call", sorted(CALLS))
def test_tensors_on_two_gpus_are_refused(fake, call):
    """One argument on another GPU: refused before the library sees an
    address it cannot reach."""
    run, make = CALLS[call]
    args = make()
    key = sorted(args)[-1]
    t = args[key]
    args[key] = FakeCuda(t.shape, t.dtype, device=1)
    with pytest.raises(ValueError, match="same GPU"):
        run(args)
    assert not fake.calls


@pytest.mark.parametrize("call", sorted(CALLS))
def test_call_runs_on_the_tensors_gpu(fake, call):
    """All arguments on cuda:1 while cuda:0 is current: the library call is
    made with cuda:1 current (the C library launches on the current device)."""
    run, make = CALLS[call]
    args = {k: FakeCuda(t.shape, t.dtype, t.stride(), device=1) for k, t in make().items()}
    run(args)
    assert len(fake.calls) == 1
    assert fake.devices == [1]


@pytest.mark.parametrize("call,arg,dtype", [
    ("fp8", "gamma", F32),              # read as pairs of bf16 halves
    ("fp8", "y", F32),
    ("fp8", "scale", torch.float16),
    ("fp8", "q", torch.int8),
    ("mxfp4", "scale", F32),
    ("mxfp4", "q", BF16),
    ("mma_scales", "scale_tiles", torch.int32),
    ("qknorm", "gamma_kv", torch.float16),
    ("norm", "out", F32),
    ("gemm", "b_scale_tiles", torch.int8),
])
def test_wrong_dtypes_are_refused(fake, call, arg, dtype):
    run, make = CALLS[call]
    args = make()
    t = args[arg]
    # same byte size as the correct buffer, so only the dtype check can refuse it
    nbytes = t.numel() * t.element_size()
    esize = torch.empty((), dtype=dtype).element_size()
    args[arg] = FakeCuda(((nbytes + esize - 1) // esize,), dtype)
    with pytest.raises(ValueError, match=arg):
        run(args)
    assert not fake.calls
