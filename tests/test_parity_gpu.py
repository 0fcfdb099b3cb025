"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every test here needs a GPU. Inputs are the seeded workloads of
mxfp4_activation_quant_gb300.synth; the rules are those of tests/parity.py.
"""

import json
import os

import numpy as np
import pytest
import torch

from mxfp4_activation_quant_gb300 import rmsq, synth
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")


def _gpu(d):
    return {k: v.to(DEV) for k, v in d.items()}


def run_fp8(d, w_eps, layout="row", keep=False, residual=True, opts=None):
    g = _gpu(d)
    out, res_out = rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], g.get("residual") if residual else None,
                                              eps=w_eps, scale_layout=layout, keep_bf16=keep, opts=opts)
    torch.cuda.synchronize()
    got = {"q": out[-2], "scale": out[-1], "residual_out": res_out, "y": out[0] if keep else None}
    return got


def ref_fp8(O, d, eps, layout="row", residual=True):
    return O.add_rmsnorm_quant_fp8(d["x"], d.get("residual") if residual else None, d["gamma"], eps,
                                   layout=layout)


def run_mx(d, eps, keep=False, residual=True, opts=None):
    g = _gpu(d)
    out, res_out = rmsq.add_rmsnorm_quant_mxfp4(g["x"], g["gamma"], g.get("residual") if residual else None,
                                                eps=eps, keep_bf16=keep, opts=opts)
    torch.cuda.synchronize()
    return {"q": out[-2], "scale": out[-1], "residual_out": res_out, "y": out[0] if keep else None}


# ------------------------------------------------------------- workloads

@pytest.mark.parametrize("name,M", [("tiny", None), ("decode", None), ("prefill", 300),
                                    ("prefill", 37), ("mxfp4", 129)])
def test_workload_rows(oracle_mod, name, M):
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w, M=M)
    if w.kind == "fp8":
        got = run_fp8(d, w.eps, layout=w.scale_layout, keep=w.keep_bf16)
        ref = ref_fp8(oracle_mod, d, w.eps, layout=w.scale_layout)
        st = parity.compare_fp8(got, ref, w.scale_layout, what=name)
    else:
        got = run_mx(d, w.eps, keep=True)
        ref = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], w.eps)
        st = parity.compare_mx(got, ref, what=name)
    print(name, M, st)


def test_qknorm_workload(oracle_mod):
    w = synth.WORKLOADS["qknorm"]
    d = synth.make_inputs(w, M=301)
    g = _gpu(d)
    (qy, qq, qs), (ky, kq, ks) = rmsq.qknorm_quant_fp8(g["q_a"], g["kv_a"], g["gamma_q"], g["gamma_kv"],
                                                       eps=w.eps, keep_bf16=True)
    torch.cuda.synchronize()
    ref = oracle_mod.qknorm_quant_fp8(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], w.eps)
    parity.compare_fp8({"q": qq, "scale": qs, "y": qy}, ref["q"], what="q_a")
    parity.compare_fp8({"q": kq, "scale": ks, "y": ky}, ref["kv"], what="kv_a")


@pytest.mark.parametrize("name", ["decode", "prefill", "qknorm", "mxfp4"])
def test_full_size_workloads(oracle_mod, name):
    """Full-size workloads, every row compared, default launch configuration."""
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w)
    if w.kind == "qknorm":
        g = _gpu(d)
        (qq, qs), (kq, ks) = rmsq.qknorm_quant_fp8(g["q_a"], g["kv_a"], g["gamma_q"], g["gamma_kv"], eps=w.eps)
        torch.cuda.synchronize()
        ref = oracle_mod.qknorm_quant_fp8(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], w.eps)
        st = [parity.compare_fp8({"q": qq, "scale": qs}, ref["q"], what="q_a"),
              parity.compare_fp8({"q": kq, "scale": ks}, ref["kv"], what="kv_a")]
    elif w.kind == "fp8":
        got = run_fp8(d, w.eps, layout=w.scale_layout, keep=w.keep_bf16)
        st = parity.compare_fp8(got, ref_fp8(oracle_mod, d, w.eps, w.scale_layout), w.scale_layout, what=name)
    else:
        got = run_mx(d, w.eps)
        ref = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], w.eps)
        st = parity.compare_mx(got, ref, what=name)
    print(name, st)


# ------------------------------------------------------ hand-worked rows

def _golden_rows():
    p = os.path.join(os.path.dirname(__file__), "golden", "handworked_rows.json")
    return json.load(open(p))["rows"]


def _vec(spec, H):
    v = np.full(H, spec["fill"], dtype=np.float64)
    for i, val in spec["set"]:
        v[i] = val
    return torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r["name"])
def test_handworked_rows_on_gpu(row):
    H = row["H"]
    x = _vec(row["x"], H)[None, :].to(DEV)
    res = None if row["residual"] is None else _vec(row["residual"], H)[None, :].to(DEV)
    gamma = _vec(row["gamma"], H).to(DEV)
    exp = row["expect"]
    if row["kind"] == "fp8":
        (y, q, s), _ = rmsq.add_rmsnorm_quant_fp8(x, gamma, res, eps=row["eps"], keep_bf16=True)
        torch.cuda.synchronize()
        want_q = np.full(H, exp["q"]["fill"], dtype=np.uint8)
        for i, c in exp["q"]["set"]:
            want_q[i] = c
        np.testing.assert_array_equal(parity.u8(q)[0], want_q)
        if "y" in exp:
            np.testing.assert_array_equal(y[0].float().cpu().numpy(), _vec(exp["y"], H).float().numpy())
    else:
        (y, q, s), _ = rmsq.add_rmsnorm_quant_mxfp4(x, gamma, res, eps=row["eps"], keep_bf16=True)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(parity.u8(s)[0], np.array(exp["mx_scale"], dtype=np.uint8))
        codes = np.full(H, exp["codes"]["fill"], dtype=np.uint8)
        for i, c in exp["codes"]["set"]:
            codes[i] = c
        np.testing.assert_array_equal(parity.u8(q)[0], codes[0::2] | (codes[1::2] << 4))


# -------------------------------------------------------------- edge cases

@pytest.mark.parametrize("H", [128, 256, 384, 512, 640, 1024, 1536, 2048, 3072, 4096, 5120, 7168, 8192, 16384])
def test_shapes_fp8(oracle_mod, H):
    M = 19                                          # ragged against every rows-per-block
    d = {"x": synth.random_bf16(10 + H, (M, H)), "residual": synth.random_bf16(20 + H, (M, H), var=4.0,
                                                                               tensor="residual"),
         "gamma": synth.gaussian_bf16(30 + H, "gamma", (H,), mean=1.0, var=0.1)}
    got = run_fp8(d, 1e-6, keep=True)
    parity.compare_fp8(got, ref_fp8(oracle_mod, d, 1e-6), what=f"H={H}")


@pytest.mark.parametrize("H", [32, 64, 96, 128, 160, 256, 512, 1024, 1536, 2048, 4096, 5120, 7168, 8192])
def test_shapes_mxfp4(oracle_mod, H):
    M = 23
    d = {"x": synth.student_t3_bf16(40 + H, "x", (M, H)),
         "residual": synth.random_bf16(50 + H, (M, H), tensor="residual"),
         "gamma": synth.gaussian_bf16(60 + H, "gamma", (H,), mean=1.0, var=0.1)}
    got = run_mx(d, 1e-6, keep=True)
    ref = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], 1e-6)
    parity.compare_mx(got, ref, what=f"H={H}")


@pytest.mark.parametrize("vpt", [1, 2, 4, 7])
def test_team_shapes_agree(oracle_mod, vpt):
    """Every vectors-per-thread choice for H=7168 meets the bar; outside
    boundary rows they are bit-identical to the oracle and so to each other."""
    w = synth.WORKLOADS["prefill"]
    d = synth.make_inputs(w, M=64)
    if 7168 // 8 // vpt > 512:
        pytest.skip("team larger than a block")
    got = run_fp8(d, w.eps, keep=True, opts=rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, vpt=vpt))
    parity.compare_fp8(got, ref_fp8(oracle_mod, d, w.eps), what=f"vpt={vpt}")


@pytest.mark.parametrize("rpb", [1, 2])
def test_rows_per_block(oracle_mod, rpb):
    w = synth.WORKLOADS["prefill"]
    d = synth.make_inputs(w, M=41)
    got = run_fp8(d, w.eps, opts=rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, rows_per_block=rpb))
    parity.compare_fp8(got, ref_fp8(oracle_mod, d, w.eps), what=f"rpb={rpb}")


def test_no_residual_and_column_major(oracle_mod):
    w = synth.WORKLOADS["decode"]
    d = synth.make_inputs(w, M=33)
    got = run_fp8(d, w.eps, layout="col", residual=False, keep=True)
    assert got["residual_out"] is None
    parity.compare_fp8(got, ref_fp8(oracle_mod, d, w.eps, layout="col", residual=False), "col", what="nores")


def test_single_row_and_in_place_residual(oracle_mod):
    w = synth.WORKLOADS["decode"]
    d = synth.make_inputs(w, M=1)
    g = _gpu(d)
    res = g["residual"].clone()
    (q, s), r = rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], res, eps=w.eps, out_residual=res)
    torch.cuda.synchronize()
    assert r.data_ptr() == res.data_ptr()
    parity.compare_fp8({"q": q, "scale": s, "residual_out": res}, ref_fp8(oracle_mod, d, w.eps), what="inplace")


def test_strided_rows(oracle_mod):
    """kv_a as a column slice of a wider projection output (leading dim > H)."""
    wide = synth.random_bf16(77, (40, 576 + 64))
    d = {"x": wide[:, :512], "gamma": synth.gaussian_bf16(78, "gamma", (512,), mean=1.0, var=0.1)}
    g = {"x": wide.to(DEV)[:, :512], "gamma": d["gamma"].to(DEV)}
    (q, s), _ = rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], None, eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle_mod.add_rmsnorm_quant_fp8(parity.u16(d["x"].contiguous()), None, d["gamma"], 1e-6)
    parity.compare_fp8({"q": q, "scale": s}, ref, what="strided")


def test_zero_and_extreme_rows(oracle_mod):
    """All-zero rows; huge and tiny magnitudes (the wide-range fp64 path);
    bf16 subnormals (no flush to zero anywhere)."""
    H = 1024
    rng = np.random.default_rng(0)
    base = rng.standard_normal((6, H)).astype(np.float32)
    rows = np.stack([np.zeros(H, np.float32), base[1] * np.float32(1e30), base[2] * np.float32(1e-30),
                     base[3] * np.float32(2.0 ** -130), base[4] * np.float32(3e38 / 8), base[5]])
    assert np.all(np.isfinite(rows))
    x = torch.from_numpy(rows).to(torch.bfloat16)
    gamma = synth.gaussian_bf16(5, "gamma", (H,), mean=1.0, var=0.1)
    for eps in (1e-6, 0.0):
        # with eps = 0 a zero row has no finite inv_rms, and a subnormal row's
        # inv_rms overflows fp32 (inf/inf codes are NaN): keep those to eps > 0
        xx = x if eps > 0 else x[[1, 2, 4, 5]]
        got = run_fp8({"x": xx, "gamma": gamma}, eps, residual=False, keep=True)
        ref = oracle_mod.add_rmsnorm_quant_fp8(xx, None, gamma, eps)
        parity.compare_fp8(got, ref, what=f"extreme eps={eps}")
        gm = run_mx({"x": xx, "gamma": gamma}, eps, residual=False, keep=True)
        parity.compare_mx(gm, oracle_mod.add_rmsnorm_quant_mxfp4(xx, None, gamma, eps), what=f"extreme mx eps={eps}")


def test_add_edge_pairs(oracle_mod):
    """Residual pairs at bf16 ties, wide exponent gaps, cancellation, subnormals."""
    H = 2048
    rng = np.random.default_rng(1)
    a = rng.standard_normal((4, H)).astype(np.float32)
    b = (rng.standard_normal((4, H)) * np.exp2(rng.integers(-40, 40, (4, H)))).astype(np.float32)
    b[0] = -a[0]
    b[1] = a[1] * np.float32(2.0 ** -8)
    a[2, ::2] = np.float32(2.0 ** -128)
    b[2, ::2] = np.float32(2.0 ** -131)
    x = torch.from_numpy(a).to(torch.bfloat16)
    res = torch.from_numpy(b).to(torch.bfloat16)
    gamma = torch.ones(H, dtype=torch.bfloat16)
    got = run_fp8({"x": x, "residual": res, "gamma": gamma}, 1e-6)
    ref = oracle_mod.add_rmsnorm_quant_fp8(x, res, gamma, 1e-6)
    np.testing.assert_array_equal(parity.u16(got["residual_out"]), ref["residual_out"])


def test_guard_bands_untouched(oracle_mod):
    """Outputs carved from larger buffers: bytes around them keep their canary."""
    w = synth.WORKLOADS["prefill"]
    M, H = 29, 7168
    d = _gpu(synth.make_inputs(w, M=M))
    pad = 4096
    qbuf = torch.full((M * H + 2 * pad,), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full((M * 56 + 2 * pad,), -7.0, dtype=torch.float32, device=DEV)
    rbuf = torch.full((M * H + 2 * pad,), 3.0, dtype=torch.bfloat16, device=DEV)
    ybuf = torch.full((M * H + 2 * pad,), 5.0, dtype=torch.bfloat16, device=DEV)
    st = rmsq.lib().rmsq_add_rmsnorm_quant_group_fp8(
        d["x"].data_ptr(), H, d["residual"].data_ptr(), H, d["gamma"].data_ptr(), 1e-6, M, H, 128,
        qbuf.data_ptr() + pad, sbuf.data_ptr() + pad * 4, 0, rbuf.data_ptr() + pad * 2,
        ybuf.data_ptr() + pad * 2, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    for buf, val, n in ((qbuf, 0xA5, M * H), (sbuf, -7.0, M * 56), (rbuf, 3.0, M * H), (ybuf, 5.0, M * H)):
        assert torch.all(buf[:pad] == val) and torch.all(buf[pad + n:] == val)


def test_misaligned_tensor_is_rejected():
    x = torch.zeros(4 * 256 + 1, dtype=torch.bfloat16, device=DEV)[1:].view(4, 256)
    gamma = torch.ones(256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rmsq.RmsqError, match="MISALIGNED"):
        rmsq.add_rmsnorm_quant_fp8(x, gamma)


# --------------------------------------------------------------- encoders

def _probe(values):
    base = np.concatenate([values, (values[:-1] + values[1:]) / 2]).astype(np.float32)
    near = [base]
    up, dn = base, base
    for _ in range(3):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(0))
        near += [up, dn]
    rng = np.random.default_rng(42)
    rand = rng.integers(0, 0x7F800000, 4_000_000, dtype=np.uint32).view(np.float32)
    mags = np.exp2(rng.uniform(-20, 12, 2_000_000)).astype(np.float32)
    special = np.array([0.0, 1e-45, 1e-40, 1.1754942e-38, 1e30, 3.4e38, np.inf], dtype=np.float32)
    v = np.concatenate(near + [rand, mags, special])
    return np.concatenate([v, -v])


def test_device_e4m3_encoder_matches_oracle(oracle_mod):
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    v = _probe(table[:0x7F].astype(np.float64))
    got = rmsq.encode_e4m3(torch.from_numpy(v).to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, oracle_mod.e4m3_encode(v))
    nan = rmsq.encode_e4m3(torch.tensor([float("nan")], device=DEV)).cpu().numpy()
    assert (nan[0] & 0x7F) == 0x7F


def test_device_e2m1_encoder_matches_oracle(oracle_mod):
    v = _probe(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]))
    got = rmsq.encode_e2m1(torch.from_numpy(v).to(DEV)).cpu().numpy()
    np.testing.assert_array_equal(got, oracle_mod.e2m1_encode(v))


# ------------------------------------------------- persistent bulk-copy kernel

PERSIST = rmsq.KERNEL_PERSISTENT


@pytest.mark.parametrize("name,M,grid", [("prefill", 1000, 0), ("prefill", 333, 7), ("decode", None, 0),
                                         ("mxfp4", 517, 0), ("prefill", 5, 0)])
def test_persistent_kernel_matches_oracle_and_rows_kernel(oracle_mod, name, M, grid):
    """Ragged row counts against the grid; grid 7 makes every block loop many times."""
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w, M=M)
    for vpt in (7, 4):
        po = rmsq.LaunchOpts(kernel=PERSIST, vpt=vpt, grid=grid)
        ro = rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, vpt=vpt)
        if w.kind == "fp8":
            a = run_fp8(d, w.eps, layout=w.scale_layout, keep=True, opts=po)
            b = run_fp8(d, w.eps, layout=w.scale_layout, keep=True, opts=ro)
            parity.compare_fp8(a, ref_fp8(oracle_mod, d, w.eps, w.scale_layout), w.scale_layout,
                               what=f"persistent {name} vpt={vpt}")
        else:
            a = run_mx(d, w.eps, keep=True, opts=po)
            b = run_mx(d, w.eps, keep=True, opts=ro)
            parity.compare_mx(a, oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], w.eps),
                              what=f"persistent {name} vpt={vpt}")
        for k in ("q", "scale", "y", "residual_out"):
            assert torch.equal(a[k].view(torch.uint8) if a[k].dtype == torch.float8_e4m3fn else a[k],
                               b[k].view(torch.uint8) if b[k].dtype == torch.float8_e4m3fn else b[k]), k
    assert rmsq.sync_status() == 0


def test_persistent_kernel_without_residual(oracle_mod):
    w = synth.WORKLOADS["prefill"]
    d = synth.make_inputs(w, M=200)
    got = run_fp8(d, w.eps, residual=False, keep=True, opts=rmsq.LaunchOpts(kernel=PERSIST, grid=16))
    parity.compare_fp8(got, ref_fp8(oracle_mod, d, w.eps, residual=False), what="persistent no residual")


def test_persistent_wait_times_out_cleanly(oracle_mod):
    """A row whose copy is never issued: its block's bounded wait gives up
    after 1 ms, the status reads RMSQ_ERR_TIMEOUT, the other blocks' rows are
    intact and the context stays usable."""
    w = synth.WORKLOADS["prefill"]
    M = 64
    d = synth.make_inputs(w, M=M)
    opts = rmsq.LaunchOpts(kernel=PERSIST, grid=8, debug_skip_row=10, wait_limit_ns=1_000_000)
    got = run_fp8(d, w.eps, opts=opts)
    assert rmsq.sync_status() == 5                     # RMSQ_ERR_TIMEOUT
    assert rmsq.sync_status() == 0                     # the word was cleared
    ref = ref_fp8(oracle_mod, d, w.eps)
    done = np.array([r % 8 != 10 % 8 for r in range(M)])   # block 2 stopped at row 10
    done |= np.array([r < 10 for r in range(M)])
    np.testing.assert_array_equal(parity.u8(got["q"])[done], ref["q"][done])
    # the context is still healthy: a normal call afterwards is exact
    again = run_fp8(d, w.eps)
    parity.compare_fp8(again, ref, what="after timeout")
    assert rmsq.sync_status() == 0


def test_group_division_is_exact_over_the_whole_domain():
    """The FP8 quantiser's per-group reciprocal + FMA-correction division gives
    the same E4M3 code as IEEE division for every (amax, y) pair it can see."""
    c = rmsq.check_group_division()
    assert c["pairs"] == sum(2 * (a + 1) for a in range(1, 0x7F80)), c
    assert c["code_mismatches"] == 0, c
    assert c["scale_mismatches"] == 0, c
    print(c)


@pytest.mark.parametrize("M,Hq,Hkv", [(301, 1536, 512), (8192, 1536, 512), (37, 96, 32), (19, 640, 160)])
def test_qknorm_mxfp4(oracle_mod, M, Hq, Hkv):
    """The MXFP4 latent pair in one launch: the compiled-in shape (1536/512) at a
    ragged and the full row count, and generic shapes."""
    d = {"q_a": synth.random_bf16(90 + Hq, (M, Hq)),
         "kv_a": synth.random_bf16(91 + Hkv, (M, Hkv), var=2.0, tensor="kv_a"),
         "gamma_q": synth.gaussian_bf16(92, "gamma_q", (Hq,), mean=1.0, var=0.1),
         "gamma_kv": synth.gaussian_bf16(93, "gamma_kv", (Hkv,), mean=1.0, var=0.1)}
    g = _gpu(d)
    (qy, qq, qs), (ky, kq, ks) = rmsq.qknorm_quant_mxfp4(g["q_a"], g["kv_a"], g["gamma_q"], g["gamma_kv"],
                                                         eps=1e-6, keep_bf16=True)
    torch.cuda.synchronize()
    ref = oracle_mod.qknorm_quant_mxfp4(d["q_a"], d["kv_a"], d["gamma_q"], d["gamma_kv"], 1e-6)
    parity.compare_mx({"q": qq, "scale": qs, "y": qy}, ref["q"], what="mx q_a")
    parity.compare_mx({"q": kq, "scale": ks, "y": ky}, ref["kv"], what="mx kv_a")


# ------------------------------------------------------- GEMM-ready scale layouts

@pytest.mark.parametrize("M", [1, 37, 64, 300])
def test_fp8_padded_column_major_scales(oracle_mod, M):
    w = synth.WORKLOADS["decode"]
    d = synth.make_inputs(w, M=M)
    g = _gpu(d)
    Mp = (M + 3) // 4 * 4
    scale = torch.full((56, Mp), -3.0, dtype=torch.float32, device=DEV)     # canary in the padding
    q = torch.empty((M, 7168), dtype=torch.uint8, device=DEV)
    ro = torch.empty((M, 7168), dtype=torch.bfloat16, device=DEV)
    rmsq.add_rmsnorm_quant_fp8_into(g["x"], g["gamma"], g["residual"], q, scale, ro, None, eps=w.eps,
                                    scale_layout="col_pad4")
    torch.cuda.synchronize()
    ref = oracle_mod.add_rmsnorm_quant_fp8(d["x"], d["residual"], d["gamma"], w.eps, layout="col_pad4")
    parity.compare_fp8({"q": q, "scale": scale[:, :M], "residual_out": ro},
                       {**ref, "scale": ref["scale"][:, :M]}, "col", what=f"col_pad4 M={M}")
    assert torch.all(scale[:, M:] == -3.0)


@pytest.mark.parametrize("M,H", [(300, 7168), (128, 7168), (5, 96), (8192, 7168)])
def test_mxfp4_mma_tile_scales(oracle_mod, M, H):
    d = {"x": synth.student_t3_bf16(70 + M, "x", (M, H)),
         "residual": synth.random_bf16(71 + M, (M, H), tensor="residual"),
         "gamma": synth.gaussian_bf16(72, "gamma", (H,), mean=1.0, var=0.1)}
    g = _gpu(d)
    nbytes = rmsq.mma_scale_bytes(M, H)
    canary = torch.full((nbytes,), 0xEE, dtype=torch.uint8, device=DEV)
    (q, s), ro = rmsq.add_rmsnorm_quant_mxfp4_mma_scales(g["x"], g["gamma"], g["residual"], eps=1e-6,
                                                          scale_out=canary)
    torch.cuda.synchronize()
    ref = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], 1e-6)
    want = oracle_mod.mx_scale_tiles(ref["scale"], fill=0xEE)
    boundary = ref["margin"] < parity.BOUNDARY
    if not boundary.any():
        np.testing.assert_array_equal(parity.u8(s), want)
    parity.compare_mx({"q": q, "scale": torch.from_numpy(ref["scale"]), "residual_out": ro}, ref,
                      what=f"mx tiles M={M}")


# ---------------------------------------------------------------- maximum sizes

def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, n)]))


def test_chunked_prefill_maximum_rows(oracle_mod):
    """131072 tokens (the largest chunked-prefill size on the pages) x 7168:
    inputs drawn on the device (torch, fixed seed), 64 sampled rows checked
    against the oracle, in the default launch configuration."""
    M, H = 131072, 7168
    gen = torch.Generator(device=DEV).manual_seed(1234)
    x = torch.randn((M, H), generator=gen, device=DEV).to(torch.bfloat16)
    res = (torch.randn((M, H), generator=gen, device=DEV) * 2).to(torch.bfloat16)
    gamma = (1 + 0.3 * torch.randn((H,), generator=gen, device=DEV)).to(torch.bfloat16)
    (y, q, s), ro = rmsq.add_rmsnorm_quant_fp8(x, gamma, res, eps=1e-6, keep_bf16=True)
    torch.cuda.synchronize()
    rows = torch.from_numpy(_sample_rows(M, 62, 5)).to(DEV)
    ref = oracle_mod.add_rmsnorm_quant_fp8(x[rows].cpu(), res[rows].cpu(), gamma.cpu(), 1e-6)
    got = {"q": q[rows], "scale": s[rows], "y": y[rows], "residual_out": ro[rows]}
    parity.compare_fp8(got, ref, what="M=131072")
    del x, res, y, q, s, ro
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["fp8", "mxfp4"])
def test_widest_row(oracle_mod, kind):
    """H = 32768, the widest row the kernels take (8 vectors x 512 threads)."""
    M, H = 9, 32768
    d = {"x": synth.random_bf16(3, (M, H)), "residual": synth.random_bf16(4, (M, H), tensor="residual"),
         "gamma": synth.gaussian_bf16(5, "gamma", (H,), mean=1.0, var=0.1)}
    if kind == "fp8":
        parity.compare_fp8(run_fp8(d, 1e-6, keep=True), ref_fp8(oracle_mod, d, 1e-6), what="H=32768")
    else:
        parity.compare_mx(run_mx(d, 1e-6, keep=True),
                          oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], 1e-6),
                          what="mx H=32768")


def test_empty_batch_is_a_no_op():
    x = torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV)
    g = torch.ones(7168, dtype=torch.bfloat16, device=DEV)
    (q, s), r = rmsq.add_rmsnorm_quant_fp8(x, g, x.clone())
    (mq, ms), _ = rmsq.add_rmsnorm_quant_mxfp4(x, g)
    torch.cuda.synchronize()
    assert q.shape == (0, 7168) and s.shape == (0, 56) and mq.shape == (0, 3584)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_device_encoder_every_fp32_pattern(oracle_mod, fmt):
    """All 2^32 fp32 bit patterns through the kernels' hardware conversion
    (cvt.rn.satfinite) against the oracle's encoder, in 64 chunks, the oracle
    threaded over the host cores. Non-NaN inputs must agree exactly; NaN
    inputs (outside every workload) must give the E4M3 NaN code, and for
    E2M1, which has no NaN, only their count of disagreements is reported."""
    from concurrent.futures import ThreadPoolExecutor
    enc_gpu = rmsq.encode_e4m3 if fmt == "e4m3" else rmsq.encode_e2m1
    enc_cpu = oracle_mod.e4m3_encode if fmt == "e4m3" else oracle_mod.e2m1_encode
    chunk = 1 << 26
    bad, nan_diff, checked = 0, 0, 0
    with ThreadPoolExecutor(max_workers=16) as ex:
        for c in range(1 << 6):
            v = np.arange(c * chunk, (c + 1) * chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
            got = enc_gpu(torch.from_numpy(v).to(DEV)).cpu().numpy()
            want = np.concatenate(list(ex.map(enc_cpu, np.array_split(v, 16))))
            nan = np.isnan(v)
            bad += int(((got != want) & ~nan).sum())
            if fmt == "e4m3":
                assert np.all((got[nan] & 0x7F) == 0x7F), "a NaN input did not give the NaN code"
            else:
                nan_diff += int(((got != want) & nan).sum())
            checked += v.size
    assert checked == 1 << 32
    assert bad == 0, f"{bad} fp32 patterns encode differently"
    print(fmt, "patterns checked:", checked, "NaN inputs encoded differently (E2M1 only):", nan_diff)


def test_debug_build_bounds_check_fires():
    """Positive control of the debug build's store checks (skipped in release
    builds): a deliberately failing check is reported as RMSQ_ERR_BOUNDS."""
    if os.environ.get("RMSQ_DEBUG") != "1":
        pytest.skip("runs against the RMSQ_DEBUG library (tests/test_zz_debug_build_gpu.py)")
    assert rmsq.lib().rmsq_debug_bounds_selftest(torch.cuda.current_stream().cuda_stream) == 0
    assert rmsq.sync_status() == 6                     # RMSQ_ERR_BOUNDS
    assert rmsq.sync_status() == 0


# ------------------------------------------ column-major scales at prefill size

@pytest.mark.parametrize("layout", ["col", "col_pad4"])
def test_full_size_column_major_scales(oracle_mod, layout):
    """The decode config's column-major scale layout at the prefill size
    (M = 16384, H = 7168, keep_bf16), every row compared, default launch."""
    w = synth.WORKLOADS["prefill"]
    d = synth.make_inputs(w)
    got = run_fp8(d, w.eps, layout=layout, keep=True)
    ref = ref_fp8(oracle_mod, d, w.eps, layout=layout)
    st = parity.compare_fp8(got, ref, "col", what=f"prefill {layout}")
    print(layout, st)


# ------------------------------------------------- rows outside fp32's range

@pytest.mark.parametrize("H", [8192, 32768])
def test_wide_range_rows_fp64_path(oracle_mod, H):
    """Rows whose sum of squares leaves the double-float range (elements near
    2^60 and near 2^-60, so sums near 2^133 and 2^-107), which take the fp64
    path: 384 rows per width, eps = 0 so that the sum alone sets inv_rms, and
    every output bit-exact against the oracle outside boundary rows."""
    M = 384
    base = synth.normals(40 + H, "x", M * H).reshape(M, H)
    scale = np.where(np.arange(M)[:, None] % 2 == 0, 2.0 ** 60, 2.0 ** -60)
    x = synth.to_bf16(base * scale, (M, H))
    assert torch.isfinite(x.float()).all()
    d = {"x": x, "gamma": synth.gaussian_bf16(41, "gamma", (H,), mean=1.0, var=0.1)}
    ref = ref_fp8(oracle_mod, d, 0.0, residual=False)
    st = parity.compare_fp8(run_fp8(d, 0.0, residual=False, keep=True), ref, what=f"wide range H={H}")
    assert st["codes_differing"] == 0 or st["boundary_rows"] > 0
    mref = oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], None, d["gamma"], 0.0)
    parity.compare_mx(run_mx(d, 0.0, residual=False, keep=True), mref, what=f"mx wide range H={H}")
    print(H, st)


# ------------------------------------------- latency form of the row kernel

@pytest.mark.parametrize("name,M,split", [("decode", None, 0), ("decode", None, 1), ("decode", None, 2),
                                          ("decode", 1, 4), ("decode", 37, 4), ("decode", 152, 0),
                                          ("prefill", 2000, 1), ("prefill", 300, 2), ("mxfp4", 64, 2),
                                          ("mxfp4", 5, 4)])
def test_latency_form_is_bit_identical(oracle_mod, name, M, split):
    """The latency form (gamma loaded with the row, every warp finalising
    inv_rms; with split > 1 each row's outputs shared by that many blocks,
    each reducing the whole row) against the throughput form: every output
    bit-identical, and both against the oracle."""
    w = synth.WORKLOADS[name]
    d = synth.make_inputs(w, M=M)
    lat = rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, form=rmsq.FORM_LATENCY, split=split)
    thr = rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, form=rmsq.FORM_THROUGHPUT)
    if w.kind == "fp8":
        a = run_fp8(d, w.eps, layout=w.scale_layout, keep=True, opts=lat)
        b = run_fp8(d, w.eps, layout=w.scale_layout, keep=True, opts=thr)
        parity.compare_fp8(a, ref_fp8(oracle_mod, d, w.eps, w.scale_layout), w.scale_layout, what="latency form")
    else:
        a = run_mx(d, w.eps, keep=True, opts=lat)
        b = run_mx(d, w.eps, keep=True, opts=thr)
        parity.compare_mx(a, oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], w.eps),
                          what="mx latency form")
    for k in ("q", "scale", "residual_out", "y"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k



@pytest.mark.parametrize("H", [256, 512, 1536, 2048, 4096, 5120, 8192])
@pytest.mark.parametrize("M", [1, 4, 37, 64, 150, 300])
def test_latency_form_across_compiled_shapes(oracle_mod, H, M):
    """At every compiled team shape the automatic choice at decode sizes --
    the latency form, its rows spread over as many blocks as keep one block
    per SM, rows split between blocks where SMs remain -- gives outputs
    bit-identical to the throughput form, FP8 and MXFP4, and meets the bar
    against the oracle."""
    d = {"x": synth.random_bf16(110 + H, (M, H)),
         "residual": synth.random_bf16(120 + H, (M, H), var=4.0, tensor="residual"),
         "gamma": synth.gaussian_bf16(130 + H, "gamma", (H,), mean=1.0, var=0.1)}
    thr = rmsq.LaunchOpts(kernel=rmsq.KERNEL_ROWS, form=rmsq.FORM_THROUGHPUT)
    a = run_fp8(d, 1e-6, keep=True)
    b = run_fp8(d, 1e-6, keep=True, opts=thr)
    parity.compare_fp8(a, ref_fp8(oracle_mod, d, 1e-6), what=f"latency form H={H} M={M}")
    for k in ("q", "scale", "residual_out", "y"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k
    a = run_mx(d, 1e-6, keep=True)
    b = run_mx(d, 1e-6, keep=True, opts=thr)
    parity.compare_mx(a, oracle_mod.add_rmsnorm_quant_mxfp4(d["x"], d["residual"], d["gamma"], 1e-6),
                      what=f"mx latency form H={H} M={M}")
    for k in ("q", "scale", "residual_out", "y"):
        assert torch.equal(a[k].view(torch.uint8), b[k].view(torch.uint8)), k

@pytest.mark.parametrize("kind,M", [("fp8", 64), ("fp8", 37), ("fp8", 8), ("mx", 4), ("mx", 64)])
def test_in_place_residual_is_not_split(kind, M):
    """Split rows read the whole residual row in every block of the row and
    write back one part each, which would race with an in-place residual
    update: such calls take one block per row (auto) and refuse an explicit
    split. Repeated in-place calls equal the out-of-place call (split rows)
    bit for bit."""
    H = 7168
    x = synth.random_bf16(300 + M, (M, H)).to(DEV)
    res = synth.random_bf16(301 + M, (M, H), var=4.0, tensor="residual").to(DEV)
    gamma = synth.gaussian_bf16(302, "gamma", (H,), mean=1.0, var=0.1).to(DEV)
    call = rmsq.add_rmsnorm_quant_fp8 if kind == "fp8" else rmsq.add_rmsnorm_quant_mxfp4
    (y0, q0, s0), r0 = call(x, gamma, res, keep_bf16=True)     # out of place: split rows at these sizes
    torch.cuda.synchronize()
    copies = [res.clone() for _ in range(20)]
    outs = [call(x, gamma, c, keep_bf16=True, out_residual=c) for c in copies]
    torch.cuda.synchronize()
    for i, ((y, q, sc), r) in enumerate(outs):
        assert r.data_ptr() == copies[i].data_ptr()
        for a, b in ((y, y0), (q, q0), (sc, s0), (r, r0)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"call {i}"
    c = res.clone()
    with pytest.raises(rmsq.RmsqError, match="in-place"):
        call(x, gamma, c, out_residual=c, opts=rmsq.LaunchOpts(form=rmsq.FORM_LATENCY, split=2))
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("mx", [False, True])
@pytest.mark.parametrize("M", [1, 5, 64, 76, 101, 102, 128, 300, 700, 808, 809, 1300])
def test_qknorm_pair_latency_form(oracle_mod, M, mx):
    """The MLA pair (q_a 1536, kv_a 512) at decode sizes takes the pair's
    latency form (gamma loaded with each row) in the smallest block that keeps
    the launch within one block per SM: 32 threads (one q_a row, two kv_a
    rows) up to 101 tokens, then 64, 128 and 256 threads up to 808 tokens;
    809 and 1300 tokens take the throughput form. Each against the oracle,
    every row."""
    Hq, Hkv = 1536, 512
    q_a = synth.random_bf16(500 + M, (M, Hq), tensor="q_a")
    kv_a = synth.random_bf16(501 + M, (M, Hkv), var=2.0, tensor="kv_a")
    gq = synth.gaussian_bf16(502, "gamma_q", (Hq,), mean=1.0, var=0.1)
    gk = synth.gaussian_bf16(503, "gamma_kv", (Hkv,), mean=1.0, var=0.1)
    fn = rmsq.qknorm_quant_mxfp4 if mx else rmsq.qknorm_quant_fp8
    outq, outk = fn(q_a.to(DEV), kv_a.to(DEV), gq.to(DEV), gk.to(DEV), keep_bf16=True)
    torch.cuda.synchronize()
    for out, x, g in ((outq, q_a, gq), (outk, kv_a, gk)):
        got = {"q": out[-2], "scale": out[-1], "y": out[0]}
        if mx:
            parity.compare_mx(got, oracle_mod.add_rmsnorm_quant_mxfp4(x, None, g), what=f"pair M={M}")
        else:
            parity.compare_fp8(got, oracle_mod.add_rmsnorm_quant_fp8(x, None, g), "row", what=f"pair M={M}")
    assert rmsq.sync_status() == 0


def test_unknown_form_and_bad_split_are_refused():
    w = synth.WORKLOADS["decode"]
    g = _gpu(synth.make_inputs(w, M=4))
    with pytest.raises(rmsq.RmsqError, match="form"):
        rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], g["residual"], opts=rmsq.LaunchOpts(form=7))
    with pytest.raises(rmsq.RmsqError, match="split"):
        rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], g["residual"], opts=rmsq.LaunchOpts(split=3))
    with pytest.raises(rmsq.RmsqError, match="split"):     # the throughput form does not split rows
        rmsq.add_rmsnorm_quant_fp8(g["x"], g["gamma"], g["residual"],
                                   opts=rmsq.LaunchOpts(form=rmsq.FORM_THROUGHPUT, split=2))


# ------------------------------------- calls that read the previous call's outputs

@pytest.mark.parametrize("M,kind,in_place", [(4, "fp8", True), (64, "fp8", False), (64, "fp8", True),
                                              (16384, "fp8", True), (64, "mx", False), (8192, "mx", True)])
def test_dependent_launches_with_no_kernel_between(M, kind, in_place):
    """Eight calls with nothing between them on the stream, each reading the
    previous call's y as its x and its residual output as its residual (in
    place, or alternating between two buffers), every output in a buffer of
    its own: each call is launched as a programmatic dependent of the one
    before and must still read what that one wrote. Back to back and from a
    CUDA graph, against the same chain synchronised after every call."""
    H, n = 7168, 8
    x0 = synth.random_bf16(70 + M, (M, H)).to(DEV)
    res0 = synth.random_bf16(71 + M, (M, H), var=4.0, tensor="residual").to(DEV)
    gamma = synth.gaussian_bf16(72, "gamma", (H,), mean=1.0, var=0.1).to(DEV)
    mx = kind == "mx"
    ys = [torch.empty((M, H), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    qs = [torch.empty((M, H // 2 if mx else H), dtype=torch.uint8, device=DEV) for _ in range(n)]
    ss = [torch.empty((M, H // 32), dtype=torch.uint8, device=DEV) if mx else
          torch.empty((M, H // 128), dtype=torch.float32, device=DEV) for _ in range(n)]
    res = [res0.clone(), torch.empty_like(res0)]

    def chain(sync):
        res[0].copy_(res0)
        torch.cuda.synchronize()
        x = x0
        for i in range(n):
            r_in = res[0] if in_place else res[i % 2]
            r_out = res[0] if in_place else res[(i + 1) % 2]
            if mx:
                rmsq.add_rmsnorm_quant_mxfp4_into(x, gamma, r_in, qs[i], ss[i], r_out, ys[i])
            else:
                rmsq.add_rmsnorm_quant_fp8_into(x, gamma, r_in, qs[i], ss[i], r_out, ys[i])
            if sync:
                torch.cuda.synchronize()
            x = ys[i]

    chain(True)
    want = [t.clone() for t in ys + qs + ss + [res[0] if in_place else res[n % 2]]]
    for t in ys + qs + ss:
        t.zero_()
    chain(False)
    torch.cuda.synchronize()
    got = ys + qs + ss + [res[0] if in_place else res[n % 2]]
    for i, (a, b) in enumerate(zip(got, want)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"tensor {i}, back to back"
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            x = x0
            for i in range(n):
                r_in = res[0] if in_place else res[i % 2]
                r_out = res[0] if in_place else res[(i + 1) % 2]
                if mx:
                    rmsq.add_rmsnorm_quant_mxfp4_into(x, gamma, r_in, qs[i], ss[i], r_out, ys[i],
                                                      stream=side.cuda_stream)
                else:
                    rmsq.add_rmsnorm_quant_fp8_into(x, gamma, r_in, qs[i], ss[i], r_out, ys[i],
                                                    stream=side.cuda_stream)
                x = ys[i]
        res[0].copy_(res0)
        for t in ys + qs + ss:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
    torch.cuda.current_stream().wait_stream(side)
    for i, (a, b) in enumerate(zip(got, want)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"tensor {i}, graph replay"
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("M", [4, 64, 8192])
def test_pair_calls_with_no_kernel_between(M):
    """The MLA pair called four times with nothing between them, each call
    normalising the previous call's bf16 outputs: back to back must equal the
    chain synchronised after every call."""
    q_a = synth.random_bf16(81, (M, 1536), tensor="q_a").to(DEV)
    kv_a = synth.random_bf16(82, (M, 512), tensor="kv_a").to(DEV)
    gq = synth.gaussian_bf16(83, "gamma_q", (1536,), mean=1.0).to(DEV)
    gk = synth.gaussian_bf16(84, "gamma_kv", (512,), mean=1.0).to(DEV)
    n = 4
    outs = [[torch.empty((M, 1536), dtype=torch.uint8, device=DEV), torch.empty((M, 12), dtype=torch.float32, device=DEV),
             torch.empty((M, 512), dtype=torch.uint8, device=DEV), torch.empty((M, 4), dtype=torch.float32, device=DEV),
             torch.empty((M, 1536), dtype=torch.bfloat16, device=DEV), torch.empty((M, 512), dtype=torch.bfloat16, device=DEV)]
            for _ in range(n)]

    def chain(sync):
        a, b = q_a, kv_a
        for o in outs:
            rmsq.qknorm_quant_fp8_into(a, b, gq, gk, o[0], o[1], o[2], o[3], qy=o[4], ky=o[5])
            if sync:
                torch.cuda.synchronize()
            a, b = o[4], o[5]
        torch.cuda.synchronize()

    chain(True)
    want = [t.clone() for o in outs for t in o]
    for o in outs:
        for t in o:
            t.zero_()
    chain(False)
    got = [t for o in outs for t in o]
    for i, (u, v) in enumerate(zip(got, want)):
        assert torch.equal(u.view(torch.uint8), v.view(torch.uint8)), f"tensor {i}"
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("M,kind", [(64, "fp8"), (8192, "fp8"), (37, "mx"), (3000, "mx")])
def test_chained_calls_read_the_previous_outputs(M, kind):
    """A chain of six calls in which each reads what the previous one wrote
    -- the residual updated in place, the next x being the previous y --
    launched back to back without synchronisation must equal the same chain
    synchronised after every call."""
    H = 7168
    x0 = synth.random_bf16(90 + M, (M, H)).to(DEV)
    res0 = synth.random_bf16(91 + M, (M, H), var=4.0, tensor="residual").to(DEV)
    gamma = synth.gaussian_bf16(92, "gamma", (H,), mean=1.0, var=0.1).to(DEV)

    def chain(sync):
        x, res, outs = x0, res0.clone(), []
        for _ in range(6):
            if kind == "fp8":
                (y, q, s), _ = rmsq.add_rmsnorm_quant_fp8(x, gamma, res, keep_bf16=True, out_residual=res)
            else:
                (y, q, s), _ = rmsq.add_rmsnorm_quant_mxfp4(x, gamma, res, keep_bf16=True, out_residual=res)
            if sync:
                torch.cuda.synchronize()
            outs.append((y, q, s, res.clone()))
            x = y
        torch.cuda.synchronize()
        return outs

    want, got = chain(True), chain(False)
    for i, (a, b) in enumerate(zip(got, want)):
        for u, v in zip(a, b):
            assert torch.equal(u.view(torch.uint8), v.view(torch.uint8)), f"call {i}"
