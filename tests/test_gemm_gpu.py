"""Parity of the block-scaled MXFP4 consumer GEMM (both placements of the
activation quant) with the CPU oracle, through the C ABI.

The operands are seeded synthetic MXFP4 data; the comparison rule is
tests/parity.py's compare_gemm (a bound derived from fp32 accumulation and
the bf16 output rounding). The two placements -- quant fused into the norm,
quant in the GEMM's prologue -- must give bit-identical outputs."""

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


def operands(seed, M, N, K):
    """A (activation-like scale bytes 124..130) and B (weights) as MXFP4."""
    a_q, a_s = synth.mxfp4_weights(seed, M, K, scale_lo=124, scale_hi=131)
    b_q, b_s = synth.mxfp4_weights(seed + 1000, N, K)
    return a_q, a_s, b_q, b_s


def gpu_gemm(a_q, a_s, b_q, b_s, bn=0, ksplit=0):
    ga, gb = a_q.to(DEV), b_q.to(DEV)
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    opts = rmsq.GemmOpts(bn=bn, ksplit=ksplit) if (bn or ksplit) else None
    d = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=opts)
    torch.cuda.synchronize()
    return d


def test_scale_tiles_match_oracle(oracle_mod):
    for R, G, fill in [(300, 56, 0), (128, 8, 7), (5, 3, 255), (1, 224, 0)]:
        s = torch.randint(0, 256, (R, G), dtype=torch.uint8, generator=torch.Generator().manual_seed(R + G))
        got = rmsq.mx_scale_tiles(s.to(DEV), fill=fill).cpu().numpy()
        assert np.array_equal(got, oracle_mod.mx_scale_tiles(s.numpy(), fill=fill)), (R, G)


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("M,N,K", [(200, 328, 512), (128, 256, 256), (4, 520, 2048), (129, 64, 1536)])
def test_mxfp4_gemm_matches_oracle(oracle_mod, bn, M, N, K):
    a_q, a_s, b_q, b_s = operands(M * 7 + N, M, N, K)
    d = gpu_gemm(a_q, a_s, b_q, b_s, bn)
    ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
    st = parity.compare_gemm(d, ref, K, what=f"bn={bn} {M}x{N}x{K}")
    assert st["bit_equal_fraction"] > 0.95, st
    assert rmsq.sync_status() == 0
    print(bn, M, N, K, st)


@pytest.mark.parametrize("ksplit", [2, 3, 8])
@pytest.mark.parametrize("bn", [64, 256])
def test_split_k_matches_oracle(oracle_mod, bn, ksplit):
    """K split over a cluster of CTAs, partial sums added through distributed
    shared memory: same bound, and no output outside D."""
    M, N, K = 70, 328, 2560
    a_q, a_s, b_q, b_s = operands(17 + ksplit, M, N, K)
    d = gpu_gemm(a_q, a_s, b_q, b_s, bn, ksplit)
    ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
    st = parity.compare_gemm(d, ref, K, what=f"bn={bn} ksplit={ksplit}")
    assert st["bit_equal_fraction"] > 0.95, st
    again = gpu_gemm(a_q, a_s, b_q, b_s, bn, ksplit)
    assert torch.equal(d, again), "split-K result is not deterministic"
    assert rmsq.sync_status() == 0
    print(bn, ksplit, st)


@pytest.mark.parametrize("bn,ksplit", [(64, 4), (64, 2), (256, 8), (128, 3)])
@pytest.mark.parametrize("rows", [4, 33, 64])
def test_split_k_rows_independent_of_m(oracle_mod, bn, ksplit, rows):
    """Split K adds the cluster's partial sums in rank order whatever the
    tile's row count, so the rows a 4-, 33- or 64-token launch computes equal
    the same rows of a 200-token launch bit for bit, and match the oracle."""
    M, N, K = 200, 264, 2048
    a_q, a_s, b_q, b_s = operands(91, M, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    opts = rmsq.GemmOpts(bn=bn, ksplit=ksplit)
    full = rmsq.mxfp4_gemm(a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV)), gb, tb, opts=opts)
    few = rmsq.mxfp4_gemm(a_q[:rows].to(DEV), rmsq.mx_scale_tiles(a_s[:rows].to(DEV)), gb, tb, opts=opts)
    torch.cuda.synchronize()
    assert torch.equal(few, full[:rows])
    ref = oracle_mod.mxfp4_gemm(a_q[:rows].numpy(), a_s[:rows].numpy(), b_q.numpy(), b_s.numpy())
    parity.compare_gemm(few, ref, K, what=f"split K, {rows} rows, bn={bn} ksplit={ksplit}")
    assert rmsq.sync_status() == 0


def test_bounded_wait_split_k_decode(oracle_mod):
    """A stalled stage at decode size (8 tokens, K split over 2 CTAs, two
    4-span stages per CTA, the second never loaded): the stalled CTA stops,
    both still meet at the cluster barriers, the host reads
    RMSQ_ERR_TIMEOUT and the next launch matches the oracle."""
    M, N, K = 8, 256, 4096
    a_q, a_s, b_q, b_s = operands(93, M, N, K)
    ga, ta = a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV))
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=64, ksplit=2, wait_limit_ns=50_000_000,
                                                       debug_stall_stage=2))
    assert rmsq.sync_status() == 5                      # RMSQ_ERR_TIMEOUT
    assert rmsq.sync_status() == 0
    again = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=64, ksplit=2))
    torch.cuda.synchronize()
    ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
    parity.compare_gemm(again, ref, K, what="after a timed-out split-K launch")
    assert rmsq.sync_status() == 0


def test_tile_choices_agree_bitwise():
    """Tiles of 64, 128 and 256 B rows run the same MMAs in the same K order."""
    a_q, a_s, b_q, b_s = operands(5, 256, 512, 1024)
    outs = [gpu_gemm(a_q, a_s, b_q, b_s, bn, 1) for bn in (64, 128, 256)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("bn,M,N", [(64, 1100, 1032), (128, 2050, 1352), (256, 4100, 1160)])
def test_persistent_schedule(oracle_mod, bn, M, N):
    """More tiles than SMs: a persistent grid (each CTA walks several tiles,
    the stage ring and the accumulator carried from one tile into the next)
    gives the one-tile-per-CTA result bit for bit, and the oracle's on
    sampled rows, ragged last row and column tiles included."""
    K = 1024
    a_q, a_s, b_q, b_s = operands(300 + bn, M, N, K)
    ga, gb = a_q.to(DEV), b_q.to(DEV)
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    one = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn, ksplit=1, schedule=1))
    walk = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn, ksplit=1, schedule=2))
    auto = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn))
    torch.cuda.synchronize()
    tiles = -(-M // 128) * -(-N // bn)
    assert tiles > torch.cuda.get_device_properties(DEV).multi_processor_count
    assert torch.equal(one, walk) and torch.equal(one, auto)
    rows = np.unique(np.concatenate([np.arange(0, M, 97), [M - 1]]))
    ref = oracle_mod.mxfp4_gemm(a_q.numpy()[rows], a_s.numpy()[rows], b_q.numpy(), b_s.numpy())
    st = parity.compare_gemm(walk[torch.from_numpy(rows).to(DEV)], ref, K, what=f"persistent bn={bn}")
    assert rmsq.sync_status() == 0
    print(bn, tiles, st)


@pytest.mark.parametrize("bn", [256, 192])
@pytest.mark.parametrize("M,N,K", [(4100, 1160, 1024), (1100, 2112, 2048), (300, 264, 256), (129, 520, 512),
                                   (1, 256, 768), (600, 8, 1280), (8192, 2112, 512)])
def test_pair_schedule(oracle_mod, M, N, K, bn):
    """CTA pairs (256 x bn tiles, M = 256 MMAs over two SMs; bn 192 with two
    accumulators and a ring of scale-factor slots): bit for bit the
    one-tile-per-CTA result, and the oracle's on sampled rows -- ragged M and
    N, a pair whose odd CTA has no rows of A (M = 129, M = 1), one span of K,
    several tiles per pair (M = 8192)."""
    a_q, a_s, b_q, b_s = operands(400 + M % 97, M, N, K)
    ga, gb = a_q.to(DEV), b_q.to(DEV)
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    one = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=256, ksplit=1, schedule=1))
    pair = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn if bn != 256 else 0, schedule=3))
    again = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn, ksplit=1, schedule=3))
    torch.cuda.synchronize()
    assert torch.equal(one, pair) and torch.equal(pair, again)
    rows = np.unique(np.concatenate([np.arange(0, M, 61), [M - 1]]))
    ref = oracle_mod.mxfp4_gemm(a_q.numpy()[rows], a_s.numpy()[rows], b_q.numpy(), b_s.numpy())
    st = parity.compare_gemm(pair[torch.from_numpy(rows).to(DEV)], ref, K, what=f"pair M={M} N={N} K={K}")
    assert st["bit_equal_fraction"] > 0.95, st
    assert rmsq.sync_status() == 0
    print(M, N, K, st)


def test_pair_schedule_strided(oracle_mod):
    """CTA pairs with leading dimensions wider than a row for A, B and D."""
    M, N, K = 700, 520, 1536
    a_q, a_s, b_q, b_s = operands(75, M, N, K)
    pa = torch.zeros((M, K // 2 + 176), dtype=torch.uint8)
    pa[:, :K // 2] = a_q
    pb = torch.zeros((N, K // 2 + 48), dtype=torch.uint8)
    pb[:, :K // 2] = b_q
    ga, gb = pa.to(DEV)[:, :K // 2], pb.to(DEV)[:, :K // 2]
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    dbig = torch.zeros((M + 9, N + 40), dtype=torch.bfloat16, device=DEV)
    d = rmsq.mxfp4_gemm(ga, ta, gb, tb, out=dbig[:M, :N], opts=rmsq.GemmOpts(schedule=3))
    one = rmsq.mxfp4_gemm(a_q.to(DEV), ta, b_q.to(DEV), tb, opts=rmsq.GemmOpts(bn=256, ksplit=1, schedule=1))
    torch.cuda.synchronize()
    assert torch.equal(d, one)
    assert (dbig[:, N:] == 0).all() and (dbig[M:] == 0).all()   # nothing past D[:M, :N] is written
    rows = np.unique(np.concatenate([np.arange(0, M, 37), [M - 1]]))
    ref = oracle_mod.mxfp4_gemm(a_q.numpy()[rows], a_s.numpy()[rows], b_q.numpy(), b_s.numpy())
    parity.compare_gemm(d[torch.from_numpy(rows).to(DEV)], ref, K, what="pair, strided A, B, D")
    assert rmsq.sync_status() == 0


def test_pair_schedule_rejects():
    M, N, K = 256, 256, 512
    a_q, a_s, b_q, b_s = operands(33, M, N, K)
    ga, ta = a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV))
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    y = synth.random_bf16(34, (M, K)).to(DEV)
    for bad in (rmsq.GemmOpts(schedule=3, bn=128), rmsq.GemmOpts(schedule=3, ksplit=2)):
        with pytest.raises(RuntimeError, match="CTA-pair"):
            rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=bad)
    for bad in (rmsq.GemmOpts(bn=192), rmsq.GemmOpts(bn=192, schedule=2)):
        with pytest.raises(RuntimeError, match="CTA-pair"):
            rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=bad)
    with pytest.raises(RuntimeError, match="CTA-pair"):
        rmsq.a16wfp4_gemm(y, gb, tb, opts=rmsq.GemmOpts(schedule=3))
    assert rmsq.sync_status() == 0


def test_persistent_schedule_rejects():
    """The persistent schedule walks whole tiles with quantised A only."""
    M, N, K = 128, 256, 512
    a_q, a_s, b_q, b_s = operands(31, M, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    y = synth.random_bf16(32, (M, K)).to(DEV)
    with pytest.raises(RuntimeError, match="persistent"):
        rmsq.a16wfp4_gemm(y, gb, tb, opts=rmsq.GemmOpts(schedule=2))
    with pytest.raises(RuntimeError, match="persistent"):
        rmsq.mxfp4_gemm(a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV)), gb, tb,
                        opts=rmsq.GemmOpts(ksplit=2, schedule=2))
    assert rmsq.sync_status() == 0


def test_long_k_wraps_the_stage_ring(oracle_mod):
    """K = 7168 is 28 stages: every ring slot is reused several times."""
    M, N, K = 130, 136, 7168
    a_q, a_s, b_q, b_s = operands(9, M, N, K)
    for bn in (64, 256):
        d = gpu_gemm(a_q, a_s, b_q, b_s, bn)
        ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
        print(bn, parity.compare_gemm(d, ref, K, what=f"long K bn={bn}"))


def test_degenerate_operands():
    M, N, K = 130, 264, 512
    z = torch.zeros((M, K // 2), dtype=torch.uint8)
    s_hi = torch.full((M, K // 32), 254, dtype=torch.uint8)       # 2^127 scales on zero codes
    b_q, b_s = synth.mxfp4_weights(3, N, K)
    d = gpu_gemm(z, s_hi, b_q, b_s)
    assert torch.count_nonzero(d.float()).item() == 0             # exact zeros, no NaN / Inf
    s_lo = torch.zeros((M, K // 32), dtype=torch.uint8)           # 2^-127: products underflow to 0
    a_q, _ = synth.mxfp4_weights(4, M, K)
    d = gpu_gemm(a_q, s_lo, b_q, b_s)
    assert torch.isfinite(d.float()).all()
    empty = torch.empty((0, K // 2), dtype=torch.uint8, device=DEV)
    out = rmsq.mxfp4_gemm(empty, torch.zeros(512, dtype=torch.uint8, device=DEV), b_q.to(DEV),
                          rmsq.mx_scale_tiles(b_s.to(DEV)))
    assert out.shape == (0, N)


@pytest.mark.parametrize("bn", [256, 192])
def test_degenerate_operands_pair(bn):
    """The same degenerate operands through CTA pairs: zero codes under 2^127
    scales give exact zeros (no NaN / Inf), 2^-127 scales give finite output,
    and a pair whose odd CTA has rows of A only past M (M = 130) is fine."""
    M, N, K = 130, 264, 512
    opts = rmsq.GemmOpts(bn=bn, schedule=3)
    z = torch.zeros((M, K // 2), dtype=torch.uint8)
    s_hi = torch.full((M, K // 32), 254, dtype=torch.uint8)
    b_q, b_s = synth.mxfp4_weights(3, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    d = rmsq.mxfp4_gemm(z.to(DEV), rmsq.mx_scale_tiles(s_hi.to(DEV)), gb, tb, opts=opts)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d.float()).item() == 0
    s_lo = torch.zeros((M, K // 32), dtype=torch.uint8)
    a_q, _ = synth.mxfp4_weights(4, M, K)
    d = rmsq.mxfp4_gemm(a_q.to(DEV), rmsq.mx_scale_tiles(s_lo.to(DEV)), gb, tb, opts=opts)
    torch.cuda.synchronize()
    assert torch.isfinite(d.float()).all()
    assert rmsq.sync_status() == 0


def test_output_guard_band():
    """The GEMM writes exactly D[:M, :N]: canary bytes around a strided D stay."""
    M, N, K = 70, 136, 512
    a_q, a_s, b_q, b_s = operands(11, M, N, K)
    big = torch.full((M + 2, N + 24), -7.0, dtype=torch.bfloat16, device=DEV)
    d = big[1:M + 1, 8:N + 8]
    rmsq.mxfp4_gemm(a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV)), b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV)),
                    out=d)
    torch.cuda.synchronize()
    ref = gpu_gemm(a_q, a_s, b_q, b_s)
    assert torch.equal(d, ref)
    mask = torch.ones_like(big, dtype=torch.bool)
    mask[1:M + 1, 8:N + 8] = False
    assert (big[mask] == -7.0).all()


def _pipeline_inputs(M, K, seed):
    w = synth.Workload("gemm_in", "mxfp4", M=M, H=K, seed=seed, group=32, x_dist="student_t3")
    return {k: v.to(DEV) for k, v in synth.make_inputs(w).items()}, synth.make_inputs(w)


@pytest.mark.parametrize("M", [4, 64, 300, 1100])
def test_placements_agree_and_match_oracle(oracle_mod, M):
    """norm + MXFP4 quant fused, then the GEMM == norm alone, then the GEMM
    with the quant in its prologue; both against the oracle's composition."""
    K, N = 7168, 2112
    g, d_cpu = _pipeline_inputs(M, K, 21)
    b_q, b_s = synth.mxfp4_weights(22, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    (a_q, a_tiles), r1 = rmsq.add_rmsnorm_quant_mxfp4_mma_scales(g["x"], g["gamma"], g["residual"])
    fused = rmsq.mxfp4_gemm(a_q, a_tiles, gb, tb)                       # library's own tile choice
    y, r2 = rmsq.add_rmsnorm(g["x"], g["gamma"], g["residual"])
    same = rmsq.GemmOpts(bn=256)                                         # equal tiles and K split
    pre = rmsq.a16wfp4_gemm(y, gb, tb, opts=same)
    torch.cuda.synchronize()
    assert torch.equal(r1, r2)
    assert torch.equal(rmsq.mxfp4_gemm(a_q, a_tiles, gb, tb, opts=same), pre), "the two placements differ"
    ref_q = oracle_mod.add_rmsnorm_quant_mxfp4(d_cpu["x"], d_cpu["residual"], d_cpu["gamma"])
    boundary = ref_q["margin"] < parity.BOUNDARY
    assert np.array_equal(parity.u16(y)[~boundary], ref_q["y"][~boundary])
    ref = oracle_mod.mxfp4_gemm(ref_q["q"], ref_q["scale"], b_q.numpy(), b_s.numpy())
    st = parity.compare_gemm(fused[~torch.from_numpy(boundary).to(DEV)],
                             {k: v[~boundary] for k, v in ref.items()}, K, what=f"pipeline M={M}")
    assert rmsq.sync_status() == 0
    print(M, st)


@pytest.mark.parametrize("M", [1, 4, 16, 64, 128, 129, 200, 256])
def test_placements_agree_at_few_tokens(oracle_mod, M):
    """Up to two row tiles of A, at every tile width and K split the library
    picks or may be asked for there: the quantising GEMM equals the
    quantised-A GEMM bit for bit under the same options, and sampled rows
    (rows are independent) match the oracle's composition."""
    K, N = 7168, 2112
    g, d_cpu = _pipeline_inputs(M, K, 41)
    b_q, b_s = synth.mxfp4_weights(42, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    (a_q, a_tiles), _ = rmsq.add_rmsnorm_quant_mxfp4_mma_scales(g["x"], g["gamma"], g["residual"])
    y, _ = rmsq.add_rmsnorm(g["x"], g["gamma"], g["residual"])
    rows = sorted(r for r in {0, 1, M // 3, M // 2, 127, 128, M - 2, M - 1} if 0 <= r < M)
    sub = {k: (v[rows] if v.dim() == 2 else v) for k, v in d_cpu.items()}
    ref_q = oracle_mod.add_rmsnorm_quant_mxfp4(sub["x"], sub["residual"], sub["gamma"])
    keep = ref_q["margin"] >= parity.BOUNDARY
    ref = oracle_mod.mxfp4_gemm(ref_q["q"], ref_q["scale"], b_q.numpy(), b_s.numpy())
    ref = {k: v[keep] for k, v in ref.items()}
    pick = torch.tensor(rows, device=DEV)[torch.from_numpy(keep).to(DEV)]
    for bn, ksplit in [(0, 0), (64, 0), (128, 0), (128, 4), (128, 6), (256, 0), (256, 4)]:
        o = rmsq.GemmOpts(bn=bn, ksplit=ksplit)
        pre = rmsq.a16wfp4_gemm(y, gb, tb, opts=o)
        plain = rmsq.mxfp4_gemm(a_q, a_tiles, gb, tb, opts=o)
        torch.cuda.synchronize()
        assert torch.equal(pre, plain), (M, bn, ksplit)
        parity.compare_gemm(pre[pick], ref, K, what=f"M={M} bn={bn} ksplit={ksplit}")
    assert rmsq.sync_status() == 0


def test_full_size_sampled(oracle_mod):
    """The benchmarked shape (M=8192 tokens, N=2112, K=7168): the placements
    agree on every output; sampled rows (rows are independent) against the
    oracle's composition computed from the same input rows."""
    M, K, N = 8192, 7168, 2112
    g, d_cpu = _pipeline_inputs(M, K, 31)
    b_q, b_s = synth.mxfp4_weights(32, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    (a_q, a_tiles), _ = rmsq.add_rmsnorm_quant_mxfp4_mma_scales(g["x"], g["gamma"], g["residual"])
    fused = rmsq.mxfp4_gemm(a_q, a_tiles, gb, tb)
    y, _ = rmsq.add_rmsnorm(g["x"], g["gamma"], g["residual"])
    pre = rmsq.a16wfp4_gemm(y, gb, tb)
    torch.cuda.synchronize()
    assert torch.equal(fused, pre)          # neither splits K here: every sum runs in the same order
    rows = [0, 1, 127, 128, 4095, 5000, 8190, 8191]
    sub = {k: (v[rows] if v.dim() == 2 else v) for k, v in d_cpu.items()}
    ref_q = oracle_mod.add_rmsnorm_quant_mxfp4(sub["x"], sub["residual"], sub["gamma"])
    keep = ref_q["margin"] >= parity.BOUNDARY
    ref = oracle_mod.mxfp4_gemm(ref_q["q"], ref_q["scale"], b_q.numpy(), b_s.numpy())
    got = fused[torch.tensor(rows, device=DEV)][torch.from_numpy(keep).to(DEV)]
    st = parity.compare_gemm(got, {k: v[keep] for k, v in ref.items()}, K, what="full size")
    assert rmsq.sync_status() == 0
    print(st)


@pytest.mark.parametrize("pre,ksplit", [(False, 1), (False, 2), (True, 1)])
def test_bounded_wait_reports_timeout(oracle_mod, pre, ksplit):
    """A stage whose loads are never issued (test hook) makes a wait run
    out: the kernel stops, drains and frees its tensor memory, the host reads
    RMSQ_ERR_TIMEOUT, and the next GEMM on the same context is correct."""
    M, N, K = 128, 256, 2048           # at least two stages in every CTA
    a_q, a_s, b_q, b_s = operands(61, M, N, K)
    ga, ta = a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV))
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    stuck = rmsq.GemmOpts(bn=128, ksplit=ksplit, wait_limit_ns=50_000_000, debug_stall_stage=2)
    if pre:
        y = synth.random_bf16(62, (M, K)).to(DEV)
        rmsq.a16wfp4_gemm(y, gb, tb, opts=stuck)
    else:
        rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=stuck)
    assert rmsq.sync_status() == 5                      # RMSQ_ERR_TIMEOUT
    assert rmsq.sync_status() == 0                      # read and cleared
    d = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=128, ksplit=ksplit))
    torch.cuda.synchronize()
    ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
    parity.compare_gemm(d, ref, K, what="after a timed-out launch")
    assert rmsq.sync_status() == 0


def test_bounded_wait_in_a_later_tile():
    """Persistent schedule: the stalled stage sits in the second tile of the
    CTAs that walk two (160 tiles of 128 x 128 on fewer SMs, four stages
    per tile). Those CTAs stop and drain, the host reads RMSQ_ERR_TIMEOUT,
    and the next launch matches the one-tile schedule bit for bit."""
    M, N, K = 2048, 1280, 2048
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert 80 <= sms < 160
    a_q, a_s, b_q, b_s = operands(63, M, N, K)
    ga, ta = a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV))
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    stuck = rmsq.GemmOpts(bn=128, ksplit=1, wait_limit_ns=50_000_000, debug_stall_stage=6, schedule=2)
    rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=stuck)
    assert rmsq.sync_status() == 5                      # RMSQ_ERR_TIMEOUT
    assert rmsq.sync_status() == 0
    walk = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=128, ksplit=1, schedule=2))
    one = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=128, ksplit=1, schedule=1))
    torch.cuda.synchronize()
    assert torch.equal(walk, one)
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("bn", [256, 192])
def test_pair_bounded_wait_in_a_later_tile(bn):
    """CTA pairs: the stalled stage (never loaded by either CTA) sits in the
    second tile of the pairs that walk two (M = 4096, N = 2560: 160 tiles of
    256 x 256, four stages each). Both CTAs of a stalled pair stop within
    their wait limits; the host reads RMSQ_ERR_TIMEOUT; the next launch
    matches the one-tile schedule bit for bit."""
    M, N, K = 4096, 2560, 1024
    a_q, a_s, b_q, b_s = operands(64, M, N, K)
    ga, ta = a_q.to(DEV), rmsq.mx_scale_tiles(a_s.to(DEV))
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    stuck = rmsq.GemmOpts(bn=bn, wait_limit_ns=50_000_000, debug_stall_stage=6, schedule=3)
    rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=stuck)
    assert rmsq.sync_status() == 5                      # RMSQ_ERR_TIMEOUT
    assert rmsq.sync_status() == 0
    pair = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=bn, schedule=3))
    one = rmsq.mxfp4_gemm(ga, ta, gb, tb, opts=rmsq.GemmOpts(bn=256, ksplit=1, schedule=1))
    torch.cuda.synchronize()
    assert torch.equal(pair, one)
    assert rmsq.sync_status() == 0


def test_strided_operands(oracle_mod):
    """Leading dimensions wider than a row for A (codes and bf16), B and D."""
    M, N, K = 150, 200, 768
    a_q, a_s, b_q, b_s = operands(71, M, N, K)
    pa = torch.zeros((M, K // 2 + 48), dtype=torch.uint8)
    pa[:, :K // 2] = a_q
    pb = torch.zeros((N, K // 2 + 80), dtype=torch.uint8)
    pb[:, :K // 2] = b_q
    ga, gb = pa.to(DEV)[:, :K // 2], pb.to(DEV)[:, :K // 2]
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    dbig = torch.zeros((M, N + 24), dtype=torch.bfloat16, device=DEV)
    d = rmsq.mxfp4_gemm(ga, ta, gb, tb, out=dbig[:, :N])
    torch.cuda.synchronize()
    ref = oracle_mod.mxfp4_gemm(a_q.numpy(), a_s.numpy(), b_q.numpy(), b_s.numpy())
    parity.compare_gemm(d, ref, K, what="strided A, B, D")
    assert (dbig[:, N:] == 0).all()
    # bf16 A with a wider row pitch, quantised in the GEMM
    y_cpu = synth.random_bf16(72, (M, K + 64))
    y = y_cpu.to(DEV)[:, :K]
    same = rmsq.GemmOpts(bn=256)
    pre = rmsq.a16wfp4_gemm(y, gb, tb, opts=same)
    q, s = oracle_mod.group_quant_mxfp4(parity.u16(y_cpu[:, :K].contiguous()))
    ref = oracle_mod.mxfp4_gemm(q, s, b_q.numpy(), b_s.numpy())
    parity.compare_gemm(pre, ref, K, what="strided bf16 A")
    assert rmsq.sync_status() == 0


def test_default_wait_limit_is_far_above_the_runtime():
    """Every wait inside the GEMM gives up after 2 s by default; the largest
    shape the library is measured on (M = 16384 tokens, N = 2112, K = 7168,
    both placements; the quantising GEMM is the slower, about a millisecond)
    must finish in under a two-hundredth of that, so the limit only ever
    trips on a stalled GPU. check=True raises if it did."""
    M, N, K = 16384, 2112, 7168
    a_q, a_s, b_q, b_s = operands(61, M, N, K)
    ga, gb = a_q.to(DEV), b_q.to(DEV)
    ta, tb = rmsq.mx_scale_tiles(a_s.to(DEV)), rmsq.mx_scale_tiles(b_s.to(DEV))
    a_bf16 = torch.randn((M, K), device=DEV).to(torch.bfloat16)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    worst = 0.0
    for fn in (lambda: rmsq.mxfp4_gemm(ga, ta, gb, tb, out=d, check=True),
               lambda: rmsq.a16wfp4_gemm(a_bf16, gb, tb, out=d, check=True)):
        fn()
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            worst = max(worst, e0.elapsed_time(e1) * 1e-3)
    print(f"slowest launch {worst * 1e3:.3f} ms against the 2 s wait limit")
    assert worst < 2.0 / 200
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("M,pre", [(4, False), (64, False), (300, False), (4, True), (64, True)])
def test_gemm_after_the_quant_reads_its_output(M, pre):
    """The single-CTA GEMM is launched as a programmatic dependent of the
    kernel before it: right after the fused norm + quant (or the norm alone,
    for the prequant GEMM) on the same stream, with no synchronisation, it
    may start early but must read that call's activation, never what the
    buffers held before. Six different activations through the same buffers,
    back to back and inside a CUDA graph, each against a synchronised run."""
    K, N = 7168, 2112
    b_q, b_s = synth.mxfp4_weights(22, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    ins = [_pipeline_inputs(M, K, 200 + i)[0] for i in range(6)]
    x = torch.empty_like(ins[0]["x"])
    res = torch.empty_like(ins[0]["residual"])
    gamma = ins[0]["gamma"]
    q = torch.empty((M, K // 2), dtype=torch.uint8, device=DEV)
    t = torch.zeros(rmsq.mma_scale_bytes(M, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ro = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)

    def step():
        if pre:
            rmsq.add_rmsnorm(x, gamma, res, out=y, out_residual=ro)
            rmsq.a16wfp4_gemm(y, gb, tb, out=d)
        else:
            rmsq.add_rmsnorm_quant_mxfp4_mma_scales_into(x, gamma, res, q, t, ro)
            rmsq.mxfp4_gemm(q, t, gb, tb, out=d)

    refs = []
    for inp in ins:                      # synchronised between the two kernels
        x.copy_(inp["x"])
        res.copy_(inp["residual"])
        if pre:
            rmsq.add_rmsnorm(x, gamma, res, out=y, out_residual=ro)
            torch.cuda.synchronize()
            refs.append(rmsq.a16wfp4_gemm(y, gb, tb).clone())
        else:
            rmsq.add_rmsnorm_quant_mxfp4_mma_scales_into(x, gamma, res, q, t, ro)
            torch.cuda.synchronize()
            refs.append(rmsq.mxfp4_gemm(q, t, gb, tb).clone())
        torch.cuda.synchronize()
    outs = []
    for inp in ins:                      # back to back on one stream
        x.copy_(inp["x"])
        res.copy_(inp["residual"])
        step()
        outs.append(d.clone())
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(outs, refs)):
        assert torch.equal(a, b), f"activation {i}, back to back"
    side = torch.cuda.Stream(DEV)        # the same pair replayed from a CUDA graph
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step()
        for i, inp in enumerate(ins):
            x.copy_(inp["x"])
            res.copy_(inp["residual"])
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(d, refs[i]), f"activation {i}, graph replay"
    torch.cuda.current_stream().wait_stream(side)
    assert rmsq.sync_status() == 0


@pytest.mark.parametrize("M,pre", [(4, False), (64, False), (8192, False), (64, True)])
def test_quant_gemm_chain_with_no_kernel_between(M, pre):
    """Norm (+ quant) and GEMM alternate on one stream with nothing between
    them: each norm is a programmatic dependent of the GEMM before it and
    overwrites the activation that GEMM reads, each GEMM a dependent of the
    norm before it. Five activations staged in their own buffers beforehand,
    five outputs; back to back and replayed from a CUDA graph, each must
    equal the same step run alone and synchronised."""
    K, N = 7168, 2112
    b_q, b_s = synth.mxfp4_weights(23, N, K)
    gb, tb = b_q.to(DEV), rmsq.mx_scale_tiles(b_s.to(DEV))
    ins = [_pipeline_inputs(M, K, 300 + i)[0] for i in range(5)]
    gamma = ins[0]["gamma"]
    q = torch.empty((M, K // 2), dtype=torch.uint8, device=DEV)
    t = torch.zeros(rmsq.mma_scale_bytes(M, K), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ro = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ds = [torch.empty((M, N), dtype=torch.bfloat16, device=DEV) for _ in ins]

    def step(i):
        if pre:
            rmsq.add_rmsnorm(ins[i]["x"], gamma, ins[i]["residual"], out=y, out_residual=ro)
            rmsq.a16wfp4_gemm(y, gb, tb, out=ds[i])
        else:
            rmsq.add_rmsnorm_quant_mxfp4_mma_scales_into(ins[i]["x"], gamma, ins[i]["residual"], q, t, ro)
            rmsq.mxfp4_gemm(q, t, gb, tb, out=ds[i])

    refs = []
    for i in range(len(ins)):
        step(i)
        torch.cuda.synchronize()
        refs.append(ds[i].clone())
    for d in ds:
        d.zero_()
    torch.cuda.synchronize()
    for i in range(len(ins)):            # back to back
        step(i)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(ds, refs)):
        assert torch.equal(a, b), f"activation {i}, back to back"
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(len(ins)):
                step(i)
        for d in ds:
            d.zero_()
        g.replay()
        torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(ds, refs)):
        assert torch.equal(a, b), f"activation {i}, graph replay"
    torch.cuda.current_stream().wait_stream(side)
    assert rmsq.sync_status() == 0
