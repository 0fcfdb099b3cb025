"""The GEMM's launch choice (tile width, K split, schedule) through the host-only
plan query rmsq_gemm_plan_for, which runs the same function the GEMM entry
points run before they launch. No GPU is needed: the SM count and the CTA-pair
capacities are arguments here (152 SMs holding 76 pairs of either width, one
pair per two SMs, stand for the GB300 the widths were measured on)."""

import ctypes
import itertools

import pytest

from mxfp4_activation_quant_gb300 import build as lib_build
from mxfp4_activation_quant_gb300 import rmsq

SMS, PAIRS = 152, 76
N, K = 2112, 7168                      # the consumer projection the widths were measured on


@pytest.fixture(scope="module")
def L():
    lib_build.build()
    return rmsq.lib()


def plan(M, n=N, k=K, prequant=False, opts=None, sms=SMS, pairs=(PAIRS, PAIRS)):
    p = rmsq.gemm_plan(M, n, k, sms=sms, pairs_256=pairs[0], pairs_192=pairs[1], prequant=prequant, opts=opts)
    return p.bn, p.ksplit, p.schedule, p.persistent_ctas


def raw_plan(L, M, n, k, opts, prequant=0, sms=SMS, pairs=(PAIRS, PAIRS)):
    p = rmsq.GemmPlan(7, 7, 7, 7)
    st = L.rmsq_gemm_plan_for(prequant, M, n, k, ctypes.byref(opts) if opts is not None else None, sms,
                              pairs[0], pairs[1], ctypes.byref(p))
    return st, (p.bn, p.ksplit, p.schedule, p.persistent_ctas)


@pytest.mark.parametrize("prequant,M,want", [
    # quantised A: 64-row B tiles and K split 4 for one row tile of A (decode) ...
    (False, 1, (64, 4, 1, 0)),
    (False, 4, (64, 4, 1, 0)),
    (False, 64, (64, 4, 1, 0)),
    (False, 128, (64, 4, 1, 0)),
    # ... 128-row tiles from two row tiles of A on, K split to fill the SMs ...
    (False, 256, (128, 4, 1, 0)),
    (False, 512, (128, 2, 1, 0)),
    # ... CTA pairs once 256-row tiles give half the SMs a tile, 256 x 256 tiles
    # (the 192-wide tile's busiest pair has fewer columns at 8192 tokens, but
    # not 15 % fewer)
    (False, 2048, (256, 1, 3, 0)),
    (False, 8192, (256, 1, 3, 0)),
    (False, 16384, (256, 1, 3, 0)),
    # A in bf16 (quantised in the GEMM): 64-row tiles up to 16 tokens ...
    (True, 1, (64, 4, 1, 0)),
    (True, 16, (64, 4, 1, 0)),
    # ... the widest tile for the rest of one row tile (K split 8: 9 clusters) ...
    (True, 17, (256, 8, 1, 0)),
    (True, 128, (256, 8, 1, 0)),
    # ... 128-row tiles for two row tiles (18 clusters of 8 would not fit at once) ...
    (True, 129, (128, 4, 1, 0)),
    (True, 256, (128, 4, 1, 0)),
    # ... and the widest tile again from three row tiles on; no pairs, no persistent grid
    (True, 257, (256, 5, 1, 0)),
    (True, 512, (256, 4, 1, 0)),
    (True, 8192, (256, 1, 1, 0)),
])
def test_measured_choices(L, prequant, M, want):
    assert plan(M, prequant=prequant) == want


def test_explicit_schedules(L):
    # persistent grid: one CTA per SM walks 64 x 17 tiles of 128 x 128
    assert plan(8192, opts=rmsq.GemmOpts(bn=128, ksplit=1, schedule=2)) == (128, 1, 2, SMS)
    # with fewer tiles than SMs the persistent grid has one CTA per tile
    assert plan(128, opts=rmsq.GemmOpts(bn=256, ksplit=1, schedule=2)) == (256, 1, 2, 9)
    # one tile per CTA where the library would pair CTAs
    assert plan(8192, opts=rmsq.GemmOpts(schedule=1)) == (256, 1, 1, 0)
    # CTA pairs at a small size and an explicit width: no capacity needed
    assert plan(4, opts=rmsq.GemmOpts(schedule=3, bn=256), pairs=(0, 0)) == (256, 1, 3, 0)
    assert plan(4, opts=rmsq.GemmOpts(schedule=3, bn=192)) == (192, 1, 3, 0)


def test_pair_width_follows_the_capacity(L):
    # the width is the one whose busiest pair does the least work, a 192-wide
    # column charged 15 %: at 8192 tokens (9 x 32 = 288 tiles of 256 x 256,
    # 11 x 32 = 352 of 256 x 192) 44 resident pairs give the busiest pair 7
    # wide tiles (1792 columns) against 8 narrow ones (1536 x 1.15 = 1766)
    assert plan(8192, pairs=(44, 44))[0] == 192
    assert plan(8192, pairs=(48, 48))[0] == 256
    assert plan(8192, pairs=(288, 288))[0] == 256
    assert plan(8192, pairs=(PAIRS, PAIRS))[0] == 256


SHAPES_M = [1, 3, 16, 17, 100, 128, 129, 256, 257, 300, 1000, 2048, 8192, 16384]
SHAPES_N = [8, 64, 136, 520, 2112, 7168]
SHAPES_K = [256, 512, 1536, 7168]
OPTS = [rmsq.GemmOpts(bn=bn, ksplit=ks, schedule=sc)
        for bn, ks, sc in itertools.product([0, 64, 128, 192, 256], [0, 1, 2, 3, 8], [0, 1, 2, 3])]


def test_plan_invariants(L):
    ok = 0
    for prequant, M, n, k, o, sms in itertools.product([0, 1], SHAPES_M, SHAPES_N, SHAPES_K, OPTS, [SMS, 8]):
        st, (bn, ks, sc, ctas) = raw_plan(L, M, n, k, o, prequant, sms)
        if st != 0:
            assert (bn, ks, sc, ctas) == (0, 0, 0, 0)
            continue
        ok += 1
        case = (prequant, M, n, k, o.bn, o.ksplit, o.schedule, sms)
        assert bn in (64, 128, 192, 256), case
        assert 1 <= ks <= min(8, k // 256), case
        if o.bn:
            assert bn == o.bn, case
        if o.ksplit and sc != 3:
            assert ks == o.ksplit, case
        if o.schedule:
            assert sc == o.schedule, case
        if sc == 3:                                       # pairs: quantised A, no K split
            assert not prequant and ks == 1 and ctas == 0 and bn in (192, 256), case
        elif bn == 192:
            raise AssertionError(("192-row tiles outside the pair schedule", case))
        tiles = -(-M // 128) * -(-n // bn)
        if sc == 2:                                       # persistent: one CTA per SM, at most one per tile
            assert not prequant and ks == 1 and ctas == min(tiles, sms), case
        else:
            assert ctas == 0, case
        if not o.ksplit and sc == 1:                      # the automatic split never oversubscribes the SMs
            assert tiles * ks <= max(sms, tiles), case
            assert ks == 1 or tiles < sms, case
    assert ok > 10000


@pytest.mark.parametrize("opts,shape,status", [
    (rmsq.GemmOpts(bn=96), (64, 256, 1024), 1),
    (rmsq.GemmOpts(bn=192), (64, 256, 1024), 3),          # 192 only with CTA pairs
    (rmsq.GemmOpts(ksplit=9), (64, 256, 1024), 1),
    (rmsq.GemmOpts(ksplit=-1), (64, 256, 1024), 1),
    (rmsq.GemmOpts(wait_limit_ns=-1), (64, 256, 1024), 1),
    (rmsq.GemmOpts(debug_stall_stage=-1), (64, 256, 1024), 1),
    (rmsq.GemmOpts(schedule=4), (64, 256, 1024), 1),
    (rmsq.GemmOpts(), (64, 256, 1000), 3),                # K % 256
    (rmsq.GemmOpts(), (64, 260, 1024), 3),                # N % 8
    (rmsq.GemmOpts(), (-1, 256, 1024), 1),
    (rmsq.GemmOpts(), (64, 256, 0), 1),
])
def test_rejections_match_the_gemm_calls(L, opts, shape, status):
    """The GEMM calls check options and shape before anything else, so the
    same arguments give the same status with no GPU present."""
    M, n, k = shape
    base = 1 << 40
    got_gemm = L.rmsq_mxfp4_gemm_ex(base, k // 2, base + (1 << 32), base + (2 << 32), k // 2, base + (3 << 32),
                                    base + (4 << 32), n, M, n, k, None, ctypes.byref(opts))
    got_pre = L.rmsq_a16wfp4_gemm_ex(base, k, base + (2 << 32), k // 2, base + (3 << 32), base + (4 << 32), n, M, n,
                                     k, None, ctypes.byref(opts))
    st0, p0 = raw_plan(L, M, n, k, opts, 0)
    st1, p1 = raw_plan(L, M, n, k, opts, 1)
    assert got_gemm == got_pre == st0 == st1 == status
    assert p0 == p1 == (0, 0, 0, 0)


def test_plan_specific_rejections(L):
    unsupported, invalid = 3, 1
    assert raw_plan(L, 64, N, K, rmsq.GemmOpts(schedule=3), prequant=1)[0] == unsupported
    assert raw_plan(L, 64, N, K, rmsq.GemmOpts(schedule=3, bn=128))[0] == unsupported
    assert raw_plan(L, 64, N, K, rmsq.GemmOpts(schedule=3, ksplit=2))[0] == unsupported
    assert raw_plan(L, 64, N, K, rmsq.GemmOpts(schedule=2), prequant=1)[0] == unsupported
    assert raw_plan(L, 64, N, K, rmsq.GemmOpts(schedule=2, ksplit=2))[0] == unsupported
    assert raw_plan(L, 64, N, 1024, rmsq.GemmOpts(ksplit=8))[0] == invalid       # 4 spans of K
    assert raw_plan(L, 64, N, K, None, sms=0)[0] == invalid
    assert raw_plan(L, 8192, N, K, None, pairs=(0, PAIRS))[0] == invalid        # capacity needed, not given
    assert raw_plan(L, 65535 * 128 + 1, N, K, None)[0] == unsupported
    assert raw_plan(L, 65535 * 128, N, K, None)[0] == 0
    assert L.rmsq_gemm_plan_for(0, 64, N, K, None, SMS, PAIRS, PAIRS, None) == invalid
    with pytest.raises(rmsq.RmsqError, match="INVALID_ARG"):
        plan(64, sms=-3)


def test_nothing_launched_for_empty_products(L):
    assert raw_plan(L, 0, N, K, None) == (0, (0, 0, 0, 0))
    assert raw_plan(L, 64, 0, K, None, prequant=1) == (0, (0, 0, 0, 0))
