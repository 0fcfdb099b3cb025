// CTA-pair MXFP4 GEMM: 256 x 256 or 256 x 192 tiles of D computed by the
// tensor cores of two SMs (tcgen05 cta_group::2), persistent over the tiles.
// Shared helpers and layouts: rmsq_gemm_common.cuh; entry points, host
// checks and the tile policy that chooses this kernel: rmsq_gemm.cu.
#include "rmsq_gemm_common.cuh"

namespace rmsq {
namespace gemm {

// ------------------------------------------------------ CTA-pair kernel
// A cluster of two CTAs computes 256 x BN tiles of D (persistent: pair
// blockIdx.x / 2 walks tiles pair, pair + pairs, ... in N-fastest order) with
// M = 256 MMAs issued by the even CTA. CTA r loads its 128 rows of A and rows
// (BN/2)r.. of the tile's BN rows of B, so a span of K costs each SM 32 KB of
// operands at BN = 256 (48 KB for a 128 x 256 tile of its own). Each CTA also
// loads the tile's A scales for its rows and ALL of its B scales (the MMA
// reads both from each SM's own tensor memory); every copy of both CTAs
// completes on the even CTA's `full` barrier, which the even CTA arms for
// both. The MMA commits arrive on both CTAs' `empty` and `accum` barriers;
// both epilogues (their own 128 rows, in their own tensor memory) arrive on
// the even CTA's `tmem_empty`.
// BN = 256: one accumulator. BN = 192: two accumulators (the MMAs of the
// next tile run while the epilogue drains the last); 2 x 192 accumulator
// columns leave room for five stages' scale factors. Both take five ring
// stages: a sixth does not fit the shared memory next to the eight epilogue
// warps' staging (and with half the staging per warp, six stages measured
// 47.6 against 45.9 us). Each stage's scale factors keep their own tensor-memory slot, so
// a slot is free again when the producer may refill the stage. (A separate
// ring of five slots under seven stages, where the MMA warp waited for the
// commit of stage g - 5 before reusing a slot, starved the tensor pipe:
// 64.4 us at M = 8192 against 48.2 us.)
// Eight epilogue warps (two per lane quarter of tensor memory, each with half
// of the tile's columns) load all of their accumulator columns before their
// first store and hand the accumulator back at once, so with a single
// accumulator the next tile's MMAs wait only for those loads: at M = 8192,
// N = 2112, K = 7168 the 256-wide tile went from 49.3 us (four epilogue warps,
// release after the last of eight interleaved load/store rounds, six stages)
// to 45.9 us, past the 192-wide tile's 48.2 us.
// Stage shape measured on GB300 (BN = 256, N = 2112, K = 7168, M = 8192): one
// span x six stages 50.7 us, one x five 51.6 us, two spans x three 56.2 us.
// The 256-wide tile keeps six stages next to the full epilogue staging: that
// fits only because the dynamic shared memory starts 1024-byte aligned, so
// the layout needs no alignment slack (checked on entry: a CTA that finds it
// otherwise sets status bit 8 and writes nothing). Six stages against five:
// 45.1 against 46.2 us at M = 8192, 15.4 against 16.1 us at M = 2048.
template <int BN_>
struct PairCfg {
    static constexpr int BN = BN_;                     // columns of D per tile
    static constexpr int kRowsB = BN / 2;              // rows of B per CTA
    static constexpr int kSpanA = kBM * kSpanBytes;
    static constexpr int kSpanB = kRowsB * kSpanBytes;
    static constexpr int kStage = kSpanA + kSpanB;     // one span of K per stage
    static constexpr int kSfbAtoms = 2;                // 128-row scale tiles of B a tile touches
    static constexpr int kStages = BN == 256 ? 6 : 5;  // 192: the stages' scale factors fill the tensor memory
    static constexpr int kAcc = BN == 256 ? 1 : 2;     // accumulators in tensor memory
    static constexpr int kOffSfa = kStages * kStage;
    static constexpr int kOffSfb = kOffSfa + kStages * 1024;
    static constexpr int kOffOut = kOffSfb + kStages * kSfbAtoms * 1024;
    static constexpr int kEpiWarps = 8;                // warps 4..11
    static constexpr int kThreads = 32 * (4 + kEpiWarps);
    static constexpr int kChunks = BN / 64;            // 32-column chunks of D per epilogue warp
    static constexpr int kOutBytes = kEpiWarps * 2048; // each epilogue warp: 32 rows x 64 bytes of D
    static constexpr int kOffBar = kOffOut + kOutBytes;
    static constexpr int kBarBytes = (2 * kStages + 2 * kAcc + 1) * 8 + 16;
    static constexpr size_t kSmem = kOffBar + kBarBytes;   // no slack: the base is 1024-byte aligned
    static constexpr int kSfCols = 8 + 8 * kSfbAtoms;  // scale-factor TMEM columns per stage
    static constexpr int kTmemCols = pow2_at_least(kAcc * BN + kStages * kSfCols);
    static constexpr uint32_t kCtaTx = kSpanA + kSpanB + 1024 + kSfbAtoms * 1024;   // bytes per CTA per stage
    static_assert(BN == 256 || BN == 192, "tile width");
    static_assert(kAcc * BN + kStages * kSfCols <= 512, "tensor memory");
    static_assert(kSmem <= 232448, "shared memory");
};

template <int BN>
__global__ void __launch_bounds__(PairCfg<BN>::kThreads, 1)
    mxfp4_gemm_pair_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap map_a,
                           const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_sfa,
                           const __grid_constant__ CUtensorMap map_sfb)
{
    using C = PairCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if (smem != smem_raw) {   // every CTA of the launch sees the same base, so all leave here
        if (threadIdx.x == 0)
            atomicOr(p.status, 8u);
        return;
    }
    uint64_t *full = (uint64_t *)(smem + C::kOffBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *accum = empty + C::kStages;          // [kAcc]
    uint64_t *tmem_empty = accum + C::kAcc;        // [kAcc]
    uint64_t *drain = tmem_empty + C::kAcc;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
    auto tile_at = [&](int i, int &mt, int &nt) -> bool {   // mt: 256-row tile of A, nt: BN-row tile of B
        const int64_t t = (int64_t)pair + (int64_t)i * npairs;
        if (t >= (int64_t)p.m_tiles * p.n_tiles)
            return false;
        mt = (int)(t / p.n_tiles);
        nt = (int)(t % p.n_tiles);
        return true;
    };
    const int KS = p.k_spans;   // stages per tile

    if (threadIdx.x == 32) {
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_a) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_b) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_sfa) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_sfb) : "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(full + s)));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(empty + s)));
        }
        for (int a = 0; a < C::kAcc; ++a) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(accum + a)));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(tmem_empty + a)),
                         "r"(2 * C::kEpiWarps));   // the epilogue warps of both CTAs
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(drain)));
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                     "r"(C::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers exist before either signals the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_sf = tmem + C::kAcc * BN;
    const uint32_t full_lead = cluster_addr(saddr(full), 0);
    int issued = 0;

    if (warp == 0) {
        // ---------------------------------------------------------- loads
        int g = 0, mt, nt;
        bool stop = false;
        for (int ti = 0; !stop && tile_at(ti, mt, nt); ++ti) {
            const int a_row = mt * 256 + kBM * (int)rank;
            const int b_row = nt * BN + C::kRowsB * (int)rank;
            const int bt0 = (nt * BN) >> 7;                       // the tile's first 128-row scale tile of B
            const int sfa_tile = mt * 2 + (int)rank;
            for (int j = 0; j < KS; ++j, ++g) {
                const int s = g % C::kStages;
                if (g >= C::kStages &&
                    !warp_wait(saddr(empty + s), ((uint32_t)(g / C::kStages) & 1u) ^ 1u, abort, p)) {
                    stop = true;
                    break;
                }
                if (g != p.debug_skip_stage && elect_one()) {   // test hook: that stage never arrives
                    if (rank == 0)
                        mbar_arrive_tx(saddr(full + s), 2 * C::kCtaTx);
                    const uint32_t fb = full_lead + 8 * s;
                    uint8_t *st = smem + s * C::kStage;
                    tma_2d_pair(saddr(st), &map_a, j * kSpanBytes, a_row, fb);
                    tma_2d_pair(saddr(st + C::kSpanA), &map_b, j * kSpanBytes, b_row, fb);
                    tma_2d_pair(saddr(smem + C::kOffSfa + s * 1024), &map_sfa, 0, 4 * (sfa_tile * KS + j), fb);
#pragma unroll
                    for (int t = 0; t < C::kSfbAtoms; ++t)
                        tma_2d_pair(saddr(smem + C::kOffSfb + (s * C::kSfbAtoms + t) * 1024), &map_sfb, 0,
                                    4 * ((bt0 + t) * KS + j), fb);
                }
                __syncwarp();
                issued = g + 1;
            }
        }
        __syncwarp();
    } else if (warp == 1 && rank == 0) {
        // ------------------------------------------------------------ MMA
        int g = 0, mt, nt;
        bool any = false, stop = false;
        for (int ti = 0; !stop && tile_at(ti, mt, nt); ++ti) {
            const int acc_slot = ti % C::kAcc, use = ti / C::kAcc;
            if (use > 0) {   // both epilogues have read this accumulator's previous tile
                if (!warp_wait(saddr(tmem_empty + acc_slot), (uint32_t)((use - 1) & 1), abort, p))
                    break;
                tc_fence_after();
            }
            const uint32_t d_tmem = tmem + acc_slot * BN;
            // a tile that starts half-way into a 128-row scale tile of B (BN =
            // 192, odd tiles) reads its rows' scale columns from 2 on
            const uint32_t sfb_row_col = (uint32_t)(((nt * BN) >> 6) & 1) * 2;
            for (int j = 0; j < KS; ++j, ++g) {
                const int s = g % C::kStages;
                if (!warp_wait(saddr(full + s), (uint32_t)(g / C::kStages) & 1u, abort, p)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t sfa_col = tmem_sf + s * C::kSfCols, sfb_col = sfa_col + 8;
                    const uint32_t sfa_smem = saddr(smem + C::kOffSfa + s * 1024);
                    const uint32_t sfb_smem = saddr(smem + C::kOffSfb + s * C::kSfbAtoms * 1024);
                    const uint32_t a_smem = saddr(smem + s * C::kStage), b_smem = a_smem + C::kSpanA;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        cp_sf_pair(sfa_col + 4 * c, desc_sf(sfa_smem + c * 512));
#pragma unroll
                        for (int t = 0; t < C::kSfbAtoms; ++t)
                            cp_sf_pair(sfb_col + 4 * C::kSfbAtoms * c + 4 * t, desc_sf(sfb_smem + t * 1024 + c * 512));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = k >> 1;
                        mma_mxf4_pair(d_tmem, desc_sw128(a_smem + 32 * k), desc_sw128(b_smem + 32 * k),
                                      idesc_mxf4(BN, (k & 1) * 2, 2 * kBM), sfa_col + 4 * c,
                                      sfb_col + 4 * C::kSfbAtoms * c + sfb_row_col, (j | k) != 0);
                    }
                    mma_commit_pair(saddr(empty + s), 3);
                }
                __syncwarp();
                any = true;
            }
            if (!stop && elect_one())
                mma_commit_pair(saddr(accum + acc_slot), 3);   // this tile's accumulators are complete
            __syncwarp();
        }
        if (*abort && any && elect_one()) {
            // drain the tensor cores before the tensor memory is freed
            mma_commit_pair(saddr(drain), 1);
            const uint64_t t0 = gtimer();
            while (!mbar_test(saddr(drain), 0) && gtimer() - t0 < (uint64_t)p.wait_limit_ns) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------- epilogue
        // Warp w reads tensor-memory lanes 32 (w % 4).. (32 of this CTA's
        // rows) and column half (w - 4) / 4 of the tile: all of its chunks
        // are loaded before the first store and the accumulator is handed
        // back, then the chunks go to D through shared memory, 32 columns at
        // a time, so that each store instruction writes eight rows' whole
        // 64-byte pieces (16-byte piece j of row i at j ^ ((i / 2) mod 4):
        // conflict-free both ways).
        constexpr int NCH = C::kChunks;
        const int q = warp & 3, half = (warp - 4) >> 2;
        uint8_t *const stage_w = smem + C::kOffOut + (warp - 4) * 2048;
        const int cj = lane & 3;
        int mt, nt;
        for (int ti = 0; tile_at(ti, mt, nt); ++ti) {
            const int acc_slot = ti % C::kAcc, use = ti / C::kAcc;
            if (!warp_wait(saddr(accum + acc_slot), (uint32_t)(use & 1), abort, p))
                break;
            tc_fence_after();
            const int64_t row0 = (int64_t)mt * 256 + kBM * (int)rank + q * 32, n0 = (int64_t)nt * BN;
            const int c_first = half * NCH;   // first 32-column chunk of this warp
            const uint32_t trow = tmem + acc_slot * BN + ((uint32_t)(q * 32) << 16) + c_first * 32;
            const uint32_t tmem_empty_lead = cluster_addr(saddr(tmem_empty + acc_slot), 0);
            // chunks of this warp that hold columns < N (warp-uniform; N is a multiple of 8)
            const int64_t cols_left = p.N - n0 - (int64_t)c_first * 32;
            const int nch = row0 < p.M ? (int)max((int64_t)0, min((int64_t)NCH, (cols_left + 31) / 32)) : 0;
            uint32_t acc[NCH][32];
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                if (c < nch)
                    tmem_ld32_issue(trow + c * 32, acc[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                tmem_hold(acc[c]);
            // the accumulator may now be overwritten by the next tile's MMAs
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(tmem_empty_lead);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if (c >= nch)
                    continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 o;
                    o.x = pack_bf16x2(__uint_as_float(acc[c][8 * j + 0]), __uint_as_float(acc[c][8 * j + 1]));
                    o.y = pack_bf16x2(__uint_as_float(acc[c][8 * j + 2]), __uint_as_float(acc[c][8 * j + 3]));
                    o.z = pack_bf16x2(__uint_as_float(acc[c][8 * j + 4]), __uint_as_float(acc[c][8 * j + 5]));
                    o.w = pack_bf16x2(__uint_as_float(acc[c][8 * j + 6]), __uint_as_float(acc[c][8 * j + 7]));
                    *reinterpret_cast<uint4 *>(stage_w + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = o;
                }
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int rr = it * 8 + (lane >> 2);
                    const uint4 v = *reinterpret_cast<const uint4 *>(stage_w + rr * 64 + ((cj ^ ((rr >> 1) & 3)) << 4));
                    const int64_t gm = row0 + rr, gn = n0 + (c_first + c) * 32 + cj * 8;
                    if (gm < p.M && gn < p.N && RMSQ_IN_BOUNDS(p.status, gn + 8 <= p.N))
                        *reinterpret_cast<uint4 *>(p.d + gm * p.ldd + gn) = v;
                }
                __syncwarp();
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 0 && rank == 0) {
        // let the copies of stages this pair armed land before either CTA goes
        const uint64_t t0 = gtimer();
        for (int i = (issued > C::kStages ? issued - C::kStages : 0); i < issued; ++i) {
            if (i == p.debug_skip_stage)
                continue;
            const uint32_t fb = saddr(full + i % C::kStages);
            const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
            while (!mbar_test(fb, ph) && gtimer() - t0 < (uint64_t)p.wait_limit_ns) {
            }
        }
    }
    cluster_sync();   // neither CTA leaves while the other may still signal its barriers or read its memory
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
    }
}

namespace {

// CTA pairs resident at once with the pair kernel's shared memory (cached per device)
template <int BN>
int pair_capacity_t(int dev)
{
    using C = PairCfg<BN>;
    static std::atomic<int> cap[128];   // every thread stores the same value
    if (dev < 0 || dev >= 128)
        return 0;
    int c = cap[dev].load(std::memory_order_acquire);
    if (!c) {
        if (cudaFuncSetAttribute(mxfp4_gemm_pair_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::kSmem) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(C::kThreads, 1, 1);
        cfg.dynamicSmemBytes = C::kSmem;
        cudaLaunchAttribute cl[1];
        cl[0].id = cudaLaunchAttributeClusterDimension;
        cl[0].val.clusterDim.x = 2;
        cl[0].val.clusterDim.y = 1;
        cl[0].val.clusterDim.z = 1;
        cfg.attrs = cl;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mxfp4_gemm_pair_kernel<BN>, &cfg) != cudaSuccess || n <= 0)
            return 0;
        cap[dev].store(n, std::memory_order_release);
        c = n;
    }
    return c;
}

template <int BN>
cudaError_t launch_pair_t(const GemmLaunch &g, cudaStream_t st)
{
    using C = PairCfg<BN>;
    GemmParams p{};
    p.d = (uint16_t *)g.d;
    p.ldd = g.ldd;
    p.M = g.M;
    p.N = g.N;
    p.k_spans = (int32_t)(g.K / kSpanK);
    p.b_row_tiles = (int32_t)((g.N + 127) / 128);
    p.a_box_rows = kBM;
    p.ksplit = 1;
    p.persistent = 1;
    p.m_tiles = (int32_t)((g.M + 255) / 256);
    p.n_tiles = (int32_t)((g.N + BN - 1) / BN);
    p.debug_skip_stage = g.debug_skip_stage;
    p.wait_limit_ns = g.wait_limit_ns;
    p.status = g.status;
    const int64_t m_tiles128 = (g.M + 127) / 128;
    CUtensorMap ma, mb, msa, msb;
    if (!make_code_map(&ma, g.a_q, g.M, g.K / 2, g.lda, kBM) ||
        !make_code_map(&mb, g.b_q, g.N, g.K / 2, g.ldb, C::kRowsB) ||
        !make_scale_map(&msa, g.a_scale, m_tiles128 * p.k_spans * 4) ||
        !make_scale_map(&msb, g.b_scale, (int64_t)p.b_row_tiles * p.k_spans * 4))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int cap = pair_capacity_t<BN>(dev);
    if (cap <= 0)
        return cudaErrorInvalidConfiguration;
    const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
    const int pairs = (int)(tiles < cap ? tiles : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute cl[1];
    cl[0].id = cudaLaunchAttributeClusterDimension;
    cl[0].val.clusterDim.x = 2;
    cl[0].val.clusterDim.y = 1;
    cl[0].val.clusterDim.z = 1;
    cfg.attrs = cl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mxfp4_gemm_pair_kernel<BN>, p, ma, mb, msa, msb);
}

}  // namespace

int pair_capacity(int dev, int bn)
{
    return bn == 192 ? pair_capacity_t<192>(dev) : bn == 256 ? pair_capacity_t<256>(dev) : 0;
}

cudaError_t launch_pair(const GemmLaunch &g, cudaStream_t st)
{
    switch (g.bn) {
    case 256: return launch_pair_t<256>(g, st);
    case 192: return launch_pair_t<192>(g, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gemm
}  // namespace rmsq
