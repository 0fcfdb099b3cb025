// Block-scaled MXFP4 GEMM on the 5th-generation tensor cores (tcgen05): the
// consumer of the fused norm + MXFP4 quant,
//     D[M, N] (bf16) = A[M, K] B[N, K]^T,
// A and B in MXFP4 along K (E2M1 codes two per byte, one E8M0 scale per 32
// elements; OCP Microscaling Formats v1.0). It serves the comparison of the
// two places the activation quant can sit (ATOM PR "Triton fusion/GEMM
// optimizations for DS FP4 and FP8": fused RMSNorm + quant ahead of the GEMM
// above concurrency 4, the quant inside an A16W-FP4 GEMM, "prequant", at
// concurrency 4):
//   * A already quantised -- codes [M, K/2] and scales in the MMA tile layout,
//     as rmsq_add_rmsnorm_quant_mxfp4_mma_scales writes them -- loaded by TMA;
//   * A in bf16 (prequant): eight warps quantise each K span of A into shared
//     memory with the fused kernel's own group-32 rule.
//
// One CTA computes a 128 x BN tile (BN = 64, 128 or 256): the MMA's M = 128
// rows of A, N = BN rows of B. K advances in spans of 256 elements = 128
// bytes per row (one 128-byte swizzle span, four MMAs of K = 64); a ring
// stage holds one to four spans behind one barrier phase (GemmCfg). With
// fewer tiles than SMs, the CTAs of a thread-block cluster split K and add
// their fp32 partial sums through distributed shared memory, in rank order;
// with more, a persistent grid walks the tiles (the ring runs on from one
// tile into the next). For 256-row B tiles without a K split, CTA pairs
// (mxfp4_gemm_pair_kernel in rmsq_gemm_pair.cu, tcgen05 cta_group::2)
// compute 256 x 256 or 256 x 192 tiles with the tensor cores of two SMs.
// Warp roles (256 threads): warp 0 issues the TMA and bulk loads; warp 1
// owns the tensor memory and issues tcgen05.cp (scale factors, shared ->
// tensor memory) and tcgen05.mma (one elected lane each); warps 4-7 run the
// epilogue (tcgen05.ld -> bf16 -> shared memory -> whole 128-byte lines of
// D, or 64-byte pieces of rows for 64-row tiles). The prequant kernel has 384
// threads: warps 4-11 quantise A and then share the epilogue.
// Every mbarrier wait is bounded; a wait that runs out sets the status word,
// makes the other roles stop, drains what is in flight and frees the tensor
// memory before the CTA exits.
//
// Layouts (measured on GB300 with a self-checking probe before this kernel
// was written, and pinned by the parity tests):
//   * operands in shared memory: K-major rows of 128 bytes, 8-row / 1024-byte
//     atoms with the 128-byte swizzle (16-byte chunk c of row r stored at
//     chunk c ^ (r % 8)); the descriptor's start address moves 32 bytes per
//     MMA (K = 64 E2M1 elements), stride between 8-row groups 1024 bytes;
//   * scale factors in tensor memory, per 128-element K chunk: A in 4
//     columns, B in 4 columns per 128 rows of B. Row m of A reads lane m,
//     column m / 32, bytes sf_id and sf_id + 1 (its two 32-element groups of
//     the MMA's K = 64); row n of B reads lane n % 32, column n / 32. That is
//     the 512-byte tile of 128 rows x 4 groups at (r % 32) * 16 + (r / 32) * 4
//     + g copied by tcgen05.cp .32x128b.warpx4 (rows r % 32 -> lanes, the
//     same data in all four lane quarters).
#include "rmsq_gemm_common.cuh"

namespace rmsq {
namespace gemm {

// A stage of the ring is kSpans K-spans of 256 elements (one 128-byte
// swizzle span each: four MMAs of K = 64) behind ONE barrier phase. Measured
// on GB300: a TMA completion phase costs ~0.25 us, serialised per SM,
// whatever it carries (8 KB per phase gave 29 GB/s per CTA, 32 KB 80 GB/s,
// and more phases in flight did not help), so stages carry as many bytes as
// the ring allows -- except that the widest tile of the plain GEMM keeps a
// deeper ring of single-span stages, which measured faster for it (M = 8192:
// 65.7 us with 4 x 1 span against 86.7 us with 2 x 2 spans), while the
// prequant kernel's widest tile takes 2 x 2 (8.7 against 11.9 us at 4
// tokens, equal at 64 and more). 64-row tiles: 4 spans x 2 stages (6.1
// against 6.8 us at 4 tokens); 128-row tiles: 2 spans x 3 stages.
// A stage's operands come in few copies, since issuing each costs the
// producer time as well: A of all its spans in one 3-D box, B likewise, the
// A scale tiles of its spans in one bulk copy and the B scale tiles in one
// per 128-row scale tile (at 4 tokens the GEMM alone went from 6.1 to 5.8 us
// against one box and one copy per span). The stage holds A's spans, then
// B's spans; B's scale tiles by scale tile, then span.
template <int BN, bool PRE = false>
struct GemmCfg {
    static constexpr int kSpans = BN == 64 ? 4 : (BN == 128 ? 2 : (PRE ? 2 : 1));
    static constexpr int kStages = BN == 64 ? 2 : (BN == 128 ? 3 : (PRE ? 2 : 4));
    static constexpr int kSfbAtoms = BN >= 128 ? BN / 128 : 1;   // 128-row scale tiles of B per K chunk
    static constexpr int kSpanA = kBM * kSpanBytes;             // A codes of one span (16 KB)
    static constexpr int kSpanB = BN * kSpanBytes;
    // a stage: A of its spans, then B of its spans (each loaded by one 3-D box)
    static constexpr int kAB = kSpans * (kSpanA + kSpanB);        // operand bytes of a stage
    static constexpr int kStageA = kSpans * kSpanA;
    static constexpr int kSfaSpan = 2 * 512;                      // two 128-element K chunks
    static constexpr int kSfbSpan = kSfbAtoms * 2 * 512;
    static constexpr int kSfColsSpan = 8 + 8 * kSfbAtoms;        // scale-factor TMEM columns per span
    static constexpr int kSfCols = kSpans * kSfColsSpan;          // ... per stage
    static constexpr int kTmemCols = pow2_at_least(BN + kStages * kSfCols);
    static constexpr int kOffSfa = kStages * kAB;
    static constexpr int kOffSfb = kOffSfa + kStages * kSpans * kSfaSpan;
    // plain GEMM: each epilogue warp stages 32 rows x kStoreCols columns of D
    // here. 64-row tiles stage 32 columns (64-byte pieces of rows), so that
    // the CTA's shared memory leaves room on its SM for a block of the norm +
    // quant kernel it is launched behind (both then run at once).
    static constexpr int kStoreCols = BN == 64 ? 32 : 64;
    static constexpr int kOffOut = kOffSfb + kStages * kSpans * kSfbSpan;
    static constexpr int kOutBytes = PRE ? 0 : 4 * 32 * kStoreCols * 2;
    static constexpr int kOffBar = kOffOut + kOutBytes;
    static constexpr int kBarBytes = (2 * kStages + 3) * 8 + 16;
    static constexpr size_t kSmem = 1024 + kOffBar + kBarBytes;
    static_assert(kTmemCols <= 512, "tensor memory");
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(kBM * (BN + 4) * 4 <= kOffSfa, "split-K partials fit in the operand ring");
};

// ---------------------------------------------------- prequant (A in bf16)

// The 256 threads of warps 4-11 quantise the valid rows R of the A tile for
// each K span of this CTA. Item i = t + 256 j of a span is 16-byte vector
// (i % 32) of row (i / 32): warp w takes rows w, w + 8, ..., a row's 32 lanes
// read its 512 contiguous bytes, and the 4 lanes of a 32-element group find
// the group's amax with two shuffles. The arithmetic is the fused kernel's:
// X from the group's largest magnitude, elements times 2^-X (exact),
// saturating round-to-nearest-even E2M1.
//
// A thread's items of a stage (its spans x NI) go in chunks of up to 8 that
// never cross a stage: the wait for the stage's slot comes before its first
// chunk and the arrival after its last, and the next chunk's loads (possibly
// the next stage's) are issued before the current chunk is processed. The
// chunk's items go through each step together without branches, so their
// load -> shuffle -> convert chains overlap.
template <int BN>
__device__ __forceinline__ bool prequant_loop(const GemmParams &p, int64_t m0, int R, int ks0, int KL,
                                              uint8_t *smem, uint64_t *full, uint64_t *empty, volatile int *abort)
{
    using C = GemmCfg<BN, true>;
    const int t = threadIdx.x - 128;          // 0 .. kQuantThreads - 1
    const int w = t >> 5, vec = t & 31, g = vec >> 2;
    const int NI = (R + 7) >> 3;              // items per thread per span
    const int NST = (KL + C::kSpans - 1) / C::kSpans;
    const uint4 *base = p.a_bf16 + m0 * p.lda_v + vec;
    auto items = [&](int j) { return min(C::kSpans, KL - j * C::kSpans) * NI; };
    uint4 cur[8], nxt[8];

    auto load_chunk = [&](int j, int c0, uint4 (&v)[8]) {
        const int n = items(j);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = c0 + u, sp = idx / NI, row = w + 8 * (idx - sp * NI);
            const bool ok = idx < n && row < R;
            v[u] = ok ? __ldg(base + row * p.lda_v + (int64_t)(ks0 + j * C::kSpans + sp) * (kSpanK / 8))
                      : make_uint4(0, 0, 0, 0);
        }
    };

    int j = 0, c0 = 0;
    if (NST > 0)
        load_chunk(0, 0, cur);
    while (j < NST) {
        const int n = items(j), s = j % C::kStages;
        int jn = j, cn = c0 + 8;
        if (cn >= n) {
            jn = j + 1;
            cn = 0;
        }
        if (jn < NST)
            load_chunk(jn, cn, nxt);
        if (c0 == 0 && !warp_wait(saddr(empty + s), ((uint32_t)(j / C::kStages) & 1u) ^ 1u, abort, p))
            return false;
        uint32_t am[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            am[u] = amax_bits_bf16x8(cur[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            am[u] = max(am[u], __shfl_xor_sync(0xffffffffu, am[u], 1));
#pragma unroll
        for (int u = 0; u < 8; ++u)
            am[u] = max(am[u], __shfl_xor_sync(0xffffffffu, am[u], 2));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = c0 + u, sp = idx / NI, row = w + 8 * (idx - sp * NI);
            const bool ok = idx < n && row < R;
            const int X = mx_exponent_from_bits(am[u]);
            const float2 mult = f2(__uint_as_float((uint32_t)(127 - X) << 23));   // 2^-X
            const uint4 v = cur[u];
            const uint32_t codes = e2m1x8(mul2(unpack_bf16x2(v.x), mult), mul2(unpack_bf16x2(v.y), mult),
                                          mul2(unpack_bf16x2(v.z), mult), mul2(unpack_bf16x2(v.w), mult));
            if (ok) {
                uint8_t *sA = smem + s * C::kAB + sp * C::kSpanA;
                *reinterpret_cast<uint32_t *>(sA + row * kSpanBytes + ((g ^ (row & 7)) << 4) + (vec & 3) * 4) =
                    codes;
                if ((vec & 3) == 0)            // scale tile g/4: (row % 32) * 16 + (row / 32) * 4 + g % 4
                    smem[C::kOffSfa + (s * C::kSpans + sp) * C::kSfaSpan + (g >> 2) * 512 + (row & 31) * 16 +
                         (row >> 5) * 4 + (g & 3)] = (uint8_t)(X + 127);
            }
        }
        if (c0 + 8 >= n) {                     // the stage's last chunk
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(saddr(full + s));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            cur[u] = nxt[u];
        j = jn;
        c0 = cn;
    }
    return true;
}

// ------------------------------------------------------------------ kernel

template <int BN, bool PREQUANT>
__global__ void __launch_bounds__(gemm_threads<PREQUANT>(), 1)
    mxfp4_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b)
{
    using C = GemmCfg<BN, PREQUANT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + C::kOffBar);
    uint64_t *empty = full + C::kStages;
    uint64_t *accum = empty + C::kStages;
    uint64_t *tmem_empty = accum + 1;
    uint64_t *drain = tmem_empty + 1;
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    volatile int *abort = (volatile int *)(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tiles: one per CTA from the grid, or -- persistent launches -- tiles
    // blockIdx.x, blockIdx.x + gridDim.x, ... of the n-fastest tile order.
    // (m0, n0, R) below are the CTA's first tile; the split-K reduction, which
    // only one-tile launches use, refers to them.
    auto tile_at = [&](int i, int &mt, int &nt) -> bool {
        if (!p.persistent) {
            mt = (int)blockIdx.y;
            nt = (int)blockIdx.x;
            return i == 0;
        }
        const int64_t t = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;
        if (t >= (int64_t)p.m_tiles * p.n_tiles)
            return false;
        mt = (int)(t / p.n_tiles);
        nt = (int)(t % p.n_tiles);
        return true;
    };
    int m_tile = 0, n_tile = 0;
    tile_at(0, m_tile, n_tile);
    const int64_t m0 = (int64_t)m_tile * kBM, n0 = (int64_t)n_tile * BN;
    // this CTA's spans of K: all of them, or its share when a cluster splits K
    const int KS = p.k_spans;
    const int kz = (int)blockIdx.z;
    const int ks0 = (int)((int64_t)KS * kz / p.ksplit), KL = (int)((int64_t)KS * (kz + 1) / p.ksplit) - ks0;
    const int R = (int)min((int64_t)kBM, p.M - m0);    // rows of the tile that exist

    if (threadIdx.x == 32) {
        // bring both tensor maps into the descriptor cache before the first copy
        asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_b) : "memory");
        if (!PREQUANT)
            asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&map_a) : "memory");
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(full + s)),
                         "r"(PREQUANT ? 1 + kQuantThreads : 1));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(empty + s)));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(accum)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(tmem_empty)),
                     "r"(PREQUANT ? kQuantThreads : 128));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(drain)));
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                     "r"(C::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_sf = tmem + BN;   // scale-factor columns follow the accumulator
    int issued = 0;                       // warp 0: stages (counted over all tiles) whose loads were issued

    // Stages are counted over all of the CTA's tiles (g): the ring runs on
    // from one tile into the next.
    const int NST = (KL + C::kSpans - 1) / C::kSpans;            // stages per tile
    const int a_pitch = PREQUANT ? C::kSpanA : p.a_box_rows * kSpanBytes;   // bytes between A's spans in a stage
    if (warp == 0) {
        // ---------------------------------------------------------- loads
        // The whole warp runs the loop (its values stay warp-uniform) and one
        // elected lane issues the copies.
        int g = 0;
        int mt, nt;
        for (int ti = 0; tile_at(ti, mt, nt); ++ti) {
            const int64_t tm0 = (int64_t)mt * kBM, tn0 = (int64_t)nt * BN;
            const int bt0 = (int)(tn0 >> 7);                         // first 128-row scale tile of B
            int atoms = 0;
            for (int t = 0; t < C::kSfbAtoms; ++t)
                atoms += (bt0 + t < p.b_row_tiles);
            // Bytes a stage of nsp spans brings: the 3-D boxes of A and B always
            // carry kSpans spans (spans past the end of K read as zero, spans past
            // this CTA's share of K are the next share's, which no MMA here
            // reads), the scale copies exactly nsp.
            auto stage_tx = [&](int nsp) -> uint32_t {
                return (uint32_t)(C::kSpans * C::kSpanB + nsp * atoms * 1024) +
                       (PREQUANT ? 0u : (uint32_t)(C::kSpans * p.a_box_rows * kSpanBytes + nsp * C::kSfaSpan));
            };
            // B and its scales for stage j of this tile (one elected lane): one
            // 3-D box of all the stage's spans, one copy of their scale tiles per
            // 128-row scale tile of B
            auto load_b = [&](int j, int s, int nsp, uint32_t fb) {
                const int ks = ks0 + j * C::kSpans;
                tma_3d(saddr(smem + s * C::kAB + C::kStageA), &map_b, 0, (int)tn0, ks, fb);
                for (int t = 0; t < C::kSfbAtoms; ++t)
                    if (bt0 + t < p.b_row_tiles)
                        bulk_g2s(saddr(smem + C::kOffSfb + ((s * C::kSfbAtoms + t) * C::kSpans) * 1024),
                                 p.b_scale + ((int64_t)(bt0 + t) * (2 * KS) + 2 * ks) * 512, 1024u * nsp, fb);
            };
            // The first tile's first stages are free from the start: their B
            // loads (which do not depend on the kernel before this one) are
            // issued before the wait for that kernel, their A loads after it.
            int pre = 0;
            if (!PREQUANT && ti == 0) {
                pre = min(C::kStages, NST);
                if (elect_one()) {
                    for (int j = 0; j < pre; ++j) {
                        if (j == p.debug_skip_stage)        // test hook: that stage never arrives
                            continue;
                        const int nsp = min(C::kSpans, KL - j * C::kSpans);
                        mbar_arrive_tx(saddr(full + j), stage_tx(nsp));
                        load_b(j, j, nsp, saddr(full + j));
                    }
                }
                __syncwarp();
                grid_dep_wait();
            }
            bool stop = false;
            for (int j = 0; j < NST; ++j, ++g) {
                const int s = g % C::kStages;
                if (g >= C::kStages &&
                    !warp_wait(saddr(empty + s), ((uint32_t)(g / C::kStages) & 1u) ^ 1u, abort, p)) {
                    stop = true;
                    break;
                }
                if (g != p.debug_skip_stage && elect_one()) {   // test hook: that stage never arrives
                    const int nsp = min(C::kSpans, KL - j * C::kSpans);
                    const uint32_t fb = saddr(full + s);
                    if (j >= pre)
                        mbar_arrive_tx(fb, stage_tx(nsp));
                    if (!PREQUANT) {   // A of the stage's spans in one 3-D box, their scale tiles in one copy
                        const int ks = ks0 + j * C::kSpans;
                        tma_3d(saddr(smem + s * C::kAB), &map_a, 0, (int)tm0, ks, fb);
                        bulk_g2s(saddr(smem + C::kOffSfa + s * C::kSpans * C::kSfaSpan),
                                 p.a_scale + ((int64_t)mt * (2 * KS) + 2 * ks) * 512, (uint32_t)(C::kSfaSpan * nsp), fb);
                    }
                    if (j >= pre)
                        load_b(j, s, nsp, fb);
                }
                __syncwarp();
                issued = g + 1;
            }
            if (stop)
                break;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        // warp-uniform loop, one elected lane issues the tensor-core work
        int g = 0;
        int mt, nt;
        bool any = false, stop = false;
        for (int ti = 0; !stop && tile_at(ti, mt, nt); ++ti) {
            // the accumulator is free once the epilogue has read the previous tile
            if (ti > 0) {
                if (!warp_wait(saddr(tmem_empty), (uint32_t)((ti - 1) & 1), abort, p))
                    break;
                tc_fence_after();
            }
            // a tile that starts half-way into a 128-row scale tile (64-row
            // tiles) reads its rows' scale columns from 2 on
            const uint32_t sfb_row_col = (BN == 64) ? (uint32_t)((((int64_t)nt * BN) >> 6 & 1) * 2) : 0u;
            for (int j = 0; j < NST; ++j, ++g) {
                const int s = g % C::kStages, nsp = min(C::kSpans, KL - j * C::kSpans);
                if (!warp_wait(saddr(full + s), (uint32_t)(g / C::kStages) & 1u, abort, p)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    for (int sp = 0; sp < nsp; ++sp) {
                        const uint32_t sfa_col = tmem_sf + s * C::kSfCols + sp * C::kSfColsSpan;
                        const uint32_t sfb_col = sfa_col + 8;
                        const uint32_t sfa_smem = saddr(smem + C::kOffSfa + (s * C::kSpans + sp) * C::kSfaSpan);
                        // B scales: tile t's spans after tile t - 1's
                        const uint32_t sfb_smem = saddr(smem + C::kOffSfb + (s * C::kSfbAtoms * C::kSpans + sp) * 1024);
                        // A's spans lie a_box_rows rows apart as loaded (128 when quantised here)
                        const uint32_t a_smem = saddr(smem + s * C::kAB + sp * a_pitch),
                                       b_smem = saddr(smem + s * C::kAB + C::kStageA + sp * C::kSpanB);
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            cp_sf(sfa_col + 4 * c, desc_sf(sfa_smem + c * 512));
#pragma unroll
                            for (int t = 0; t < C::kSfbAtoms; ++t)
                                cp_sf(sfb_col + 4 * C::kSfbAtoms * c + 4 * t,
                                      desc_sf(sfb_smem + t * C::kSpans * 1024 + c * 512));
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int c = k >> 1;
                            mma_mxf4(tmem, desc_sw128(a_smem + 32 * k), desc_sw128(b_smem + 32 * k),
                                     idesc_mxf4(BN, (k & 1) * 2), sfa_col + 4 * c,
                                     sfb_col + 4 * C::kSfbAtoms * c + sfb_row_col, (j | sp | k) != 0);
                        }
                    }
                    mma_commit(saddr(empty + s));
                }
                __syncwarp();
                any = true;
            }
            if (!stop && elect_one())
                mma_commit(saddr(accum));    // this tile's accumulator is complete
            __syncwarp();
        }
        if (*abort && any && elect_one()) {
            // drain the tensor core before the tensor memory is freed
            mma_commit(saddr(drain));
            const uint64_t t0 = gtimer();
            while (!mbar_test(saddr(drain), 0) && gtimer() - t0 < (uint64_t)p.wait_limit_ns) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int q = warp & 3;              // lane quarter of tensor memory this warp may access
        const int r = q * 32 + lane;         // row of the tile
        // prequant: warps 4-7 and 8-11 share the epilogue by column halves
        const int c_lo = (PREQUANT && warp >= 8) ? BN / 2 : 0;
        const int c_hi = (PREQUANT && warp < 8) ? BN / 2 : BN;
        bool ok = true;
        grid_dep_wait();    // before reading A (prequant) or writing D
        if (PREQUANT)
            ok = prequant_loop<BN>(p, m0, R, ks0, KL, smem, full, empty, abort);
        // ------------------------------------------------------- epilogue
        // plain GEMM: this warp's staging rows for the stores of D
        uint8_t *const stage_w = smem + C::kOffOut + (warp - 4) * (32 * C::kStoreCols * 2);
        int mt, nt;
        for (int ti = 0; ok && tile_at(ti, mt, nt); ++ti) {
            if (!warp_wait(saddr(accum), (uint32_t)(ti & 1), abort, p))
                break;
            tc_fence_after();
            const int64_t tm0 = (int64_t)mt * kBM, tn0 = (int64_t)nt * BN;
            const int64_t m = tm0 + r;
            const int tR = (int)min((int64_t)kBM, p.M - tm0);
            const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
            uint16_t *drow = p.d + m * p.ldd + tn0;
            // split-K: this CTA's partial sums go to its shared memory (the
            // operand ring is free now), padded rows against bank conflicts
            float *red = (float *)smem + r * (BN + 4);
            if (!PREQUANT && p.ksplit == 1) {
                // Stores of D, SC columns at a time: each lane holds its row's
                // SC * 2 bytes; they pass through shared memory (16-byte piece j
                // of row i at j ^ swz(i): no bank conflicts either way) so that
                // every store instruction writes whole pieces of 32 / V rows
                // (four 128-byte lines, or eight rows' 64 bytes) instead of 32
                // rows' 16 bytes.
                constexpr int SC = C::kStoreCols;   // 64 or 32
                constexpr int V = SC / 8;           // 16-byte pieces per staged row
                constexpr int RPI = 32 / V;         // rows per store instruction
                auto swz = [](int i) { return V == 8 ? (i & 7) : ((i >> 1) & 3); };
                const int64_t row0 = tm0 + q * 32;
                const int cj = lane % V;
#pragma unroll 1
                for (int c0 = 0; c0 < BN && row0 < p.M && tn0 + c0 < p.N; c0 += SC) {   // warp-uniform
                    uint32_t lo[32], hi[32];
                    tmem_ld32_issue(trow + c0, lo);
                    if (SC == 64)
                        tmem_ld32_issue(trow + c0 + 32, hi);
                    tmem_ld_wait();
                    tmem_hold(lo);
                    if (SC == 64)
                        tmem_hold(hi);
#pragma unroll
                    for (int j = 0; j < V; ++j) {
                        const uint32_t *a = j < 4 ? lo + 8 * j : hi + 8 * (j - 4);
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(a[0]), __uint_as_float(a[1]));
                        o.y = pack_bf16x2(__uint_as_float(a[2]), __uint_as_float(a[3]));
                        o.z = pack_bf16x2(__uint_as_float(a[4]), __uint_as_float(a[5]));
                        o.w = pack_bf16x2(__uint_as_float(a[6]), __uint_as_float(a[7]));
                        *reinterpret_cast<uint4 *>(stage_w + lane * (2 * SC) + ((j ^ swz(lane)) << 4)) = o;
                    }
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < V; ++it) {
                        const int rr = it * RPI + lane / V;
                        const uint4 v = *reinterpret_cast<const uint4 *>(stage_w + rr * (2 * SC) + ((cj ^ swz(rr)) << 4));
                        const int64_t gm = row0 + rr, gn = tn0 + c0 + cj * 8;
                        if (gm < p.M && gn < p.N && RMSQ_IN_BOUNDS(p.status, gn + 8 <= p.N))
                            *reinterpret_cast<uint4 *>(p.d + gm * p.ldd + gn) = v;
                    }
                    __syncwarp();                // the rows are read before they are overwritten
                }
            }
            // split K / prequant: 32-column chunks, two per wait for the
            // tensor-memory loads in the plain GEMM (the prequant kernel keeps
            // to one, which holds its registers at 128 a thread: its CTA then
            // fits on an SM beside a block of the norm kernel it follows)
            constexpr int kStep = PREQUANT ? 32 : 64;
#pragma unroll 1
            for (int c0 = c_lo; c0 < c_hi && (PREQUANT || p.ksplit > 1); c0 += kStep) {
                const bool two = kStep == 64 && c0 + 32 < c_hi;   // warp-uniform
                uint32_t acc2[2][32];
                tmem_ld32_issue(trow + c0, acc2[0]);
                if (two)
                    tmem_ld32_issue(trow + c0 + 32, acc2[1]);
                tmem_ld_wait();
                tmem_hold(acc2[0]);
                tmem_hold(acc2[1]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && !two)
                        continue;
                    const int cc = c0 + 32 * h;
                    const uint32_t(&acc)[32] = acc2[h];
                    if (p.ksplit > 1) {
                        if (r < tR) {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                *reinterpret_cast<float4 *>(red + cc + 4 * v) =
                                    make_float4(__uint_as_float(acc[4 * v]), __uint_as_float(acc[4 * v + 1]),
                                                __uint_as_float(acc[4 * v + 2]), __uint_as_float(acc[4 * v + 3]));
                        }
                        continue;
                    }
                    const int64_t valid = p.N - (tn0 + cc);
                    if (r >= tR)
                        continue;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (valid >= 8 * (v + 1)) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(acc[8 * v + 0]), __uint_as_float(acc[8 * v + 1]));
                            o.y = pack_bf16x2(__uint_as_float(acc[8 * v + 2]), __uint_as_float(acc[8 * v + 3]));
                            o.z = pack_bf16x2(__uint_as_float(acc[8 * v + 4]), __uint_as_float(acc[8 * v + 5]));
                            o.w = pack_bf16x2(__uint_as_float(acc[8 * v + 6]), __uint_as_float(acc[8 * v + 7]));
                            if (RMSQ_IN_BOUNDS(p.status, m < p.M && tn0 + cc + 8 * (v + 1) <= p.N))
                                *reinterpret_cast<uint4 *>(drow + cc + 8 * v) = o;
                        }
                    }
                }
            }
            // the accumulator may be overwritten by the next tile's MMAs
            tc_fence_before();
            mbar_arrive(saddr(tmem_empty));
        }
    }

    if (p.ksplit > 1) {
        // ------------------------------------------- split-K reduction
        // Every CTA of the cluster reaches both barriers, whatever happened
        // before (an aborted CTA contributes garbage and has set the status
        // word), so no CTA waits on one that left. CTA z sums a contiguous
        // share of the tile's (row, 4-column) units over the cluster's
        // partials in rank order 0, 1, ... (deterministic), then rounds to bf16.
        cluster_sync();
        grid_dep_wait();    // every thread of the CTA writes D here
        const int units = R * (BN / 4);
        const int u0 = (int)((int64_t)units * kz / p.ksplit), u1 = (int)((int64_t)units * (kz + 1) / p.ksplit);
        for (int u = u0 + (int)threadIdx.x; u < u1; u += (int)blockDim.x) {
            const int row = u / (BN / 4), c = (u - row * (BN / 4)) * 4;
            if (n0 + c >= p.N)
                continue;
            const float *src = (const float *)smem + row * (BN + 4) + c;
            // all ranks' loads in flight before the first add (rank order kept)
            float4 part[8];
#pragma unroll
            for (int z = 0; z < 8; ++z)
                if (z < p.ksplit)
                    part[z] = ld_peer_f4(src, (uint32_t)z);
            float4 acc = part[0];
#pragma unroll
            for (int z = 1; z < 8; ++z) {
                if (z < p.ksplit) {
                    acc.x += part[z].x;
                    acc.y += part[z].y;
                    acc.z += part[z].z;
                    acc.w += part[z].w;
                }
            }
            if (RMSQ_IN_BOUNDS(p.status, m0 + row < p.M && n0 + c + 4 <= p.N))
                *reinterpret_cast<uint2 *>(p.d + (m0 + row) * p.ldd + n0 + c) =
                    make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        }
        cluster_sync_exit();
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 0) {
        // every role has stopped, so the abort is final: let the copies this
        // CTA issued and nobody consumed land before it goes away (one
        // deadline for all of them)
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
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
    }
}

// ----------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    // looked up once; the initialisation of a function-local static is thread-safe
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return (EncodeTiledFn)f;
        return (EncodeTiledFn) nullptr;
    }();
    return fn;
}

// 2-D map over `rows` rows of `row_bytes` code bytes (leading dimension
// `ld` bytes), boxes of 128 bytes x box_rows rows, 128-byte swizzle; rows
// past the end read as zero codes.
bool make_code_map(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int64_t ld, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)kSpanBytes, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the codes seen as (128 bytes of a K span, row, span): rows ld
// bytes apart, spans 128 bytes apart, 128-byte swizzle; a box covers box_rows
// rows of box_spans spans and lands span after span, each span laid out as
// the 2-D box; rows and spans past the end read as zero codes.
bool make_code_map3(CUtensorMap *map, const void *base, int64_t rows, int64_t spans, int64_t ld, int box_rows,
                    int box_spans)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {(cuuint64_t)kSpanBytes, (cuuint64_t)rows, (cuuint64_t)spans};
    cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)kSpanBytes};
    cuuint32_t box[3] = {(cuuint32_t)kSpanBytes, (cuuint32_t)box_rows, (cuuint32_t)box_spans};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool PRE>
cudaError_t launch_gemm_t(const GemmParams &p, const CUtensorMap &ma, const CUtensorMap &mb, int m_tiles,
                          int n_tiles, int persistent_ctas, cudaStream_t st)
{
    using C = GemmCfg<BN, PRE>;
    static std::atomic<bool> attr[128];   // shared-memory limit raised on this device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (!attr[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(mxfp4_gemm_kernel<BN, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::kSmem);
        if (e != cudaSuccess)
            return e;
        attr[dev].store(true, std::memory_order_release);
    }
    // Launched as a programmatic dependent of the previous kernel in the
    // stream: the CTAs may start, set up and load B while that kernel (the
    // fused norm + quant) finishes; griddepcontrol.wait in the kernel holds
    // back every read of A and write of D until it has.
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(gemm_threads<PRE>(), 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (p.persistent) {     // one CTA per SM walks the tiles
        cfg.gridDim = dim3(persistent_ctas, 1, 1);
    } else if (p.ksplit == 1) {
        cfg.gridDim = dim3(n_tiles, m_tiles, 1);
    } else {
        // the CTAs that split one tile's K form a cluster (they exchange
        // partial sums through distributed shared memory)
        cfg.gridDim = dim3(n_tiles, m_tiles, p.ksplit);
        at[1].id = cudaLaunchAttributeClusterDimension;
        at[1].val.clusterDim.x = 1;
        at[1].val.clusterDim.y = 1;
        at[1].val.clusterDim.z = (unsigned)p.ksplit;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, mxfp4_gemm_kernel<BN, PRE>, p, ma, mb);
}

bool pre_of(const GemmLaunch &g) { return g.a_bf16 != nullptr; }

// K spans per ring stage of the one-CTA kernel (0 for a width it lacks)
int stage_spans(int bn, bool pre)
{
    switch (bn) {
    case 64: return pre ? GemmCfg<64, true>::kSpans : GemmCfg<64, false>::kSpans;
    case 128: return pre ? GemmCfg<128, true>::kSpans : GemmCfg<128, false>::kSpans;
    case 256: return pre ? GemmCfg<256, true>::kSpans : GemmCfg<256, false>::kSpans;
    }
    return 0;
}

// 2-D map over a scale-tile array viewed as rows of 256 bytes (one K span of
// a 128-row tile is four such rows, 1 KB); rows past the end read as zero.
bool make_scale_map(CUtensorMap *map, const void *base, int64_t rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {256, (cuuint64_t)rows};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, 4};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_mxfp4_gemm(const GemmLaunch &g, cudaStream_t st)
{
    if (g.pair)
        return pre_of(g) ? cudaErrorInvalidValue : launch_pair(g, st);
    GemmParams p{};
    p.a_scale = (const uint8_t *)g.a_scale;
    p.b_scale = (const uint8_t *)g.b_scale;
    p.a_bf16 = (const uint4 *)g.a_bf16;
    p.lda_v = g.a_bf16 ? g.lda / 8 : 0;
    p.d = (uint16_t *)g.d;
    p.ldd = g.ldd;
    p.M = g.M;
    p.N = g.N;
    p.k_spans = (int32_t)(g.K / kSpanK);
    p.b_row_tiles = (int32_t)((g.N + 127) / 128);
    // Rows of the A tile past M are never stored, so with fewer than 128
    // rows only those (rounded up to a swizzle atom of 8) are loaded. A 3-D
    // box lands its spans a_box_rows * 128 bytes apart; the MMA reads each
    // span there, and its rows past a_box_rows -- later bytes of the same
    // stage's A area, which its own copies have filled or an earlier stage
    // left -- feed only discarded rows of D.
    p.a_box_rows = g.M >= kBM ? kBM : (int32_t)((g.M + 7) / 8 * 8);
    p.ksplit = g.ksplit;
    p.debug_skip_stage = g.debug_skip_stage;
    p.persistent = g.persistent_ctas > 0;
    if (p.ksplit < 1 || p.ksplit > 8 || p.ksplit > p.k_spans)
        return cudaErrorInvalidValue;
    p.wait_limit_ns = g.wait_limit_ns;
    p.status = g.status;
    // 3-D boxes of a ring stage's spans (the stage's span count depends on the
    // tile width and the kernel)
    const int sps = stage_spans(g.bn, g.a_bf16 != nullptr);
    if (!sps)
        return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    if (!make_code_map3(&mb, g.b_q, g.N, p.k_spans, g.ldb, g.bn, sps))
        return cudaErrorInvalidValue;
    if (g.a_bf16) {
        ma = mb;   // unused by the prequant kernel
    } else if (!make_code_map3(&ma, g.a_q, g.M, p.k_spans, g.lda, p.a_box_rows, sps)) {
        return cudaErrorInvalidValue;
    }
    const int m_tiles = (int)((g.M + kBM - 1) / kBM), n_tiles = (int)((g.N + g.bn - 1) / g.bn);
    p.m_tiles = m_tiles;
    p.n_tiles = n_tiles;
    if (p.persistent && (pre_of(g) || p.ksplit != 1))
        return cudaErrorInvalidValue;
    const bool pre = g.a_bf16 != nullptr;
    switch (g.bn) {
    case 64: return pre ? launch_gemm_t<64, true>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st)
                        : launch_gemm_t<64, false>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st);
    case 128: return pre ? launch_gemm_t<128, true>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st)
                         : launch_gemm_t<128, false>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st);
    case 256: return pre ? launch_gemm_t<256, true>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st)
                         : launch_gemm_t<256, false>(p, ma, mb, m_tiles, n_tiles, g.persistent_ctas, st);
    }
    return cudaErrorInvalidValue;
}

bool tensor_map_encoder_available() { return encode_fn() != nullptr; }

namespace {

// --------------------------------------------------------- host checks

rmsq_status failf(rmsq_status s, const char *fmt, ...)
{
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    return set_error(s, msg);
}

struct Range {
    uintptr_t lo, hi;
};

Range mat_range(const void *p, int64_t M, int64_t H, int64_t ld, int64_t elem)
{
    uintptr_t lo = (uintptr_t)p;
    return Range{lo, lo + (uintptr_t)(((M - 1) * ld + H) * elem)};
}

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// ------------------------------------------------------------ consumer GEMM

__global__ void mx_scale_tiles_kernel(const uint8_t *s, int64_t ld, int64_t R, int64_t G, uint8_t *out,
                                      int64_t total, int64_t ktiles, uint8_t fill)
{
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
         o += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = o >> 9;
        const int w = (int)(o & 511);
        const int r = ((w & 15) >> 2) * 32 + (w >> 4), c = w & 3;   // inverse of (r%32)*16 + (r/32)*4 + c
        const int64_t row = (tile / ktiles) * 128 + r, g = (tile % ktiles) * 4 + c;
        out[o] = (row < R && g < G) ? s[row * ld + g] : fill;
    }
}

const rmsq_gemm_opts kDefaultGemmOpts = {0, 0, 0, 0, 0};

// Option and shape checks shared by the GEMM entry points and the plan query.
rmsq_status check_gemm_args(int64_t M, int64_t N, int64_t K, const rmsq_gemm_opts &o)
{
    if (M < 0 || N < 0 || K <= 0)
        return set_error(RMSQ_ERR_INVALID_ARG, "need M >= 0, N >= 0, K > 0");
    if (o.bn != 0 && o.bn != 64 && o.bn != 128 && o.bn != 192 && o.bn != 256)
        return failf(RMSQ_ERR_INVALID_ARG, "bn must be 0, 64, 128, 192 or 256 (got %d)", o.bn);
    if (o.bn == 192 && o.schedule != 3)
        return failf(RMSQ_ERR_UNSUPPORTED, "bn 192 is a width of the CTA-pair schedule only");
    if (o.ksplit < 0 || o.ksplit > 8)
        return failf(RMSQ_ERR_INVALID_ARG, "ksplit must be 0..8 (got %d)", o.ksplit);
    if (o.wait_limit_ns < 0)
        return failf(RMSQ_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
    if (o.debug_stall_stage < 0)
        return failf(RMSQ_ERR_INVALID_ARG, "debug_stall_stage must be >= 0");
    if (o.schedule < 0 || o.schedule > 3)
        return failf(RMSQ_ERR_INVALID_ARG, "schedule must be 0, 1, 2 or 3 (got %d)", o.schedule);
    if (K % 256)
        return failf(RMSQ_ERR_UNSUPPORTED, "K=%lld is not a multiple of 256", (long long)K);
    if (N % 8)
        return failf(RMSQ_ERR_UNSUPPORTED, "N=%lld is not a multiple of 8", (long long)N);
    return RMSQ_OK;
}

// What one GEMM launches: B-tile width, K split (CTAs of a cluster per
// tile), CTA pairs or not, and the persistent grid's size (0: one CTA, or
// one cluster, per tile).
struct GemmPlan {
    int bn, ksplit;
    bool pair;
    int persistent_ctas;
};

// The launch for a shape (M, N > 0; arguments already checked) on a device
// with `sms` SMs. pair_caps(w) gives how many CTA pairs of width w fit on the
// device at once; it is asked only when the library picks the pair width,
// and a non-positive answer fails with caps_status.
template <class PairCaps>
rmsq_status plan_gemm(bool prequant, int64_t M, int64_t N, int64_t K, const rmsq_gemm_opts &o, int sms,
                      PairCaps &&pair_caps, rmsq_status caps_status, GemmPlan &plan)
{
    const int64_t m_tiles = (M + 127) / 128;
    // Tile width, from measurements on GB300 (N = 2112, K = 7168). The
    // prequant kernel quantises A once per B tile, so it mostly takes the
    // widest tile, except: up to 16 tokens, 64-row tiles (K split 4; 8.4
    // against 8.7 us at 4 tokens), where quantising is nearly free and the
    // CTAs load less of B; and with two row tiles of A, 128-row tiles (K
    // split 4: 37.8 against 52.4 us at 256 tokens), because 18 clusters of
    // 8 CTAs do not all fit on the GPU at once and the last ones run in a
    // second wave. The plain GEMM takes 256-row B tiles once they give at
    // least half the SMs a tile, 128 from two row tiles of A on, and 64 for
    // a single row tile (decode). With fewer tiles than SMs, K is split over
    // a cluster of up to 8 CTAs (each at least one 256-element span of K).
    int bn = o.bn;
    if (o.schedule == 3) {
        if (prequant || (bn && bn != 256 && bn != 192) || (o.ksplit && o.ksplit != 1))
            return failf(RMSQ_ERR_UNSUPPORTED,
                         "the CTA-pair schedule needs quantised A, bn 192 or 256 and no K split");
        if (!bn)
            bn = 256;
    }
    if (!bn) {
        if (prequant)
            bn = m_tiles == 2 ? 128 : (M <= 16 ? 64 : 256);
        else if (m_tiles * ((N + 255) / 256) * 2 >= sms)
            bn = 256;
        else
            bn = m_tiles >= 2 ? 128 : 64;
    }
    const int64_t tiles = m_tiles * ((N + bn - 1) / bn);
    int ksplit = o.schedule == 3 ? 1 : o.ksplit;
    if (!ksplit) {
        int64_t k = tiles >= sms ? 1 : sms / tiles;
        if (k > 8)
            k = 8;
        if (k > K / 256)
            k = K / 256;
        ksplit = (int)(k < 1 ? 1 : k);
    }
    if (ksplit > K / 256)
        return failf(RMSQ_ERR_INVALID_ARG, "ksplit=%d exceeds the %lld 256-element spans of K", ksplit,
                     (long long)(K / 256));
    // More tiles than SMs (no K split, A quantised): one persistent CTA per
    // SM walks the tiles, so set-up, the ring's first fill and the epilogue
    // overlap the neighbouring tiles' work.
    // 256-row tiles without a K split (the widest tiles already fill the
    // SMs): CTA pairs with 256 x 256 tiles, the fastest form measured from
    // 2048 tokens on (N = 2112, K = 7168).
    bool persistent = !prequant && ksplit == 1 && tiles > sms;
    bool pair = o.schedule == 3 || (o.schedule == 0 && !prequant && ksplit == 1 && bn == 256);
    if (o.schedule == 1 || pair)
        persistent = false;
    if (pair && !o.bn) {
        // Pair tile width: the one whose busiest pair does the least work,
        // counting a 192-wide tile as 0.75 of a 256-wide one and charging it
        // 15 % for its lower efficiency per column (measured at N = 2112,
        // K = 7168, 8192 tokens: 51.6 against 44.8 ns per column and pair).
        const int cap256 = pair_caps(256), cap192 = pair_caps(192);
        if (cap256 <= 0 || cap192 <= 0)
            return failf(caps_status,
                         "CTA-pair capacity unavailable (cluster occupancy query failed or not given)");
        const int64_t mt2 = (M + 255) / 256;
        const int64_t w256 = (mt2 * ((N + 255) / 256) + cap256 - 1) / cap256 * 256;
        const int64_t w192 = (mt2 * ((N + 191) / 192) + cap192 - 1) / cap192 * 192;
        bn = w192 * 115 < w256 * 100 ? 192 : 256;
    }
    else if (o.schedule == 2) {
        if (prequant || ksplit != 1)
            return failf(RMSQ_ERR_UNSUPPORTED, "the persistent schedule needs quantised A and no K split");
        persistent = true;
    }
    plan.bn = bn;
    plan.ksplit = ksplit;
    plan.pair = pair;
    plan.persistent_ctas = persistent ? (int)(tiles < sms ? tiles : sms) : 0;
    return RMSQ_OK;
}

// Shared by both placements: a_q / ld_a (bytes) for MXFP4 A, a / ld_a
// (elements) for bf16 A.
rmsq_status gemm_common(bool prequant, const void *a, int64_t ld_a, const void *a_scale, const void *b_q,
                        int64_t ld_b, const void *b_scale, void *d, int64_t ld_d, int64_t M, int64_t N,
                        int64_t K, void *stream, const rmsq_gemm_opts *opts)
{
    const rmsq_gemm_opts o = opts ? *opts : kDefaultGemmOpts;
    const rmsq_status cs = check_gemm_args(M, N, K, o);
    if (cs != RMSQ_OK)
        return cs;
    if (M == 0 || N == 0)
        return clear_error();
    if (!a || !b_q || !b_scale || !d || (!prequant && !a_scale))
        return failf(RMSQ_ERR_INVALID_ARG, "operand, scale and output pointers are required");
    const int64_t a_row_bytes = prequant ? K * 2 : K / 2;
    const int64_t lda_bytes = prequant ? ld_a * 2 : ld_a;
    if (lda_bytes < a_row_bytes || ld_b < K / 2 || ld_d < N)
        return failf(RMSQ_ERR_INVALID_ARG, "leading dimensions must cover a row");
    if (!aligned(a, 16) || !aligned(b_q, 16) || !aligned(b_scale, 16) || !aligned(d, 16) ||
        (!prequant && !aligned(a_scale, 16)) || lda_bytes % 16 || ld_b % 16 || ld_d % 8)
        return failf(RMSQ_ERR_MISALIGNED,
                    "operands, scale tiles and D need 16-byte aligned bases and 16-byte row pitches");
    const int64_t m_tiles = (M + 127) / 128;
    if (m_tiles > 65535)
        return failf(RMSQ_ERR_UNSUPPORTED, "M=%lld exceeds %d rows", (long long)M, 65535 * 128);
    const int64_t tile_bytes = (K / 128) * 512;
    Range rd = mat_range(d, M, N, ld_d, 2);
    Range ins[4] = {mat_range(a, M, a_row_bytes, lda_bytes, 1), mat_range(b_q, N, K / 2, ld_b, 1),
                    mat_range(b_scale, 1, (N + 127) / 128 * tile_bytes, 0, 1), {0, 0}};
    if (!prequant)
        ins[3] = mat_range(a_scale, 1, m_tiles * tile_bytes, 0, 1);
    for (const Range &r : ins)
        if (r.hi > r.lo && overlaps(rd, r))
            return failf(RMSQ_ERR_INVALID_ARG, "D overlaps an input");
    if (!tensor_map_encoder_available())
        return failf(RMSQ_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return failf(RMSQ_ERR_CUDA, "no current device");
    unsigned int *status = device_status_word(dev);
    if (!status)
        return failf(RMSQ_ERR_CUDA, "status word address unavailable");
    const int sms = device_sm_count();
    if (sms <= 0)
        return failf(RMSQ_ERR_CUDA, "SM count query failed");
    GemmPlan plan{};
    const rmsq_status ps = plan_gemm(
        prequant, M, N, K, o, sms, [dev](int w) { return pair_capacity(dev, w); }, RMSQ_ERR_CUDA, plan);
    if (ps != RMSQ_OK)
        return ps;
    GemmLaunch g{};
    if (prequant) {
        g.a_bf16 = a;
    } else {
        g.a_q = a;
        g.a_scale = a_scale;
    }
    g.lda = ld_a;
    g.b_q = b_q;
    g.b_scale = b_scale;
    g.ldb = ld_b;
    g.d = d;
    g.ldd = ld_d;
    g.M = M;
    g.N = N;
    g.K = K;
    g.bn = plan.bn;
    g.ksplit = plan.ksplit;
    g.persistent_ctas = plan.persistent_ctas;
    g.pair = plan.pair;
    g.debug_skip_stage = o.debug_stall_stage - 1;   // -1: off
    g.wait_limit_ns = o.wait_limit_ns > 0 ? o.wait_limit_ns : 2000000000LL;
    g.status = status;
    cudaError_t e = launch_mxfp4_gemm(g, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return failf(RMSQ_ERR_CUDA, "GEMM launch failed: %s", cudaGetErrorString(e));
    return clear_error();
}

}  // namespace
}  // namespace gemm
}  // namespace rmsq

using namespace rmsq;
using namespace rmsq::gemm;

extern "C" {

rmsq_status rmsq_mxfp4_gemm_ex(
    const void *a_q, int64_t ld_a, const void *a_scale_tiles, const void *b_q, int64_t ld_b,
    const void *b_scale_tiles, void *d, int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream,
    const rmsq_gemm_opts *opts)
{
    return gemm_common(false, a_q, ld_a, a_scale_tiles, b_q, ld_b, b_scale_tiles, d, ld_d, M, N, K, stream,
                       opts);
}

rmsq_status rmsq_mxfp4_gemm(
    const void *a_q, int64_t ld_a, const void *a_scale_tiles, const void *b_q, int64_t ld_b,
    const void *b_scale_tiles, void *d, int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream)
{
    return gemm_common(false, a_q, ld_a, a_scale_tiles, b_q, ld_b, b_scale_tiles, d, ld_d, M, N, K, stream,
                       nullptr);
}

rmsq_status rmsq_a16wfp4_gemm_ex(
    const void *a, int64_t ld_a, const void *b_q, int64_t ld_b, const void *b_scale_tiles, void *d,
    int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream, const rmsq_gemm_opts *opts)
{
    return gemm_common(true, a, ld_a, nullptr, b_q, ld_b, b_scale_tiles, d, ld_d, M, N, K, stream, opts);
}

rmsq_status rmsq_a16wfp4_gemm(
    const void *a, int64_t ld_a, const void *b_q, int64_t ld_b, const void *b_scale_tiles, void *d,
    int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream)
{
    return gemm_common(true, a, ld_a, nullptr, b_q, ld_b, b_scale_tiles, d, ld_d, M, N, K, stream, nullptr);
}

rmsq_status rmsq_gemm_plan_for(int32_t prequant, int64_t M, int64_t N, int64_t K, const rmsq_gemm_opts *opts,
                               int32_t sms, int32_t pairs_256, int32_t pairs_192, rmsq_gemm_plan *plan)
{
    if (!plan)
        return failf(RMSQ_ERR_INVALID_ARG, "plan is required");
    *plan = rmsq_gemm_plan{0, 0, 0, 0};
    const rmsq_gemm_opts o = opts ? *opts : kDefaultGemmOpts;
    const rmsq_status cs = check_gemm_args(M, N, K, o);
    if (cs != RMSQ_OK)
        return cs;
    if (sms <= 0)
        return failf(RMSQ_ERR_INVALID_ARG, "sms must be > 0 (got %d)", sms);
    if (M == 0 || N == 0)
        return clear_error();
    if ((M + 127) / 128 > 65535)
        return failf(RMSQ_ERR_UNSUPPORTED, "M=%lld exceeds %d rows", (long long)M, 65535 * 128);
    GemmPlan p{};
    const rmsq_status ps = plan_gemm(
        prequant != 0, M, N, K, o, sms, [=](int w) { return w == 192 ? pairs_192 : pairs_256; },
        RMSQ_ERR_INVALID_ARG, p);
    if (ps != RMSQ_OK)
        return ps;
    plan->bn = p.bn;
    plan->ksplit = p.ksplit;
    plan->schedule = p.pair ? 3 : (p.persistent_ctas > 0 ? 2 : 1);
    plan->persistent_ctas = p.persistent_ctas;
    return clear_error();
}

rmsq_status rmsq_mx_scale_tiles(const uint8_t *scale, int64_t ld, int64_t R, int64_t G, uint8_t *out,
                                uint8_t fill, void *stream)
{
    if (R < 0 || G <= 0 || ld < G)
        return failf(RMSQ_ERR_INVALID_ARG, "need R >= 0, G > 0, ld >= G");
    if (R == 0)
        return clear_error();
    if (!scale || !out)
        return failf(RMSQ_ERR_INVALID_ARG, "scale and out are required");
    const int64_t ktiles = (G + 3) / 4, total = (R + 127) / 128 * ktiles * 512;
    if (overlaps(mat_range(out, 1, total, 0, 1), mat_range(scale, R, G, ld, 1)))
        return failf(RMSQ_ERR_INVALID_ARG, "out overlaps scale");
    int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    mx_scale_tiles_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(scale, ld, R, G, out, total, ktiles, fill);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? clear_error() : failf(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
}

}  // extern "C"
