// Shared by the block-scaled MXFP4 GEMM kernels (rmsq_gemm.cu: one CTA per
// tile, K split over a cluster, prequant; rmsq_gemm_pair.cu: CTA pairs on
// cta_group::2): the launch record, the kernel parameters, the PTX wrappers
// (mbarrier, TMA, tcgen05) and the host helpers both launch paths use.
#pragma once

#include <cuda.h>
#include <atomic>
#include <cstdarg>
#include <cstdio>

#include "rmsq.h"
#include "rmsq_device.cuh"
#include "rmsq_internal.h"

namespace rmsq {
namespace gemm {


// One GEMM launch as the host checks leave it. A is either MXFP4 codes +
// tiled scales (a_q, a_scale; lda in bytes) or bf16 (a_bf16; lda in
// elements, quantised in the kernel).
struct GemmLaunch {
    const void *a_q, *a_scale, *a_bf16;
    int64_t lda;
    const void *b_q, *b_scale;
    int64_t ldb;               // bytes
    void *d;
    int64_t ldd;               // elements
    int64_t M, N, K;
    int bn;                    // 64, 128 or 256
    int ksplit;                // 1..8 CTAs (a cluster) per tile splitting K
    int persistent_ctas;       // > 0: a persistent grid of this many CTAs walks the tiles
    bool pair;                 // 256 x 256 tiles on CTA pairs (persistent, bn 256, quantised A)
    int debug_skip_stage;      // test hook: a ring stage (counted over the CTA's tiles) whose loads
                               // are never issued (-1 = off; a zero-initialised GemmLaunch must set it)
    int64_t wait_limit_ns;
    unsigned int *status;
};

constexpr int kBM = 128;          // MMA M: rows of A per tile
constexpr int kSpanBytes = 128;   // bytes of one operand row per span (256 E2M1)
constexpr int kSpanK = 256;       // K elements per span
// 8 warps; the prequant kernel has 4 more, so that 8 warps quantise A
template <bool PREQUANT>
constexpr int gemm_threads() { return PREQUANT ? 384 : 256; }
constexpr int kQuantThreads = 256;   // warps 4-11 of the prequant kernel

constexpr int pow2_at_least(int v)
{
    int p = 32;
    while (p < v)
        p <<= 1;
    return p;
}

struct GemmParams {
    const uint8_t *a_scale;     // MMA tile layout, ceil(M/128) x K/128 tiles of 512 bytes
    const uint8_t *b_scale;     // same for B
    const uint4 *a_bf16;        // prequant: bf16 rows, 16-byte vectors
    int64_t lda_v;              // prequant: leading dimension in vectors
    uint16_t *d;                // bf16 [M, ldd]
    int64_t ldd;
    int64_t M, N;
    int32_t k_spans;            // K / 256: spans of K (a ring stage holds one or more)
    int32_t b_row_tiles;        // ceil(N / 128): 128-row scale tiles that exist for B
    int32_t a_box_rows;         // rows of A per TMA box (128; rows past M read as zero)
    int32_t ksplit;             // CTAs of a cluster that split K (1 = no split)
    int32_t persistent;         // 1: a grid of gridDim.x CTAs walks the m_tiles x n_tiles tiles
    int32_t m_tiles, n_tiles;   // tiles of the launch (the pair kernel: 256-row tiles of A and B)
    int32_t debug_skip_stage;   // test hook: this ring stage (counted over the CTA's tiles) is never loaded (-1 = off)
    int64_t wait_limit_ns;
    unsigned int *status;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity. Returns false
// (after raising the CTA's abort flag and the status word) if it ran out, or
// if another role of the CTA already aborted.
// The clock and the abort flag are looked at only every 64 polls: reading
// %globaltimer on every poll made the waiting thread notice a completed
// phase hundreds of nanoseconds late (measured on GB300).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          const GemmParams &p)
{
    if (mbar_test(bar, parity))
        return true;
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_test(bar, parity))
            return true;
        if ((n & 63) == 0) {
            if (*abort)
                return false;
            const uint64_t t = gtimer();
            if (!t0) {
                t0 = t;
            } else if (t - t0 > (uint64_t)p.wait_limit_ns) {
                *abort = 1;
                atomicOr(p.status, 2u);
                return false;
            }
        }
    }
}

// The same wait taken by lane 0 for the whole warp (warp-uniform result, so
// that the .sync.aligned tensor-memory instructions after it see all lanes).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          const GemmParams &p)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0)
        ok = mbar_wait(bar, parity, abort, p) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// One lane of the (fully active) warp, chosen by the hardware.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// A 3-D box (coordinates x, y, z innermost first) whose bytes count on `bar`.
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Descriptor of a 32-row x 16-byte scale tile (no swizzle, 8-row core
// matrices 128 bytes apart) for tcgen05.cp.
__device__ __forceinline__ uint64_t desc_sf(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::mxf4 (E2M1 x E2M1, UE8M0 scales, fp32
// accumulator, both operands K-major; M = 128, or 256 for a CTA pair).
__host__ __device__ constexpr uint32_t idesc_mxf4(int n, int sf_id, int m = kBM)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(m >> 4) << 24) |
           ((uint32_t)sf_id << 29) | ((uint32_t)sf_id << 4);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void cp_sf(uint32_t taddr, uint64_t desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// ---- the same for a CTA pair (cta_group::2), issued by the even CTA. Measured
// with a self-checking probe on GB300: the MMA reads A rows 128r.. and B rows
// (N/2)r.. from CTA r's shared memory at the same offsets, and each CTA's
// tensor memory holds D for its 128 rows, the scale factors of its rows of A
// and those of ALL N rows of B; tcgen05.cp copies each CTA's own shared memory
// into its own tensor memory; the commit can arrive on both CTAs' barriers.
__device__ __forceinline__ void mma_mxf4_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                              uint32_t sfb, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void cp_sf_pair(uint32_t taddr, uint64_t desc)
{
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// arrives on the barrier at this offset in every CTA of `mask`
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     bar),
                 "h"(mask)
                 : "memory");
}

// TMA load into this CTA's shared memory whose completion counts on a
// barrier of either CTA of the pair (a cluster address)
__device__ __forceinline__ void tma_2d_pair(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Relaxed arrival on a barrier of either CTA of the pair. The epilogue uses it
// to hand the accumulator back: the only ordering needed is that its
// tensor-memory loads are complete, which tcgen05.wait::ld has established
// before the arrival is issued. (A cluster-scope release here would also wait
// for the warp's outstanding stores of D.)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of fp32 from tensor memory (issue only; the values
// are valid after tmem_ld_wait + tmem_hold).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties the registers of a tensor-memory load to a point after the wait, so
// that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_hold(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    tmem_ld32_issue(taddr, r);
    tmem_ld_wait();
    tmem_hold(r);
}

// ------------------------------------------- programmatic dependent launch

// A GEMM launched as a programmatic dependent of the kernel before it in the
// stream (the fused norm + quant) may start while that kernel still runs:
// every thread waits here before its first read of memory the previous
// kernel writes (A) and before its first write of D. Without the launch
// attribute the previous kernel has finished and the wait returns at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------- cluster (split K)

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The split-K cluster's last barrier, before its CTAs leave: each CTA's reads
// of the others' shared memory have returned (their values were used) before
// it arrives, so a relaxed arrival suffices -- measured 2.5-4 % faster than a
// release at 4-512 tokens.
__device__ __forceinline__ void cluster_sync_exit()
{
    asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}

__device__ __forceinline__ float4 ld_peer_f4(const float *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr(local)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote)
                 : "memory");
    return v;
}

// ------------------------------------------------------- host (shared)

// 2-D map over `rows` rows of `row_bytes` code bytes (leading dimension `ld`
// bytes), boxes of 128 bytes x box_rows rows, 128-byte swizzle.
bool make_code_map(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int64_t ld, int box_rows);
// 3-D map over the same codes seen as (128 bytes of a K span, row, span):
// rows ld bytes apart, spans 128 bytes apart; a box of box_rows rows and
// box_spans spans lands span after span, each span laid out as the 2-D box.
bool make_code_map3(CUtensorMap *map, const void *base, int64_t rows, int64_t spans, int64_t ld, int box_rows,
                    int box_spans);
// 2-D map over a scale-tile array viewed as rows of 256 bytes.
bool make_scale_map(CUtensorMap *map, const void *base, int64_t rows);
// CTA-pair kernel (rmsq_gemm_pair.cu): pairs resident at once for tile width
// bn (192 or 256; 0 if the query failed), and the launch.
int pair_capacity(int dev, int bn);
cudaError_t launch_pair(const GemmLaunch &g, cudaStream_t st);

}  // namespace gemm
}  // namespace rmsq
