// Register-resident row kernels: each team loads its row of x (and residual)
// straight into registers with 16-byte streaming loads, adds, writes the
// residual back, and finishes the row (rmsq_rows.cuh).
//   rows_kernel<VPT, TPR, MX, LAT>  one tensor; LAT > 0: the latency form for
//                                   launches of at most one block per SM
//                                   (gamma loaded with the row, one barrier),
//                                   each row's outputs shared by LAT blocks
//   dual_kernel<V0, T0, V1, T1, MX> two tensors (the MLA q_a / kv_a pair),
//                                   blocks [0, seg[0].blocks) on the first
// TPR / T0 / T1 = 0 means the team size is read at run time.
//
// Every one of them is launched as a programmatic dependent of the previous
// kernel in its stream (launch_pdl): its blocks may be scheduled while that
// kernel finishes, and griddepcontrol.wait holds them back, before their first
// access to global memory, until it has completed and its writes are visible.
// Only after that wait does a block let the grid's own dependents (a following
// GEMM or norm) launch: a trigger before the wait lets a chain of calls pile up
// waiting blocks on the SMs (64-token decode measured 2.49 -> 4.57 us per call
// that way, against 2.31 us with the trigger after the wait).
#pragma once

#include <atomic>

#include "rmsq_rows.cuh"

namespace rmsq {

// LAT = 0: the throughput form; LAT = 1, 2, 4: the latency form with the
// outputs of each row shared by LAT blocks (block b: row b / LAT, part
// b % LAT; one team per block).
template <int VPT, int TPR, bool MX, int LAT = 0>
__device__ __forceinline__ void block_rows(const Seg &s, int b, RedSmem &red)
{
    constexpr int SPLIT = LAT > 1 ? LAT : 1;
    const int tpr = TPR ? TPR : s.tpr;
    const int team = threadIdx.x / tpr;
    if (team >= s.rpb)
        return;                                   // idle team of a shared-size block
    const int t = threadIdx.x - team * tpr;
    const int64_t row = SPLIT > 1 ? (int64_t)(b / SPLIT) : (int64_t)b * s.rpb + team;
    const int part = SPLIT > 1 ? b % SPLIT : 0;
    if (row >= s.M)
        return;                                   // whole teams leave together
    if (s.prefetch_rows && t == 0) {
        // Keep HBM busy while the resident blocks are in their reduction and
        // quantise phases: pull the x / residual rows of a later block into L2
        // with one 1-D bulk prefetch each.
        const int64_t pr = row + s.prefetch_rows;
        if (pr < s.M) {
            const uint32_t bytes = (uint32_t)s.H * 2;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s.x + pr * s.ldx_v), "r"(bytes)
                         : "memory");
            if (s.res)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s.res + pr * s.ldres_v),
                             "r"(bytes)
                             : "memory");
        }
    }
    row_from_global<VPT, TPR, MX, (LAT > 0), SPLIT>(s, row, t, team, 0, red, part);
}

// Start of every row and pair kernel: wait for the kernel this one depends on
// (a no-op when launched without the programmatic attribute), then allow the
// next kernel in the stream to be scheduled; it waits in turn for this grid's
// completion before it reads or overwrites what this grid touches.
__device__ __forceinline__ void grid_dep_sync()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

// Launch a row or pair kernel as a programmatic dependent of the previous
// kernel in the stream (static shared memory only).
template <typename Kernel>
cudaError_t launch_pdl(Kernel k, int grid, int threads, cudaStream_t st, const LaunchParams &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
}

template <int VPT, int TPR, bool MX, int LAT>
__global__ void __launch_bounds__(kMaxThreads) rows_kernel(const __grid_constant__ LaunchParams p)
{
    __shared__ RedSmem red;
    grid_dep_sync();
    block_rows<VPT, TPR, MX, LAT>(p.seg[0], blockIdx.x, red);
}

template <int V0, int T0, int V1, int T1, bool MX>
__global__ void __launch_bounds__(kMaxThreads, 2) dual_kernel(const __grid_constant__ LaunchParams p)
{
    __shared__ RedSmem red;
    grid_dep_sync();
    if ((int)blockIdx.x < p.seg[0].blocks)
        block_rows<V0, T0, MX>(p.seg[0], blockIdx.x, red);
    else
        block_rows<V1, T1, MX>(p.seg[1], blockIdx.x - p.seg[0].blocks, red);
}

// The latency form of the pair, for launches of at most one block per SM
// (decode sizes): gamma is loaded with each row; with so few blocks the
// registers need no cap for occupancy.
template <int V0, int T0, int V1, int T1, bool MX>
__global__ void __launch_bounds__(kMaxThreads, 1) dual_kernel_lat(const __grid_constant__ LaunchParams p)
{
    __shared__ RedSmem red;
    grid_dep_sync();
    if ((int)blockIdx.x < p.seg[0].blocks)
        block_rows<V0, T0, MX, 1>(p.seg[0], blockIdx.x, red);
    else
        block_rows<V1, T1, MX, 1>(p.seg[1], blockIdx.x - p.seg[0].blocks, red);
}

// Team shapes compiled with a fixed team size: exact fits of common hidden
// sizes (vectors per thread x threads x 8 = H).
#define RMSQ_STATIC_SHAPES(X) \
    X(4, 224) /* H = 7168 */  \
    X(4, 256) /* H = 8192 */  \
    X(4, 160) /* H = 5120 */  \
    X(4, 128) /* H = 4096 */  \
    X(4, 64)  /* H = 2048 */  \
    X(3, 64)  /* H = 1536 */  \
    X(4, 16)  /* H = 512  */  \
    X(2, 16)  /* H = 256  */

// The latency form: at most one block per SM, typically followed by a GEMM
// launched as its programmatic dependent. The SMs its blocks occupy are asked
// for the largest shared-memory carveout, so that the GEMM's CTAs (about
// 220 KB of shared memory each) can start beside them instead of waiting for
// the blocks to leave: an SM's carveout is set when an idle SM takes a block
// and cannot grow while the block runs.
template <int V, int T, bool MX, int LAT>
cudaError_t launch_latency(const LaunchParams &p, int grid, int threads, cudaStream_t st)
{
    static std::atomic<uint64_t> carved{0};   // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 64 && !((carved.load(std::memory_order_acquire) >> dev) & 1u)) {
        e = cudaFuncSetAttribute(rows_kernel<V, T, MX, LAT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        carved.fetch_or(1ull << dev, std::memory_order_acq_rel);
    }
    return launch_pdl(rows_kernel<V, T, MX, LAT>, grid, threads, st, p);
}

// One compiled team shape in the throughput form (lat 0) or the latency form
// with each row's outputs shared by lat = 1, 2 or 4 blocks (a split that
// divides V).
template <int V, int T, bool MX>
cudaError_t launch_static(int lat, const LaunchParams &p, int grid, int threads, cudaStream_t st)
{
    if (lat == 0)
        return launch_pdl(rows_kernel<V, T, MX, 0>, grid, threads, st, p);
    if (lat == 1)
        return launch_latency<V, T, MX, 1>(p, grid, threads, st);
    if constexpr (V % 2 == 0) {
        if (lat == 2)
            return launch_latency<V, T, MX, 2>(p, grid, threads, st);
    }
    if constexpr (V % 4 == 0) {
        if (lat == 4)
            return launch_latency<V, T, MX, 4>(p, grid, threads, st);
    }
    return cudaErrorInvalidValue;
}

// The latency form exists for the compiled team shapes only; `lat` (0 =
// throughput form, else the latency form's split) is ignored for runtime
// team sizes.
template <bool MX>
cudaError_t launch_rows_impl(int vpt, int tpr_static, int lat, const LaunchParams &p, int grid,
                             int threads, cudaStream_t st)
{
    if (tpr_static) {
#define RMSQ_LAUNCH_STATIC(V, T)                                                \
        if (vpt == V && tpr_static == T)                                        \
            return launch_static<V, T, MX>(lat, p, grid, threads, st);
        RMSQ_STATIC_SHAPES(RMSQ_LAUNCH_STATIC)
#undef RMSQ_LAUNCH_STATIC
        return cudaErrorInvalidValue;
    }
    switch (vpt) {
    case 1: return launch_pdl(rows_kernel<1, 0, MX, 0>, grid, threads, st, p);
    case 2: return launch_pdl(rows_kernel<2, 0, MX, 0>, grid, threads, st, p);
    case 3: return launch_pdl(rows_kernel<3, 0, MX, 0>, grid, threads, st, p);
    case 4: return launch_pdl(rows_kernel<4, 0, MX, 0>, grid, threads, st, p);
    case 5: return launch_pdl(rows_kernel<5, 0, MX, 0>, grid, threads, st, p);
    case 6: return launch_pdl(rows_kernel<6, 0, MX, 0>, grid, threads, st, p);
    case 7: return launch_pdl(rows_kernel<7, 0, MX, 0>, grid, threads, st, p);
    case 8: return launch_pdl(rows_kernel<8, 0, MX, 0>, grid, threads, st, p);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rmsq
