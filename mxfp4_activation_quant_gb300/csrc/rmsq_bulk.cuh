// Persistent bulk-copy kernel: a grid of resident blocks, each looping over
// rows blockIdx.x, blockIdx.x + gridDim.x, ... . One block is one team. The
// x (and residual) row of the next NSTAGE rows is copied global -> shared
// memory by one thread with 1-D bulk copies (cp.async.bulk, completion
// counted in bytes on an mbarrier), so the loads of later rows are in flight
// while the current row is finished from registers. gamma is staged once
// per block.
//
// Every mbarrier wait is bounded by wait_limit_ns of %globaltimer. When a
// wait runs out the block agrees on it (barrier vote), sets the status word,
// waits (again bounded) for its other copies still in flight, and returns;
// rmsq_sync_status reports RMSQ_ERR_TIMEOUT. debug_skip_row makes one row's
// copy never be issued, which is how the tests exercise that path.
#pragma once

#include "rmsq_rows.cuh"

namespace rmsq {

constexpr int kStages = 2;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase with the given parity; false when it ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if ((int64_t)(global_timer_ns() - t0) > limit_ns)
            return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Dynamic shared memory: [gamma H*2][stage 0: x H*2 | res H*2][stage 1 ...]
// [NSTAGE mbarriers][NSTAGE issued flags]
__host__ __device__ inline size_t bulk_smem_bytes(int H, bool has_res)
{
    size_t row = (size_t)H * 2;
    size_t stage = row * (has_res ? 2 : 1);
    return row + stage * kStages + kStages * sizeof(uint64_t) + kStages * sizeof(int) + 16;
}

template <int VPT, int TPR, bool MX>
__global__ void __launch_bounds__(kMaxThreads) bulk_kernel(const __grid_constant__ BulkParams p)
{
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ RedSmem red;
    constexpr bool GUARD = TPR == 0;
    const Seg &s = p.s;
    const int tpr = TPR ? TPR : s.tpr;   // == blockDim.x
    const int t = threadIdx.x;
    const int nvec = s.H >> 3;
    const bool has_res = s.res != nullptr;
    const uint32_t row_bytes = (uint32_t)s.H * 2;
    uint4 *g_sm = reinterpret_cast<uint4 *>(dsm);
    unsigned char *stages = dsm + row_bytes;
    const size_t stage_bytes = (size_t)row_bytes * (has_res ? 2 : 1);
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + stage_bytes * kStages);
    int *issued = reinterpret_cast<int *>(bars + kStages);

    const int64_t first = blockIdx.x, step = gridDim.x;
    if (first >= s.M)
        return;

    auto issue = [&](int64_t row, int st) {   // thread 0 only
        if (row >= s.M) {
            issued[st] = 0;
            return;
        }
        if (row == p.debug_skip_row) {         // test hook: this copy never comes
            issued[st] = 0;
            return;
        }
        unsigned char *dst = stages + stage_bytes * st;
        mbar_arrive_expect_tx(&bars[st], row_bytes * (has_res ? 2u : 1u));
        bulk_g2s(dst, s.x + row * s.ldx_v, row_bytes, &bars[st]);
        if (has_res)
            bulk_g2s(dst + row_bytes, s.res + row * s.ldres_v, row_bytes, &bars[st]);
        issued[st] = 1;
    };

    if (t == 0) {
        for (int st = 0; st < kStages; ++st)
            mbar_init(&bars[st], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int st = 0; st < kStages; ++st)
            issue(first + st * step, st);
    }
    for (int v = t; v < nvec; v += tpr)
        g_sm[v] = ld_keep(s.gamma + v);
    __syncthreads();

    int it = 0;
    for (int64_t row = first; row < s.M; row += step, ++it) {
        const int st = it % kStages;
        const uint32_t parity = (uint32_t)((it / kStages) & 1);
        const bool got = mbar_wait_bounded(&bars[st], parity, p.wait_limit_ns);

        const uint4 *xs = reinterpret_cast<const uint4 *>(stages + stage_bytes * st);
        const uint4 *rs = xs + nvec;
        uint4 r[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + t;
            if (!GUARD || v < nvec) {
                r[k] = lds128(xs + v);
                if (has_res)
                    r[k] = add_bf16x8(r[k], lds128(rs + v));
            } else {
                r[k] = make_uint4(0, 0, 0, 0);
            }
        }
        // everyone has read the stage (and agrees whether its copy arrived)
        if (__syncthreads_or(!got)) {
            if (t == 0) {
                atomicOr(p.status, 1u);
                for (int o = 0; o < kStages; ++o) {       // drain every copy still in flight
                    const int so = (st + o) % kStages;
                    if (issued[so]) {
                        const uint32_t po = (uint32_t)(((it + o) / kStages) & 1);
                        if (!mbar_wait_bounded(&bars[so], po, p.wait_limit_ns))
                            atomicOr(p.status, 2u);
                    }
                }
            }
            __syncthreads();
            return;
        }
        if (t == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(row + (int64_t)kStages * step, st);
        }
        if (has_res) {
            const int64_t nv = nvec;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int v = k * tpr + t;
                if ((!GUARD || v < nvec) && RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && v < nvec))
                    s.out_res[row * nv + v] = r[k];
            }
        }
        row_finish<VPT, TPR, MX, GAMMA_SHARED>(s, row, t, 0, it & 1, red, r, g_sm, r);   // r: unused gamma registers
    }
}

template <bool MX>
cudaError_t launch_bulk_impl(int vpt, int tpr_static, const BulkParams &p, int grid, int threads,
                             size_t smem, cudaStream_t st)
{
    auto go = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        kern<<<grid, threads, smem, st>>>(p);
        return cudaGetLastError();
    };
    if (tpr_static)
        return (vpt == 4 && tpr_static == 224) ? go(bulk_kernel<4, 224, MX>) : cudaErrorInvalidValue;
    switch (vpt) {
    case 1: return go(bulk_kernel<1, 0, MX>);
    case 2: return go(bulk_kernel<2, 0, MX>);
    case 3: return go(bulk_kernel<3, 0, MX>);
    case 4: return go(bulk_kernel<4, 0, MX>);
    case 5: return go(bulk_kernel<5, 0, MX>);
    case 6: return go(bulk_kernel<6, 0, MX>);
    case 7: return go(bulk_kernel<7, 0, MX>);
    case 8: return go(bulk_kernel<8, 0, MX>);
    default: return cudaErrorInvalidValue;
    }
}

template <bool MX>
int bulk_blocks_per_sm(int vpt, int tpr_static, int threads, size_t smem)
{
    int n = 0;
    auto occ = [&](auto kern) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess)
            n = 0;
    };
    if (tpr_static) {
        if (vpt == 4 && tpr_static == 224)
            occ(bulk_kernel<4, 224, MX>);
        return n;
    }
    switch (vpt) {
    case 1: occ(bulk_kernel<1, 0, MX>); break;
    case 2: occ(bulk_kernel<2, 0, MX>); break;
    case 3: occ(bulk_kernel<3, 0, MX>); break;
    case 4: occ(bulk_kernel<4, 0, MX>); break;
    case 5: occ(bulk_kernel<5, 0, MX>); break;
    case 6: occ(bulk_kernel<6, 0, MX>); break;
    case 7: occ(bulk_kernel<7, 0, MX>); break;
    case 8: occ(bulk_kernel<8, 0, MX>); break;
    default: break;
    }
    return n;
}

}  // namespace rmsq
