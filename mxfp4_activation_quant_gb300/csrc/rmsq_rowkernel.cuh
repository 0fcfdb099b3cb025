// Register-resident row kernel: each team loads its row of x (and residual)
// straight into registers with 16-byte streaming loads, adds, writes the
// residual back, and finishes the row (rmsq_rows.cuh). One launch covers one
// or two segments; blocks [0, seg[0].blocks) belong to the first.
#pragma once

#include "rmsq_rows.cuh"

namespace rmsq {

template <int VPT, bool MX>
__global__ void __launch_bounds__(kMaxThreads) rows_kernel(const __grid_constant__ LaunchParams p)
{
    __shared__ RedSmem red;
    int b = blockIdx.x;
    int si = 0;
    if (p.nseg == 2 && b >= p.seg[0].blocks) {
        b -= p.seg[0].blocks;
        si = 1;
    }
    const Seg &s = p.seg[si];
    const int tpr = s.tpr;
    const int team = threadIdx.x / tpr;
    if (team >= s.rpb)
        return;                                   // idle team of a shared-size block
    const int t = threadIdx.x - team * tpr;
    const int64_t row = (int64_t)b * s.rpb + team;
    if (row >= s.M)
        return;                                   // whole teams leave together

    const int nvec = s.H >> 3;
    uint4 r[VPT];
    const uint4 *xr = s.x + row * s.ldx_v;
    // vectors past the row end (padded team shapes) read as zero and are
    // never stored; they add nothing to the sum of squares
    if (s.res) {
        const uint4 *rr = s.res + row * s.ldres_v;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + t;
            xv[k] = v < nvec ? ld_stream(xr + v) : make_uint4(0, 0, 0, 0);
            rv[k] = v < nvec ? ld_stream(rr + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + t;
            r[k] = add_bf16x8(xv[k], rv[k]);
            if (v < nvec)
                s.out_res[row * nvec + v] = r[k];
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = k * tpr + t;
            r[k] = v < nvec ? ld_stream(xr + v) : make_uint4(0, 0, 0, 0);
        }
    }
    row_finish<VPT, MX, false>(s, row, t, team, 0, red, r, s.gamma);
}

template <bool MX>
cudaError_t launch_rows_impl(int vpt, const LaunchParams &p, int grid, int threads, cudaStream_t st)
{
    switch (vpt) {
    case 1: rows_kernel<1, MX><<<grid, threads, 0, st>>>(p); break;
    case 2: rows_kernel<2, MX><<<grid, threads, 0, st>>>(p); break;
    case 3: rows_kernel<3, MX><<<grid, threads, 0, st>>>(p); break;
    case 4: rows_kernel<4, MX><<<grid, threads, 0, st>>>(p); break;
    case 5: rows_kernel<5, MX><<<grid, threads, 0, st>>>(p); break;
    case 6: rows_kernel<6, MX><<<grid, threads, 0, st>>>(p); break;
    case 7: rows_kernel<7, MX><<<grid, threads, 0, st>>>(p); break;
    case 8: rows_kernel<8, MX><<<grid, threads, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace rmsq
