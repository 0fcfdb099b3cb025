// Dual-tensor (MLA q_a / kv_a) kernel instantiations, FP8 1x128 and MXFP4.
#include "rmsq_rowkernel.cuh"

namespace rmsq {

// The MLA latent pair (q_a 1536, kv_a 512): one warp per q_a row with six
// vectors per thread (no cross-warp step: 14.73 against 15.59 us for the
// FP8 pair at M = 8192 with a two-warp team of three vectors each), and
// 16-thread teams of four vectors for kv_a. Launches of at most one block per
// SM take the pair's latency form (gamma loaded with each row).
bool static_dual_shape(int v0, int t0, int v1, int t1)
{
    return v0 == 6 && t0 == 32 && v1 == 4 && t1 == 16;
}

template <bool MX>
cudaError_t launch_dual_impl(bool lat, int v0, int t0, int v1, int t1, const LaunchParams &p, int grid,
                             int threads, cudaStream_t st)
{
    if (t0 || t1) {
        if (!static_dual_shape(v0, t0, v1, t1))
            return cudaErrorInvalidValue;
        return lat ? launch_pdl(dual_kernel_lat<6, 32, 4, 16, MX>, grid, threads, st, p)
                   : launch_pdl(dual_kernel<6, 32, 4, 16, MX>, grid, threads, st, p);
    }
    if (v0 != v1)
        return cudaErrorInvalidValue;
    switch (v0) {
    case 1: return launch_pdl(dual_kernel<1, 0, 1, 0, MX>, grid, threads, st, p);
    case 2: return launch_pdl(dual_kernel<2, 0, 2, 0, MX>, grid, threads, st, p);
    case 3: return launch_pdl(dual_kernel<3, 0, 3, 0, MX>, grid, threads, st, p);
    case 4: return launch_pdl(dual_kernel<4, 0, 4, 0, MX>, grid, threads, st, p);
    case 5: return launch_pdl(dual_kernel<5, 0, 5, 0, MX>, grid, threads, st, p);
    case 6: return launch_pdl(dual_kernel<6, 0, 6, 0, MX>, grid, threads, st, p);
    case 7: return launch_pdl(dual_kernel<7, 0, 7, 0, MX>, grid, threads, st, p);
    case 8: return launch_pdl(dual_kernel<8, 0, 8, 0, MX>, grid, threads, st, p);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dual(bool mx, bool lat, int v0, int t0, int v1, int t1, const LaunchParams &p, int grid,
                        int threads, cudaStream_t st)
{
    return mx ? launch_dual_impl<true>(lat, v0, t0, v1, t1, p, grid, threads, st)
              : launch_dual_impl<false>(lat, v0, t0, v1, t1, p, grid, threads, st);
}

}  // namespace rmsq
