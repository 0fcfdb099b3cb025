// Row-kernel instantiations for the MXFP4 (E8M0 + E2M1, group 32) quantiser.
#include "rmsq_rowkernel.cuh"

namespace rmsq {

cudaError_t launch_rows_mx(int vpt, int tpr_static, int lat, const LaunchParams &p, int grid, int threads,
                            cudaStream_t st)
{
    return launch_rows_impl<true>(vpt, tpr_static, lat, p, grid, threads, st);
}

}  // namespace rmsq
