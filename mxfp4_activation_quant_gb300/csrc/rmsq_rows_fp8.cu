// Row-kernel instantiations for the 1x128 FP8 E4M3 quantiser.
#include "rmsq_rowkernel.cuh"

namespace rmsq {

cudaError_t launch_rows_fp8(int vpt, int tpr_static, int lat, const LaunchParams &p, int grid, int threads,
                            cudaStream_t st)
{
    return launch_rows_impl<false>(vpt, tpr_static, lat, p, grid, threads, st);
}

bool vpt_instantiated(int vpt) { return vpt >= 1 && vpt <= 8; }

bool static_shape(int vpt, int tpr)
{
#define RMSQ_IS_STATIC(V, T) \
    if (vpt == V && tpr == T) \
        return true;
    RMSQ_STATIC_SHAPES(RMSQ_IS_STATIC)
#undef RMSQ_IS_STATIC
    return false;
}

}  // namespace rmsq
