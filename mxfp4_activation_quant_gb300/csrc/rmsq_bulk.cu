// Persistent bulk-copy kernel instantiations (FP8 1x128 and MXFP4 1x32).
#include "rmsq_bulk.cuh"

namespace rmsq {

cudaError_t launch_bulk(bool mx, int vpt, int tpr_static, const BulkParams &p, int grid, int threads,
                        size_t smem, cudaStream_t st)
{
    return mx ? launch_bulk_impl<true>(vpt, tpr_static, p, grid, threads, smem, st)
              : launch_bulk_impl<false>(vpt, tpr_static, p, grid, threads, smem, st);
}

int bulk_occupancy(bool mx, int vpt, int tpr_static, int threads, size_t smem)
{
    return mx ? bulk_blocks_per_sm<true>(vpt, tpr_static, threads, smem)
              : bulk_blocks_per_sm<false>(vpt, tpr_static, threads, smem);
}

size_t bulk_smem(int H, bool has_res) { return bulk_smem_bytes(H, has_res); }

}  // namespace rmsq
