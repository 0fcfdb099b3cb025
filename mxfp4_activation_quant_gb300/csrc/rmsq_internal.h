// Host/device descriptors shared by the C-ABI layer and the kernel units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "rmsq.h"

namespace rmsq {

// One tensor (a "segment") handled by a launch. A launch covers one segment,
// or two for the MLA q_a / kv_a latent pair. Pointers to bf16 rows are given
// as 16-byte vectors of 8 bf16 values; leading dimensions are in vectors.
struct Seg {
    const uint4 *x;        // [M, ldx_v] bf16 rows
    const uint4 *res;      // nullable: [M, ldres_v] bf16 residual rows
    const uint4 *gamma;    // [H] bf16
    uint4 *out_res;        // [M, H] bf16 (required iff res)
    uint4 *out_bf16;       // nullable: [M, H] bf16 normalised y
    uint8_t *out_q;        // FP8: [M, H] e4m3; MXFP4: [M, H/2] packed e2m1
    void *out_scale;       // FP8: fp32 [M, H/128] or [H/128, M]; MXFP4: e8m0 [M, H/32]
    int64_t M;
    int64_t ldx_v, ldres_v;
    int32_t H;
    int32_t tpr;           // threads per row (a "team")
    int32_t rpb;           // rows (teams) per block
    int32_t blocks;        // blocks of the row kernel that belong to this segment
    int32_t layout;        // FP8: 0 row-major, 1 column-major (either padded); MXFP4: 0 row-major,
                           // 1 the 128x4-tile layout of block-scaled MMA scale factors
    int64_t scale_ld;      // FP8 column-major: leading dimension (>= M); MXFP4 tiled: k-tiles per row tile
    float eps;
    float inv_h;           // fp32 rounding of 1/H
    int64_t prefetch_rows; // row kernel: rows ahead whose x / residual are prefetched into L2 (0 = off)
#ifdef RMSQ_DEBUG
    unsigned int *debug_flag;   // status word; bounds checks of the debug build set bit 2
    int64_t scale_elems;        // capacity of out_scale in elements
#endif
};

struct LaunchParams {
    Seg seg[2];
    int32_t nseg;
};

// Persistent bulk-copy kernel: one segment, one row per team, rows strided
// by the grid, x / residual rows staged through shared memory.
struct BulkParams {
    Seg s;
    int64_t debug_skip_row;   // -1 normally; a row whose copy is never issued
    int64_t wait_limit_ns;    // bound on every mbarrier wait
    unsigned int *status;     // device status word (set on a timed-out wait)
};

// Error reporting and device queries of the C-ABI layer (rmsq_api.cu), for
// the GEMM's host code: set_error records the message of the failing call
// on this host thread; the status word is the one bounded waits report to.
rmsq_status set_error(rmsq_status s, const char *msg);
rmsq_status clear_error();
int device_sm_count();
unsigned int *device_status_word(int dev);

constexpr int kMaxThreads = 512;

// Launchers (a switch over the instantiations each). tpr_static != 0 selects
// a kernel compiled for that exact team size (see static_shape).
// lat > 0 selects the latency form of a compiled team shape (gamma loaded
// with the row, one barrier per row; bit-identical results) with each row's
// outputs shared by `lat` blocks (1, 2 or 4; block b holds row b / lat);
// lat = 0 the throughput form.
cudaError_t launch_rows_fp8(int vpt, int tpr_static, int lat, const LaunchParams &p, int grid, int threads,
                            cudaStream_t st);
cudaError_t launch_rows_mx(int vpt, int tpr_static, int lat, const LaunchParams &p, int grid, int threads,
                           cudaStream_t st);
// lat: the latency form of the compiled MLA pair shape (ignored for others)
cudaError_t launch_dual(bool mx, bool lat, int v0, int t0, int v1, int t1, const LaunchParams &p, int grid,
                        int threads, cudaStream_t st);
cudaError_t launch_bulk(bool mx, int vpt, int tpr_static, const BulkParams &p, int grid, int threads,
                        size_t smem, cudaStream_t st);
int bulk_occupancy(bool mx, int vpt, int tpr_static, int threads, size_t smem);
size_t bulk_smem(int H, bool has_res);
bool vpt_instantiated(int vpt);
// Team shapes also compiled with a fixed team size (exact fits of common
// widths, listed in rmsq_rowkernel.cuh; H = 7168 is 4 vectors x 224 threads);
// the MLA pair q_a 1536 as 3 x 64 and kv_a 512 as 4 x 16. The persistent
// kernel has a fixed-size instantiation for 4 x 224 only.
bool static_shape(int vpt, int tpr);
bool static_dual_shape(int v0, int t0, int v1, int t1);

}  // namespace rmsq
