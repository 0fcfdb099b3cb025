// Plain device-to-device copy, the read + write peak the HBM roofline is
// taken against when no separately measured figure is at hand: a grid of
// resident blocks (a multiple of the SM count) streams 16-byte vectors, four
// in flight per thread, with loads and stores that bypass L1 and are marked
// evict-first, so every byte crosses HBM once each way.
#include "rmsq.h"
#include "rmsq_internal.h"

namespace rmsq {
namespace {

__global__ void __launch_bounds__(512) copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                   int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride), c = __ldcs(src + i + 2 * stride),
              d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride)
        __stcs(dst + i, __ldcs(src + i));
}

}  // namespace
}  // namespace rmsq

extern "C" rmsq_status rmsq_copy(const void *src, void *dst, int64_t bytes, void *stream)
{
    if (bytes < 0 || (bytes && (!src || !dst)) || bytes % 16 || ((uintptr_t)src | (uintptr_t)dst) % 16)
        return rmsq::set_error(RMSQ_ERR_INVALID_ARG,
                               "rmsq_copy needs 16-byte aligned, non-NULL buffers and a multiple of 16 bytes");
    const uintptr_t s = (uintptr_t)src, d = (uintptr_t)dst;
    if (bytes && s < d + (uintptr_t)bytes && d < s + (uintptr_t)bytes)
        return rmsq::set_error(RMSQ_ERR_INVALID_ARG, "rmsq_copy: source and destination overlap");
    if (bytes == 0)
        return rmsq::clear_error();
    const int sms = rmsq::device_sm_count();
    if (sms <= 0)
        return rmsq::set_error(RMSQ_ERR_CUDA, "rmsq_copy: SM count unavailable");
    const int64_t n = bytes / 16;
    int64_t blocks = (n + 511) / 512;
    if (blocks > (int64_t)sms * 4)
        blocks = (int64_t)sms * 4;
    rmsq::copy_kernel<<<(int)blocks, 512, 0, (cudaStream_t)stream>>>((const uint4 *)src, (uint4 *)dst, n);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return rmsq::set_error(RMSQ_ERR_CUDA, cudaGetErrorString(e));
    return rmsq::clear_error();
}
