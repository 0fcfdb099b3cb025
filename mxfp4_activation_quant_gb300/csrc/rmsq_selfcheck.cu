// Exhaustive check of the group-division shortcut used by the FP8 quantiser:
// for every positive finite bf16 amax and every bf16 y with |y| <= amax (both
// signs), the E4M3 code of the shortcut quotient is compared with the code of
// IEEE fp32 division by d = RN(amax / 448), and the shortcut scale itself with
// IEEE amax / 448. Counts are accumulated in a caller-provided device array.
#include "rmsq.h"
#include "rmsq_device.cuh"

namespace rmsq {
namespace {

__global__ void check_group_division_kernel(unsigned long long *counts)
{
    const uint32_t a = blockIdx.x + 1;                 // bf16 bits of amax: 0x0001 .. 0x7F7F
    const float amax = __uint_as_float(a << 16);
    const float d = div448(amax);
    const GroupDivisor g = make_group_divisor(d);
    if (threadIdx.x == 0 && __float_as_uint(d) != __float_as_uint(__fdiv_rn(amax, 448.0f)))
        atomicAdd(&counts[3], 1ull);
    unsigned long long code_bad = 0, quot_bad = 0, norm_bad = 0, n = 0;
    for (uint32_t b = threadIdx.x; b <= a; b += blockDim.x) {
        for (uint32_t sgn = 0; sgn < 2; ++sgn) {
            const float y = __uint_as_float((b | (sgn << 15)) << 16);
            const float ref = __fdiv_rn(y, d);
            float got = ref, got_hi = ref;
            if (g.fast) {
                // the packed form the kernels use: y in both halves of a bf16
                // pair, so both lanes' unpacking paths are exercised
                const uint32_t w = b | (sgn << 15);
                const float2 pair = div_fast_neg2(unpack_neg_bf16x2(w | (w << 16)), g);
                got = pair.x;
                got_hi = pair.y;
            }
            code_bad += (e4m3x2(got, 0.0f) & 0xffu) != (e4m3x2(ref, 0.0f) & 0xffu) ||
                        (e4m3x2(got_hi, 0.0f) & 0xffu) != (e4m3x2(ref, 0.0f) & 0xffu);
            const bool qb = __float_as_uint(got) != __float_as_uint(ref);
            quot_bad += qb;
            norm_bad += qb && fabsf(y) >= 0x1p-100f;
            ++n;
        }
    }
    for (int off = 16; off; off >>= 1) {
        code_bad += __shfl_xor_sync(0xffffffffu, code_bad, off);
        quot_bad += __shfl_xor_sync(0xffffffffu, quot_bad, off);
        n += __shfl_xor_sync(0xffffffffu, n, off);
        norm_bad += __shfl_xor_sync(0xffffffffu, norm_bad, off);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&counts[0], code_bad);
        atomicAdd(&counts[1], quot_bad);
        atomicAdd(&counts[2], n);
        atomicAdd(&counts[4], norm_bad);
    }
}

}  // namespace
}  // namespace rmsq

extern "C" rmsq_status rmsq_check_group_division(unsigned long long *counts, void *stream)
{
    if (!counts || ((uintptr_t)counts % 8))
        return RMSQ_ERR_INVALID_ARG;
    rmsq::check_group_division_kernel<<<0x7F7F, 256, 0, (cudaStream_t)stream>>>(counts);
    return cudaGetLastError() == cudaSuccess ? RMSQ_OK : RMSQ_ERR_CUDA;
}
