// C ABI of librmsq (include/rmsq.h): host-side argument checks, choice of
// kernel and team shape, launch, and status reporting. Nothing here
// allocates device memory; the only device state is the status word that
// bounded waits report through.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "rmsq.h"
#include "rmsq_device.cuh"
#include "rmsq_internal.h"

namespace rmsq {

// Set by a kernel whose bounded wait ran out; read and cleared by
// rmsq_sync_status.
__device__ unsigned int g_status_word;

namespace {

thread_local char g_last_error[512];

rmsq_status fail(rmsq_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

rmsq_status ok()
{
    g_last_error[0] = 0;
    return RMSQ_OK;
}

struct Range {
    uintptr_t lo, hi;
};

Range mat_range(const void *p, int64_t M, int64_t H, int64_t ld, int64_t elem)
{
    uintptr_t lo = (uintptr_t)p;
    return Range{lo, lo + (uintptr_t)(((M - 1) * ld + H) * elem)};
}

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Team shape for a row of nvec 16-byte vectors and groups of gv vectors: the
// smallest legal team (a multiple of gv dividing 32, or a multiple of 32)
// that holds the row with vpt vectors per thread. `waste` counts the padded
// vector slots; padding is always whole groups.
bool team_ok(int64_t nvec, int vpt, int gv, int &tpr, int64_t &waste)
{
    if (!vpt_instantiated(vpt))
        return false;
    int64_t need = (nvec + vpt - 1) / vpt;
    int64_t t;
    if (need <= 32) {
        t = gv;
        while (t < need)
            t <<= 1;
    } else {
        t = (need + 31) / 32 * 32;
    }
    if (t > kMaxThreads)
        return false;
    tpr = (int)t;
    waste = t * vpt - nvec;
    return true;
}

// Measured on GB300 (H=7168 prefill, H=1536 q_a, M=64 decode): 4 vectors per
// thread (224 threads per 7168-wide row) is fastest where it fits exactly.
const int kVptPreference[] = {4, 3, 5, 6, 2, 7, 8, 1};

// Exact shapes first, in preference order; otherwise the least padding.
int pick_vpt(int64_t nvec, int gv, int forced, int &tpr)
{
    int64_t waste;
    if (forced)
        return team_ok(nvec, forced, gv, tpr, waste) ? forced : 0;
    int best = 0, best_tpr = 0;
    int64_t best_waste = -1;
    for (int v : kVptPreference) {
        int t;
        if (!team_ok(nvec, v, gv, t, waste))
            continue;
        if (best_waste < 0 || waste < best_waste) {
            best = v;
            best_tpr = t;
            best_waste = waste;
        }
    }
    tpr = best_tpr;
    return best;
}

int default_rows_per_block(int tpr) { return tpr >= 256 ? 1 : 256 / tpr; }

const rmsq_launch_opts kDefaultOpts = {RMSQ_KERNEL_AUTO, 0, 0, 0, -1, 0, RMSQ_FORM_AUTO, 0};

// Checks shared by the single-tensor FP8 and MXFP4 calls.
rmsq_status check_single(const void *x, int64_t ld_x, const void *residual, int64_t ld_res,
                         const void *gamma, float eps, int64_t M, int64_t H, int64_t group,
                         const void *out_q, int64_t q_bytes_per_row, const void *out_scale,
                         int64_t scale_bytes, int64_t scale_align, const void *out_residual,
                         const void *out_bf16)
{
    if (M < 0 || H <= 0)
        return fail(RMSQ_ERR_INVALID_ARG, "M must be >= 0 and H > 0 (M=%lld, H=%lld)",
                    (long long)M, (long long)H);
    if (H % group)
        return fail(RMSQ_ERR_INVALID_ARG, "H=%lld is not a multiple of the group %lld",
                    (long long)H, (long long)group);
    if (H > (int64_t)8 * 8 * kMaxThreads)
        return fail(RMSQ_ERR_UNSUPPORTED, "H=%lld exceeds the largest row (%d)", (long long)H,
                    8 * 8 * kMaxThreads);
    if (!(eps >= 0.0f) || !std::isfinite(eps))
        return fail(RMSQ_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (M == 0)
        return RMSQ_OK;
    const bool norm_only = q_bytes_per_row == 0;   // rmsq_add_rmsnorm: y is the only result
    if (norm_only ? (!x || !gamma || !out_bf16 || out_q || out_scale)
                  : (!x || !gamma || !out_q || !out_scale))
        return fail(RMSQ_ERR_INVALID_ARG, norm_only ? "x, gamma and out_bf16 are required"
                                                    : "x, gamma, out_q and out_scale are required");
    if ((residual == nullptr) != (out_residual == nullptr))
        return fail(RMSQ_ERR_INVALID_ARG, "out_residual must be given exactly when residual is");
    if (ld_x < H || (residual && ld_res < H))
        return fail(RMSQ_ERR_INVALID_ARG, "leading dimensions must be >= H");
    if (!aligned(x, 16) || !aligned(gamma, 16) || ld_x % 8 || (residual && (!aligned(residual, 16) || ld_res % 8)))
        return fail(RMSQ_ERR_MISALIGNED,
                    "bf16 inputs need 16-byte aligned bases and leading dimensions that are multiples of 8");
    if (!aligned(out_q, 16) || (out_residual && !aligned(out_residual, 16)) ||
        (out_bf16 && !aligned(out_bf16, 16)) || !aligned(out_scale, (uintptr_t)scale_align))
        return fail(RMSQ_ERR_MISALIGNED, "outputs need 16-byte aligned bases (scales: element-aligned)");

    Range rx = mat_range(x, M, H, ld_x, 2);
    Range rg = mat_range(gamma, 1, H, H, 2);
    Range outs[4] = {{0, 0}, {0, 0}, {0, 0}, {0, 0}};
    int nout = 0;
    if (!norm_only) {
        outs[nout++] = mat_range(out_q, M, q_bytes_per_row, q_bytes_per_row, 1);
        outs[nout++] = mat_range(out_scale, 1, scale_bytes, scale_bytes, 1);
    }
    if (out_bf16)
        outs[nout++] = mat_range(out_bf16, M, H, H, 2);
    Range rres_out = {0, 0};
    if (out_residual) {
        rres_out = mat_range(out_residual, M, H, H, 2);
        outs[nout++] = rres_out;
    }
    for (int i = 0; i < nout; ++i) {
        if (overlaps(outs[i], rx) || overlaps(outs[i], rg))
            return fail(RMSQ_ERR_INVALID_ARG, "an output overlaps x or gamma");
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j]))
                return fail(RMSQ_ERR_INVALID_ARG, "two outputs overlap");
    }
    if (residual) {
        Range rr = mat_range(residual, M, H, ld_res, 2);
        bool in_place = out_residual == residual;
        if (in_place && ld_res != H)
            return fail(RMSQ_ERR_INVALID_ARG, "in-place residual update needs ld_res == H");
        for (int i = 0; i < nout; ++i) {
            if (in_place && outs[i].lo == rres_out.lo && outs[i].hi == rres_out.hi)
                continue;
            if (overlaps(outs[i], rr))
                return fail(RMSQ_ERR_INVALID_ARG, "an output overlaps the residual input");
        }
    }
    return RMSQ_OK;
}

Seg make_seg(const void *x, int64_t ld_x, const void *residual, int64_t ld_res,
             const void *gamma, float eps, int64_t M, int64_t H, void *out_q, void *out_scale,
             int32_t layout, void *out_residual, void *out_bf16)
{
    Seg s{};
    s.x = (const uint4 *)x;
    s.res = (const uint4 *)residual;
    s.gamma = (const uint4 *)gamma;
    s.out_res = (uint4 *)out_residual;
    s.out_bf16 = (uint4 *)out_bf16;
    s.out_q = (uint8_t *)out_q;
    s.out_scale = out_scale;
    s.M = M;
    s.ldx_v = ld_x / 8;
    s.ldres_v = residual ? ld_res / 8 : 0;
    s.H = (int32_t)H;
    s.layout = layout;
    s.scale_ld = M;
    s.eps = eps;
    s.inv_h = (float)(1.0 / (double)H);
    return s;
}

// Number of SMs of the current device (0 if the query fails).
int sm_count()
{
    static std::atomic<int> cached[128];   // every thread stores the same value
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
        return 0;
    int n = cached[dev].load(std::memory_order_acquire);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cached[dev].store(n, std::memory_order_release);
    }
    return n;
}

// Device address of the status word, looked up once per device.
unsigned int *status_word_ptr(int dev)
{
    static std::atomic<unsigned int *> ptrs[128];   // every thread stores the same value
    if (dev < 0 || dev >= 128)
        return nullptr;
    unsigned int *ptr = ptrs[dev].load(std::memory_order_acquire);
    if (!ptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess)
            return nullptr;
        ptr = (unsigned int *)p;
        ptrs[dev].store(ptr, std::memory_order_release);
    }
    return ptr;
}

// Debug build: point the segment's bounds checks at the status word and
// give them the scale buffer's capacity. Nothing in release builds.
void debug_bind(Seg &s, int64_t scale_elems)
{
#ifdef RMSQ_DEBUG
    int dev = 0;
    cudaGetDevice(&dev);
    s.debug_flag = status_word_ptr(dev);
    s.scale_elems = scale_elems;
#else
    (void)s;
    (void)scale_elems;
#endif
}

rmsq_status launch_single(Seg s, bool mx, const rmsq_launch_opts &o, cudaStream_t st)
{
    const int gv = mx ? 4 : 16;
    int tpr = 0;
    int vpt = pick_vpt(s.H / 8, gv, o.vpt, tpr);
    if (!vpt)
        return fail(RMSQ_ERR_UNSUPPORTED, "no team shape for H=%d with vpt=%d", s.H, o.vpt);
    s.tpr = tpr;
    int kernel = o.kernel == RMSQ_KERNEL_AUTO ? RMSQ_KERNEL_ROWS : o.kernel;
    if (kernel == RMSQ_KERNEL_ROWS) {
        int rpb = o.rows_per_block > 0 ? o.rows_per_block : default_rows_per_block(tpr);
        if ((int64_t)rpb * tpr > kMaxThreads || (tpr > 32 && rpb > 15))
            return fail(RMSQ_ERR_INVALID_ARG, "rows_per_block=%d too large for %d threads per row",
                        rpb, tpr);
        s.rpb = rpb;
        // L2 prefetch about three resident blocks per SM ahead (measured on
        // GB300: 300-600 rows ahead helps the MXFP4 row kernel by ~3 % and is
        // neutral for FP8; twice as far hurts both); only for long batches.
        const int64_t ahead = (int64_t)3 * sm_count() * rpb;
        s.prefetch_rows = (ahead > 0 && s.M > 4 * ahead) ? ahead : 0;
        int64_t blocks = (s.M + rpb - 1) / rpb;
        if (blocks > 0x7fffffff)
            return fail(RMSQ_ERR_UNSUPPORTED, "M too large");
        s.blocks = (int32_t)blocks;
        LaunchParams p{};
        p.seg[0] = s;
        p.nseg = 1;
        const int ts = (static_shape(vpt, tpr) && vpt * tpr * 8 == s.H) ? tpr : 0;
        // The latency form (gamma loaded with the row, one barrier per row)
        // when the launch is at most one block per SM: there the row's
        // dependent chain, not bandwidth, sets the time. With SMs to spare,
        // each row's outputs are shared by 2 or 4 blocks on as many SMs: every
        // one of them loads and reduces the whole row (the same inv_rms) and
        // normalises, quantises and stores its part.
        if (o.form != RMSQ_FORM_AUTO && o.form != RMSQ_FORM_THROUGHPUT && o.form != RMSQ_FORM_LATENCY)
            return fail(RMSQ_ERR_INVALID_ARG, "unknown kernel form %d", o.form);
        if (o.split != 0 && o.split != 1 && o.split != 2 && o.split != 4)
            return fail(RMSQ_ERR_INVALID_ARG, "split must be 0, 1, 2 or 4 (got %d)", o.split);
        const int64_t sms = sm_count();
        const bool lat = ts && (o.form == RMSQ_FORM_LATENCY || (o.form == RMSQ_FORM_AUTO && blocks <= sms));
        if (lat && o.rows_per_block <= 0) {
            // Latency form, rows per block chosen here: as few rows per block
            // (whole warps) as keep the launch within one block per SM, so
            // that the rows spread over as many SMs as there are.
            const int64_t spread = std::max<int64_t>((s.M + sms - 1) / sms, (32 + tpr - 1) / tpr);
            if (spread < rpb) {
                rpb = (int)spread;
                blocks = (s.M + rpb - 1) / rpb;
                s.rpb = rpb;
                s.blocks = (int32_t)blocks;
                p.seg[0] = s;
            }
        }
        // Every block of a split row reads the whole residual row and writes
        // back its own part, so a residual updated in place is not split: a
        // part could be written before another block of the row has read it.
        const bool in_place = s.res && (const void *)s.res == (const void *)s.out_res;
        int split = 1;
        if (in_place && o.split > 1) {
            return fail(RMSQ_ERR_UNSUPPORTED, "split rows need out_residual separate from residual "
                                              "(an in-place residual update is not split)");
        } else if (lat && rpb == 1 && !in_place) {
            if (o.split) {
                split = o.split;
            } else {
                for (int c : {4, 2})
                    if (vpt % c == 0 && s.M * c <= sms) {
                        split = c;
                        break;
                    }
            }
            if (vpt % split)
                return fail(RMSQ_ERR_UNSUPPORTED, "split %d does not divide %d vectors per thread", split, vpt);
        } else if (o.split > 1) {
            return fail(RMSQ_ERR_UNSUPPORTED, "split rows need the latency form of a compiled team shape "
                                              "with one row per block");
        }
        const int64_t grid = blocks * split;   // split > 1 only with one row per block
        if (grid > 0x7fffffff)
            return fail(RMSQ_ERR_UNSUPPORTED, "M too large");
        const int form = lat ? split : 0;
        cudaError_t e = mx ? launch_rows_mx(vpt, ts, form, p, (int)grid, rpb * tpr, st)
                           : launch_rows_fp8(vpt, ts, form, p, (int)grid, rpb * tpr, st);
        if (e != cudaSuccess)
            return fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
        return ok();
    }
    if (kernel == RMSQ_KERNEL_PERSISTENT) {
        if (tpr < 32)
            return fail(RMSQ_ERR_UNSUPPORTED, "the persistent kernel needs rows of >= 32 threads");
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        int sms = 0, smem_max = 0;
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess)
            return fail(RMSQ_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
        size_t smem = bulk_smem(s.H, s.res != nullptr);
        if (smem + sizeof(float2) * 64 + 256 > (size_t)smem_max)
            return fail(RMSQ_ERR_UNSUPPORTED, "H=%d needs %zu bytes of shared memory", s.H, smem);
        const int ts = (vpt == 4 && tpr == 224 && s.H == 7168) ? tpr : 0;
        int64_t grid = o.grid;
        if (grid <= 0) {
            int per_sm = bulk_occupancy(mx, vpt, ts, tpr, smem);
            if (per_sm <= 0)
                return fail(RMSQ_ERR_UNSUPPORTED, "persistent kernel does not fit on an SM");
            grid = (int64_t)per_sm * sms;
        }
        if (grid > s.M)
            grid = s.M;
        unsigned int *status = status_word_ptr(dev);
        if (!status)
            return fail(RMSQ_ERR_CUDA, "status word address unavailable");
        s.rpb = 1;
        BulkParams bp{};
        bp.s = s;
        bp.debug_skip_row = o.debug_skip_row;
        bp.wait_limit_ns = o.wait_limit_ns > 0 ? o.wait_limit_ns : 2000000000LL;
        bp.status = status;
        e = launch_bulk(mx, vpt, ts, bp, (int)grid, tpr, smem, st);
        if (e != cudaSuccess)
            return fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
        return ok();
    }
    return fail(RMSQ_ERR_INVALID_ARG, "unknown kernel %d", o.kernel);
}

// ------------------------------------------------ debug-build self-test

#ifdef RMSQ_DEBUG
__global__ void debug_bounds_selftest_kernel(unsigned int *flag, int64_t n)
{
    // an index equal to the extent: the check fails and the store is skipped
    if (RMSQ_IN_BOUNDS(flag, n < n))
        flag[0] |= 0u;
}
#endif

// Clears the given bits of the status word (rmsq_sync_status).
__global__ void clear_status_bits_kernel(unsigned int bits) { atomicAnd(&g_status_word, ~bits); }

// ------------------------------------------------------- encoder kernels

__global__ void encode_e4m3_kernel(const float *in, uint8_t *out, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(e4m3x2(in[i], 0.0f) & 0xffu);
}

__global__ void encode_e2m1_kernel(const float *in, uint8_t *out, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[i] = (uint8_t)(e2m1x2(in[i], 0.0f) & 0xfu);
}

// The MLA latent pair, FP8 (group 128, fp32 scales) or MXFP4 (group 32, E8M0
// bytes, q packed two per byte).
rmsq_status qknorm_common(bool mx, const void *q_a, int64_t ld_q, const void *kv_a, int64_t ld_kv,
                          const void *gamma_q, const void *gamma_kv, float eps, int64_t M, int64_t Hq,
                          int64_t Hkv, int32_t group, void *out_q_q, void *out_q_scale, void *out_kv_q,
                          void *out_kv_scale, int32_t scale_layout, void *out_q_bf16, void *out_kv_bf16,
                          void *stream)
{
    const int64_t qb = mx ? 2 : 1;                      // elements per code byte
    const int64_t sb = mx ? 1 : 4;                      // bytes per scale
    rmsq_status st = check_single(q_a, ld_q, nullptr, 0, gamma_q, eps, M, Hq, group, out_q_q, Hq / qb,
                                  out_q_scale, (Hq / group) * M * sb, sb, nullptr, out_q_bf16);
    if (st != RMSQ_OK)
        return st;
    st = check_single(kv_a, ld_kv, nullptr, 0, gamma_kv, eps, M, Hkv, group, out_kv_q, Hkv / qb,
                      out_kv_scale, (Hkv / group) * M * sb, sb, nullptr, out_kv_bf16);
    if (st != RMSQ_OK)
        return st;
    if (M == 0)
        return ok();
    // the two latents' outputs must not overlap each other or the other's inputs
    Range a[4] = {mat_range(out_q_q, M, Hq / qb, Hq / qb, 1),
                  mat_range(out_q_scale, 1, (Hq / group) * M * sb, 0, 1), {0, 0}, {0, 0}};
    Range b[4] = {mat_range(out_kv_q, M, Hkv / qb, Hkv / qb, 1),
                  mat_range(out_kv_scale, 1, (Hkv / group) * M * sb, 0, 1), {0, 0}, {0, 0}};
    int na = 2, nb = 2;
    if (out_q_bf16)
        a[na++] = mat_range(out_q_bf16, M, Hq, Hq, 2);
    if (out_kv_bf16)
        b[nb++] = mat_range(out_kv_bf16, M, Hkv, Hkv, 2);
    Range in_q = mat_range(q_a, M, Hq, ld_q, 2), in_kv = mat_range(kv_a, M, Hkv, ld_kv, 2);
    Range g_q = mat_range(gamma_q, 1, Hq, Hq, 2), g_kv = mat_range(gamma_kv, 1, Hkv, Hkv, 2);
    for (int i = 0; i < na; ++i) {
        if (overlaps(a[i], in_kv) || overlaps(a[i], g_kv))
            return fail(RMSQ_ERR_INVALID_ARG, "a q_a output overlaps a kv_a input");
        for (int j = 0; j < nb; ++j)
            if (overlaps(a[i], b[j]))
                return fail(RMSQ_ERR_INVALID_ARG, "q_a and kv_a outputs overlap");
    }
    for (int j = 0; j < nb; ++j)
        if (overlaps(b[j], in_q) || overlaps(b[j], g_q))
            return fail(RMSQ_ERR_INVALID_ARG, "a kv_a output overlaps a q_a input");

    Seg sq = make_seg(q_a, ld_q, nullptr, 0, gamma_q, eps, M, Hq, out_q_q, out_q_scale,
                      scale_layout, nullptr, out_q_bf16);
    Seg sk = make_seg(kv_a, ld_kv, nullptr, 0, gamma_kv, eps, M, Hkv, out_kv_q, out_kv_scale,
                      scale_layout, nullptr, out_kv_bf16);
    debug_bind(sq, (Hq / group) * M);
    debug_bind(sk, (Hkv / group) * M);
    // Team shapes: the compiled-in MLA pair shape when it fits exactly,
    // otherwise one vectors-per-thread value for both latents, least padding
    // first.
    int v0 = 0, v1 = 0, tq = 0, tk = 0, t0s = 0, t1s = 0;
    const int gv = mx ? 4 : 16;
    if (Hq == 6 * 32 * 8 && Hkv == 4 * 16 * 8) {
        v0 = 6; tq = 32; v1 = 4; tk = 16; t0s = 32; t1s = 16;
    } else {
        int64_t best_waste = -1;
        for (int v : kVptPreference) {
            int a, b;
            int64_t wa, wb;
            if (team_ok(Hq / 8, v, gv, a, wa) && team_ok(Hkv / 8, v, gv, b, wb) &&
                (best_waste < 0 || wa + wb < best_waste)) {
                v0 = v1 = v;
                tq = a;
                tk = b;
                best_waste = wa + wb;
            }
        }
    }
    if (!v0)
        return fail(RMSQ_ERR_UNSUPPORTED, "no common team shape for Hq=%lld, Hkv=%lld",
                    (long long)Hq, (long long)Hkv);
    int threads = default_rows_per_block(tq) * tq;
    int tk_threads = default_rows_per_block(tk) * tk;
    if (tk_threads > threads)
        threads = tk_threads;
    // The latency form of the compiled pair shape when the launch can have at
    // most one block per SM: the smallest block (32 .. 256 threads) for which
    // it does, so that the rows spread over as many SMs as there are (64 tokens
    // in 96 blocks of one q_a row and two kv_a rows: 2.69 -> 2.24 us per call).
    bool lat = false;
    if (t0s) {
        for (int th = 32; th <= threads; th *= 2) {
            const int64_t nq = (M + th / tq - 1) / (th / tq), nk = (M + th / tk - 1) / (th / tk);
            if (nq + nk <= sm_count()) {
                threads = th;
                lat = true;
                break;
            }
        }
    }
    sq.tpr = tq;
    sk.tpr = tk;
    sq.rpb = threads / tq;
    sk.rpb = threads / tk;
    if ((tq > 32 && sq.rpb > 15) || (tk > 32 && sk.rpb > 15))
        return fail(RMSQ_ERR_UNSUPPORTED, "team shape needs too many named barriers");
    int64_t bq = (M + sq.rpb - 1) / sq.rpb, bk = (M + sk.rpb - 1) / sk.rpb;
    if (bq + bk > 0x7fffffff)
        return fail(RMSQ_ERR_UNSUPPORTED, "M too large");
    sq.blocks = (int32_t)bq;
    sk.blocks = (int32_t)bk;
    LaunchParams p{};
    p.seg[0] = sq;
    p.seg[1] = sk;
    p.nseg = 2;
    cudaError_t e = launch_dual(mx, lat, v0, t0s, v1, t1s, p, (int)(bq + bk), threads, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    return ok();
}

// MXFP4 single tensor, scales row-major (layout 0) or in the block-scaled MMA
// tile layout (layout 1: ceil(M/128) x ceil(H/128) tiles of 512 bytes).
rmsq_status mxfp4_common(const void *x, int64_t ld_x, const void *residual, int64_t ld_res,
                         const void *gamma, float eps, int64_t M, int64_t H, uint8_t *out_q,
                         uint8_t *out_scale, int layout, void *out_residual, void *out_bf16, void *stream,
                         const rmsq_launch_opts *opts)
{
    const int64_t ktiles = (H / 32 + 3) / 4;
    const int64_t sbytes = layout == 0 ? (H / 32) * M : (M + 127) / 128 * ktiles * 512;
    rmsq_status st = check_single(x, ld_x, residual, ld_res, gamma, eps, M, H, 32, out_q, H / 2,
                                  out_scale, sbytes, layout == 0 ? 1 : 16, out_residual, out_bf16);
    if (st != RMSQ_OK || M == 0)
        return st == RMSQ_OK ? ok() : st;
    Seg s = make_seg(x, ld_x, residual, ld_res, gamma, eps, M, H, out_q, out_scale, layout,
                     out_residual, out_bf16);
    s.scale_ld = ktiles;
    debug_bind(s, sbytes);
    return launch_single(s, true, opts ? *opts : kDefaultOpts, (cudaStream_t)stream);
}

}  // namespace

// Helpers shared with the GEMM's host code (rmsq_gemm.cu).
rmsq_status set_error(rmsq_status s, const char *msg) { return fail(s, "%s", msg); }
rmsq_status clear_error() { return ok(); }
int device_sm_count() { return sm_count(); }
unsigned int *device_status_word(int dev) { return status_word_ptr(dev); }

}  // namespace rmsq

using namespace rmsq;

extern "C" {

const char *rmsq_status_string(rmsq_status s)
{
    switch (s) {
    case RMSQ_OK: return "ok";
    case RMSQ_ERR_INVALID_ARG: return "invalid argument";
    case RMSQ_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
    case RMSQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case RMSQ_ERR_CUDA: return "CUDA error";
    case RMSQ_ERR_TIMEOUT: return "a bounded device wait timed out";
    case RMSQ_ERR_BOUNDS: return "a bounds check of the debug build failed";
    }
    return "unknown status";
}

const char *rmsq_last_error(void) { return g_last_error; }

rmsq_status rmsq_add_rmsnorm_quant_group_fp8_ex(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, int32_t group, void *out_q, float *out_scale,
    int32_t scale_layout, void *out_residual, void *out_bf16, void *stream,
    const rmsq_launch_opts *opts)
{
    if (group != 128)
        return fail(group > 0 ? RMSQ_ERR_UNSUPPORTED : RMSQ_ERR_INVALID_ARG,
                    "FP8 group must be 128 (got %d)", group);
    if (scale_layout != RMSQ_SCALE_ROW_MAJOR && scale_layout != RMSQ_SCALE_COL_MAJOR &&
        scale_layout != RMSQ_SCALE_COL_MAJOR_PAD4)
        return fail(RMSQ_ERR_INVALID_ARG, "unknown scale layout %d", scale_layout);
    const int64_t sld = scale_layout == RMSQ_SCALE_COL_MAJOR_PAD4 ? (M + 3) / 4 * 4 : M;
    rmsq_status st = check_single(x, ld_x, residual, ld_res, gamma, eps, M, H, group, out_q, H,
                                  out_scale, (H / group) * sld * 4,
                                  scale_layout == RMSQ_SCALE_COL_MAJOR_PAD4 ? 16 : 4, out_residual,
                                  out_bf16);
    if (st != RMSQ_OK || M == 0)
        return st == RMSQ_OK ? ok() : st;
    Seg s = make_seg(x, ld_x, residual, ld_res, gamma, eps, M, H, out_q, out_scale,
                     scale_layout == RMSQ_SCALE_ROW_MAJOR ? 0 : 1, out_residual, out_bf16);
    s.scale_ld = sld;
    debug_bind(s, (H / group) * sld);
    return launch_single(s, false, opts ? *opts : kDefaultOpts, (cudaStream_t)stream);
}

rmsq_status rmsq_add_rmsnorm_quant_group_fp8(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, int32_t group, void *out_q, float *out_scale,
    int32_t scale_layout, void *out_residual, void *out_bf16, void *stream)
{
    return rmsq_add_rmsnorm_quant_group_fp8_ex(x, ld_x, residual, ld_res, gamma, eps, M, H, group,
                                               out_q, out_scale, scale_layout, out_residual,
                                               out_bf16, stream, nullptr);
}

rmsq_status rmsq_add_rmsnorm_quant_mxfp4_ex(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale, void *out_residual,
    void *out_bf16, void *stream, const rmsq_launch_opts *opts)
{
    return mxfp4_common(x, ld_x, residual, ld_res, gamma, eps, M, H, out_q, out_scale, 0, out_residual,
                        out_bf16, stream, opts);
}

rmsq_status rmsq_add_rmsnorm_quant_mxfp4_mma_scales(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale_tiles, void *out_residual,
    void *out_bf16, void *stream)
{
    return mxfp4_common(x, ld_x, residual, ld_res, gamma, eps, M, H, out_q, out_scale_tiles, 1,
                        out_residual, out_bf16, stream, nullptr);
}

rmsq_status rmsq_add_rmsnorm_quant_mxfp4(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale, void *out_residual,
    void *out_bf16, void *stream)
{
    return rmsq_add_rmsnorm_quant_mxfp4_ex(x, ld_x, residual, ld_res, gamma, eps, M, H, out_q,
                                           out_scale, out_residual, out_bf16, stream, nullptr);
}

rmsq_status rmsq_qknorm_quant_fp8(
    const void *q_a, int64_t ld_q, const void *kv_a, int64_t ld_kv, const void *gamma_q,
    const void *gamma_kv, float eps, int64_t M, int64_t Hq, int64_t Hkv, int32_t group,
    void *out_q_q, float *out_q_scale, void *out_kv_q, float *out_kv_scale,
    int32_t scale_layout, void *out_q_bf16, void *out_kv_bf16, void *stream)
{
    if (group != 128)
        return fail(group > 0 ? RMSQ_ERR_UNSUPPORTED : RMSQ_ERR_INVALID_ARG,
                    "FP8 group must be 128 (got %d)", group);
    if (scale_layout != RMSQ_SCALE_ROW_MAJOR && scale_layout != RMSQ_SCALE_COL_MAJOR)
        return fail(RMSQ_ERR_INVALID_ARG, "unknown scale layout %d", scale_layout);
    return qknorm_common(false, q_a, ld_q, kv_a, ld_kv, gamma_q, gamma_kv, eps, M, Hq, Hkv, group,
                         out_q_q, out_q_scale, out_kv_q, out_kv_scale, scale_layout, out_q_bf16,
                         out_kv_bf16, stream);
}

rmsq_status rmsq_qknorm_quant_mxfp4(
    const void *q_a, int64_t ld_q, const void *kv_a, int64_t ld_kv, const void *gamma_q,
    const void *gamma_kv, float eps, int64_t M, int64_t Hq, int64_t Hkv, uint8_t *out_q_q,
    uint8_t *out_q_scale, uint8_t *out_kv_q, uint8_t *out_kv_scale, void *out_q_bf16,
    void *out_kv_bf16, void *stream)
{
    return qknorm_common(true, q_a, ld_q, kv_a, ld_kv, gamma_q, gamma_kv, eps, M, Hq, Hkv, 32,
                         out_q_q, out_q_scale, out_kv_q, out_kv_scale, RMSQ_SCALE_ROW_MAJOR, out_q_bf16,
                         out_kv_bf16, stream);
}

rmsq_status rmsq_add_rmsnorm(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, void *out_residual, void *out_bf16, void *stream)
{
    rmsq_status st = check_single(x, ld_x, residual, ld_res, gamma, eps, M, H, 32, nullptr, 0, nullptr, 0, 1,
                                  out_residual, out_bf16);
    if (st != RMSQ_OK || M == 0)
        return st == RMSQ_OK ? ok() : st;
    Seg s = make_seg(x, ld_x, residual, ld_res, gamma, eps, M, H, nullptr, nullptr, 0, out_residual,
                     out_bf16);
    debug_bind(s, 0);
    return launch_single(s, true, kDefaultOpts, (cudaStream_t)stream);
}

rmsq_status rmsq_sync_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess)
        return fail(RMSQ_ERR_CUDA, "synchronize failed: %s", cudaGetErrorString(e));
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
    if (e == cudaSuccess && word) {
        // clear exactly the bits just read, atomically on the device, so that
        // a bit another stream's kernel sets meanwhile is kept for the next read
        clear_status_bits_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(word);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = cudaStreamSynchronize((cudaStream_t)stream);
    }
    if (e != cudaSuccess)
        return fail(RMSQ_ERR_CUDA, "status word access failed: %s", cudaGetErrorString(e));
    if (word & 4u)
        return fail(RMSQ_ERR_BOUNDS, "a debug-build bounds check failed, the store was skipped (status 0x%x)", word);
    if (word & 8u)
        return fail(RMSQ_ERR_CUDA, "a GEMM kernel found its shared memory not 1024-byte aligned and wrote nothing "
                                   "(status 0x%x)", word);
    if (word)
        return fail(RMSQ_ERR_TIMEOUT, "a bounded wait gave up (status 0x%x)", word);
    return ok();
}

rmsq_status rmsq_debug_bounds_selftest(void *stream)
{
#ifdef RMSQ_DEBUG
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return fail(RMSQ_ERR_CUDA, "no current device");
    unsigned int *status = status_word_ptr(dev);
    if (!status)
        return fail(RMSQ_ERR_CUDA, "status word address unavailable");
    debug_bounds_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(status, 1);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ok() : fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
#else
    (void)stream;
    return fail(RMSQ_ERR_UNSUPPORTED, "the bounds checks exist only in the RMSQ_DEBUG build");
#endif
}

rmsq_status rmsq_encode_e4m3(const float *in, uint8_t *out, int64_t n, void *stream)
{
    if (n < 0 || (n && (!in || !out)))
        return fail(RMSQ_ERR_INVALID_ARG, "bad encoder arguments");
    if (n == 0)
        return ok();
    int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    encode_e4m3_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(in, out, n);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ok() : fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
}

rmsq_status rmsq_encode_e2m1(const float *in, uint8_t *out, int64_t n, void *stream)
{
    if (n < 0 || (n && (!in || !out)))
        return fail(RMSQ_ERR_INVALID_ARG, "bad encoder arguments");
    if (n == 0)
        return ok();
    int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    encode_e2m1_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(in, out, n);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ok() : fail(RMSQ_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
}

}  // extern "C"
