// Per-row body of the fused (add +) RMSNorm + group quant, shared by the
// register-resident row kernel and the persistent bulk-copy kernel.
//
// Layout of work: a row of H bf16 values is split into H/8 16-byte vectors;
// a team of `tpr` threads owns a row and thread t holds vectors
// k*tpr + t (k < VPT), so every load and store of a warp is a contiguous,
// coalesced span. tpr is a multiple of the group's vector count (16 for
// 1x128 FP8, 4 for MXFP4's 32), so a quant group is held by 16 (or 4)
// consecutive lanes at the same k and its amax is a 4- (or 2-) step xor
// shuffle. tpr is either a divisor of 32 (several rows per warp) or a
// multiple of 32 (rows spanning warps, combined through shared memory with a
// per-team named barrier). When tpr * VPT exceeds H/8 the team is padded:
// the vectors past the row end are whole groups (both counts are multiples
// of the group's vector count), read as zero and never stored.
//
// What a row computes (page "fused rmsnorm quant fp8 work", Motivation;
// sglang PR "[AMD] Add fused all-reduce RMSNorm per-group quant for Qwen3.5
// FP8", Modifications; ATOM PR "Support input_rmsnorm_quant & qknorm_quant
// fused for Atom dpsk v2 model", Technical Details):
//   r = bf16(x + residual)                     -> residual output
//   inv = f32(1 / sqrt(sum(r^2) / H + eps))
//   y = bf16((r * inv) * gamma)                -> optional bf16 output
//   FP8:   scale = amax_128(|y|) / 448, q = e4m3_satfinite(y / scale)
//   MXFP4: X = clamp(floor(log2 amax_32) - 2, -127, 127), byte X + 127,
//          q = e2m1_satfinite(y * 2^-X), two per byte, even element low.
#pragma once

#include "rmsq_device.cuh"
#include "rmsq_internal.h"

namespace rmsq {

struct RedSmem {
    float2 part[2][32];   // per-warp double-float partials, two parity sets
    float inv[2][16];     // per-team inv_rms (NaN: take the fp64 path), two parity sets
    double dpart[32][2];  // per-warp double-double partials for the wide-range path
};

__device__ __forceinline__ unsigned team_lane_mask(int tpr, int lane)
{
    if (tpr >= 32)
        return 0xffffffffu;
    unsigned m = (1u << tpr) - 1u;
    return m << (lane & ~(tpr - 1));
}

// Barrier over the `tpr` threads of one team (tpr a multiple of 32):
// named barrier 1 + team; barrier 0 stays with __syncthreads.
__device__ __forceinline__ void team_bar(int team, int tpr)
{
    asm volatile("bar.sync %0, %1;" ::"r"(team + 1), "r"(tpr) : "memory");
}

// Byte offset of the E8M0 scale of (row, group g) in the scale-factor layout
// that Blackwell's block-scaled MMA reads: 128-row x 4-group tiles of 512
// bytes, tiles ordered row-tile major with `ktiles` tiles per row tile; inside
// a tile, row r and group c sit at (r % 32) * 16 + (r / 32) * 4 + c, so the
// four groups of a row are adjacent and rows r, r+32, r+64, r+96 share a
// 16-byte line.
__device__ __forceinline__ int64_t mma_scale_offset(int64_t row, int64_t g, int64_t ktiles)
{
    const int64_t r = row & 127;
    return ((row >> 7) * ktiles + (g >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (g & 3);
}

// Team-wide fp64 sum of squares and fp64 finalisation, for rows whose sum
// lies outside the fp32 range in which the double-float path is exact.
//
// The squares of bf16 values are exact in fp64 (8-bit significands, and
// exponents from 2^-266 to 2^256 are all normal fp64). They are summed as a
// double-double: Knuth's TwoSum keeps each addition's rounding error in a
// second fp64 word, and the lane butterfly and the cross-warp step add
// double-doubles the same way. Before its one rounding to fp64 the sum is
// within n^2 * 2^-106 (relative; below 2^-76 for the widest row) of the exact
// one, so the result is the correctly rounded sum that the oracle's
// compensated summation gives, except in rows whose exact sum lies that close
// to an fp64 rounding midpoint.
__device__ __forceinline__ void two_sum_f64(double a, double b, double &s, double &e)
{
    s = __dadd_rn(a, b);
    const double bb = __dsub_rn(s, a);
    e = __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb));
}

// (hi, lo) += (bhi, blo): the high words exactly, the errors into the low
// word. Commutative bit for bit (TwoSum's error is the exact rounding error
// of the sum, whichever operand comes first), so a butterfly leaves the same
// value in every lane.
__device__ __forceinline__ void dd_add(double &hi, double &lo, double bhi, double blo)
{
    double s, e;
    two_sum_f64(hi, bhi, s, e);
    hi = s;
    lo = __dadd_rn(__dadd_rn(lo, blo), e);
}

template <int VPT>
__device__ __forceinline__ float inv_rms_fp64_path(const uint4 (&r)[VPT], int H, float eps, int tpr,
                                                   int team, RedSmem &red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned tmask = team_lane_mask(tpr, lane);
    double hi = 0.0, lo = 0.0;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const uint32_t w[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const double a = (double)bf_lo(w[j]), b = (double)bf_hi(w[j]);
            double s, e;
            two_sum_f64(hi, __dmul_rn(a, a), s, e);
            lo = __dadd_rn(lo, e);
            two_sum_f64(s, __dmul_rn(b, b), hi, e);
            lo = __dadd_rn(lo, e);
        }
    }
    const int wlim = tpr < 32 ? tpr : 32;
    for (int off = 1; off < wlim; off <<= 1) {
        const double ohi = __shfl_xor_sync(tmask, hi, off), olo = __shfl_xor_sync(tmask, lo, off);
        dd_add(hi, lo, ohi, olo);
    }
    if (tpr > 32) {
        const int nw = tpr >> 5, w0 = team * nw;
        if (lane == 0) {
            red.dpart[warp][0] = hi;
            red.dpart[warp][1] = lo;
        }
        team_bar(team, tpr);
        hi = red.dpart[w0][0];
        lo = red.dpart[w0][1];
        for (int i = 1; i < nw; ++i)
            dd_add(hi, lo, red.dpart[w0 + i][0], red.dpart[w0 + i][1]);
        team_bar(team, tpr);
    }
    const double S = __dadd_rn(hi, lo);
    return (float)(1.0 / sqrt(S / (double)H + (double)eps));
}

// inv_rms of a team's row from the per-thread double-float partials of its
// sum of squares; the same value in every thread of the team. Within a warp
// an xor butterfly (bit-identical in every lane). For teams wider than a
// warp, lane 0 of each warp publishes its partial; the team's first warp
// alone combines them (butterfly over the next power of two) and finalises,
// and the result is broadcast through shared memory. `parity` alternates
// the shared slots between consecutive rows of a persistent team. A NaN
// result means the sum left the double-float range: the caller takes the
// fp64 path.
//
// LAT (latency form, for launches of one row per SM or fewer): every warp of
// the team reads all the partials after the one barrier and combines them
// itself, in the same fixed butterfly (its lane 0 finalises and shuffles the
// result to the warp), so the result is bit-identical to the throughput
// form's and the second barrier and its shared-memory broadcast leave the
// row's critical path. It needs no second slot set: a team's
// slots are written once per launch (row kernel only).
template <int TPR, bool LAT = false>
__device__ __forceinline__ float team_inv_rms(DF S, const Seg &s, int tpr, int team, int parity,
                                              RedSmem &red, unsigned tmask)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
        if (off < tpr)
            S = df_add_lazy(S, shfl_xor_df(S, off, tmask));
    float inv;
    if (tpr <= 32) {
        if (!inv_rms_df(df_renorm(S), s.H, s.inv_h, s.eps, inv))
            inv = __int_as_float(0x7fffffff);
        return inv;
    }
    const int nw = tpr >> 5, w0 = team * nw;
    if (lane == 0)
        red.part[parity][warp] = make_float2(S.hi, S.lo);
    team_bar(team, tpr);
    if (LAT || warp == w0) {
        const float2 p = lane < nw ? red.part[parity][w0 + lane] : make_float2(0.0f, 0.0f);
        DF T{p.x, p.y};
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
            if (off < nw)
                T = df_add_lazy(T, shfl_xor_df(T, off, 0xffffffffu));
        if (LAT) {
            // the butterfly spans the next power of two above nw lanes only:
            // lane 0 holds the team's sum, so it finalises and every lane
            // takes its value
            if (!inv_rms_df(df_renorm(T), s.H, s.inv_h, s.eps, inv))
                inv = __int_as_float(0x7fffffff);
            return __shfl_sync(0xffffffffu, inv, 0);
        }
        if (lane == 0) {
            if (!inv_rms_df(df_renorm(T), s.H, s.inv_h, s.eps, inv))
                inv = __int_as_float(0x7fffffff);
            red.inv[parity][team] = inv;
        }
    }
    team_bar(team, tpr);
    return red.inv[parity][team];
}

// Where row_finish takes gamma from: through the read-only cache when the
// row is normalised, from shared memory (staged by the persistent kernel), or
// from registers loaded together with the row (latency form).
enum GammaFrom { GAMMA_GLOBAL = 0, GAMMA_SHARED = 1, GAMMA_REGS = 2 };

// Vector j of part `part` of a thread's VPT vectors cut into SPLIT parts of
// VPT / SPLIT (k = part * VPT / SPLIT + j), chosen by selects so that the
// array stays in registers (part is known only at run time).
template <int SPLIT, int VPT>
__device__ __forceinline__ uint4 part_vec(const uint4 (&a)[VPT], int part, int j)
{
    constexpr int NV = VPT / SPLIT;
    uint4 v = a[j];
#pragma unroll
    for (int p = 1; p < SPLIT; ++p)
        if (part == p)
            v = a[p * NV + j];
    return v;
}

// Everything after the row is loaded: r holds the thread's VPT vectors of
// bf16 r (residual already added and written back by the caller). gamma
// comes from gamma_src (GAMMA_GLOBAL, GAMMA_SHARED) or gpre (GAMMA_REGS, the
// thread's own vectors of this part). TPR is the team size when known at
// compile time (the row is then an exact fit, tpr * VPT * 8 == H), or 0 for a
// runtime team size with padding guards. LAT selects team_inv_rms's latency
// form. SPLIT > 1 (latency form only): the row's outputs are shared by SPLIT
// blocks; each reduces the whole row (the same sum in the same order, so the
// same inv_rms) and normalises, quantises and stores only its part `part`,
// vectors k = part * VPT / SPLIT .. of each thread. Elementwise arithmetic
// runs on packed fp32 pairs.
template <int VPT, int TPR, bool MX, int GFROM, bool LAT = false, int SPLIT = 1>
__device__ __forceinline__ void row_finish(const Seg &s, int64_t row, int t, int team, int parity,
                                           RedSmem &red, const uint4 (&r)[VPT],
                                           const uint4 *gamma_src, const uint4 (&gpre)[VPT / SPLIT],
                                           int part = 0)
{
    constexpr int GV = MX ? 4 : 16;   // 16-byte vectors per quant group
    constexpr bool GUARD = TPR == 0;
    constexpr int NV = VPT / SPLIT;   // vectors of this block's part, per thread
    static_assert(VPT % SPLIT == 0 && (SPLIT == 1 || (LAT && GFROM == GAMMA_REGS)), "split rows");
    const int tpr = TPR ? TPR : s.tpr;
    const int lane = threadIdx.x & 31;
    const unsigned tmask = team_lane_mask(tpr, lane);
    const int nvec = TPR ? TPR * VPT : (s.H >> 3);
    const int kb = part * NV;         // first vector (k) of the part

    // ---- sum of squares: exact squares, two packed double-float accumulators
    float2 hi = f2(0.0f), lo = f2(0.0f);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        acc_square2(unpack_bf16x2(r[k].x), hi, lo);
        acc_square2(unpack_bf16x2(r[k].y), hi, lo);
        acc_square2(unpack_bf16x2(r[k].z), hi, lo);
        acc_square2(unpack_bf16x2(r[k].w), hi, lo);
    }
    float inv = team_inv_rms<TPR, LAT>(df_add_lazy(DF{hi.x, lo.x}, DF{hi.y, lo.y}), s, tpr, team, parity, red,
                                  tmask);
    if (inv != inv)                                   // team-uniform: NaN asks for the fp64 path
        inv = inv_rms_fp64_path<VPT>(r, s.H, s.eps, tpr, team, red);
    const float2 inv2 = f2(inv);

    // ---- normalise: y = bf16((r * inv) * gamma), this part's vectors
    uint4 y[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vk = (kb + k) * tpr + t;
        const uint4 g = (GUARD && vk >= nvec) ? make_uint4(0, 0, 0, 0)
                        : GFROM == GAMMA_REGS ? gpre[k]
                        : GFROM == GAMMA_SHARED ? gamma_src[vk] : ld_keep(gamma_src + vk);
        const uint4 rk = SPLIT == 1 ? r[k] : part_vec<SPLIT>(r, part, k);
        const uint32_t rw[4] = {rk.x, rk.y, rk.z, rk.w};
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t yw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 v = mul2(mul2(unpack_bf16x2(rw[j]), inv2), unpack_bf16x2(gw[j]));
            yw[j] = pack_bf16x2(v.x, v.y);
        }
        y[k] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
    }
    if (s.out_bf16) {
        uint4 *yrow = s.out_bf16 + row * nvec + t;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vk = (kb + k) * tpr + t;
            if ((!GUARD || vk < nvec) && RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && vk < nvec))
                yrow[(kb + k) * tpr] = y[k];
        }
    }
    if (!s.out_q)   // norm only (rmsq_add_rmsnorm)
        return;

    // ---- group amax over GV lanes (two vectors packed per shuffle)
    uint32_t am[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k)
        am[k] = amax_bits_bf16x8(y[k]);
#pragma unroll
    for (int k = 0; k < NV; k += 2) {
        uint32_t v = am[k] | ((k + 1 < NV) ? (am[k + 1] << 16) : 0u);
#pragma unroll
        for (int off = 1; off < GV; off <<= 1)
            v = max_u16x2(v, __shfl_xor_sync(tmask, v, off));
        am[k] = v & 0xffffu;
        if (k + 1 < NV)
            am[k + 1] = v >> 16;
    }

    // ---- quantise and store
    const bool leader = (t & (GV - 1)) == 0;
    if constexpr (!MX) {
        // Every group's scale and divisor first, then the quotients of all
        // vectors in one pass without control flow between them (the
        // divisions of different vectors are independent and interleave):
        // the direct IEEE division is kept for the rare groups whose scale
        // is too small for the reciprocal method.
        float scl[NV];
        GroupDivisor gd[NV];
        bool fast = true;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            scl[k] = div448(__uint_as_float(am[k] << 16));
            gd[k] = make_group_divisor(am[k] ? scl[k] : 1.0f);   // all-zero group: codes of +-0
            fast = fast && gd[k].fast;
        }
        if (leader) {
            const int64_t G = s.H >> 7;
            float *sc = (float *)s.out_scale;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int v = (kb + k) * tpr + t;
                if (GUARD && v >= nvec)
                    continue;                // padding of the team shape (whole groups)
                const int64_t g = v >> 4;
                const int64_t si = s.layout == 0 ? row * G + g : g * s.scale_ld + row;
                if (RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && si < s.scale_elems))
                    sc[si] = scl[k];
            }
        }
        uint2 *qrow = reinterpret_cast<uint2 *>(s.out_q + row * (int64_t)s.H);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = (kb + k) * tpr + t;   // vector index in the row
            if (GUARD && v >= nvec)
                continue;
            const uint32_t yw[4] = {y[k].x, y[k].y, y[k].z, y[k].w};
            float2 qv[4];
            if (fast || gd[k].fast) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    qv[j] = div_fast_neg2(unpack_neg_bf16x2(yw[j]), gd[k]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    qv[j] = make_float2(__fdiv_rn(bf_lo(yw[j]), gd[k].d), __fdiv_rn(bf_hi(yw[j]), gd[k].d));
            }
            if (RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && v < nvec))
                qrow[v] = make_uint2(e4m3x4(qv[0], qv[1]), e4m3x4(qv[2], qv[3]));
        }
    } else {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = (kb + k) * tpr + t;   // vector index in the row
            if (GUARD && v >= nvec)
                continue;                // padding of the team shape (whole groups)
            const uint32_t yw[4] = {y[k].x, y[k].y, y[k].z, y[k].w};
            const int X = mx_exponent_from_bits(am[k]);
            const float2 mult = f2(__uint_as_float((uint32_t)(127 - X) << 23));   // 2^-X
            if (leader) {
                uint8_t *sc = (uint8_t *)s.out_scale;
                const int64_t g = v >> 2;
                const int64_t si =
                    s.layout == 0 ? row * (int64_t)(s.H >> 5) + g : mma_scale_offset(row, g, s.scale_ld);
                if (RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && si < s.scale_elems))
                    sc[si] = (uint8_t)(X + 127);
            }
            if (RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && v < nvec))
                reinterpret_cast<uint32_t *>(s.out_q + row * (int64_t)(s.H >> 1))[v] =
                    e2m1x8(mul2(unpack_bf16x2(yw[0]), mult), mul2(unpack_bf16x2(yw[1]), mult),
                           mul2(unpack_bf16x2(yw[2]), mult), mul2(unpack_bf16x2(yw[3]), mult));
        }
    }
}

// Load (and add) one row from global memory, write the residual, finish it.
// LAT (latency form): gamma is loaded together with the row, so that its
// load latency overlaps the row's instead of following the reduction. SPLIT
// (latency form only): this block owns part `part` of the row's outputs,
// residual included, but loads and adds the whole row for its sum of squares.
template <int VPT, int TPR, bool MX, bool LAT = false, int SPLIT = 1>
__device__ __forceinline__ void row_from_global(const Seg &s, int64_t row, int t, int team, int parity,
                                                RedSmem &red, int part = 0)
{
    constexpr bool GUARD = TPR == 0;
    constexpr int NV = VPT / SPLIT;
    const int tpr = TPR ? TPR : s.tpr;
    const int nvec = TPR ? TPR * VPT : (s.H >> 3);
    uint4 r[VPT], g[NV];
    const uint4 *xr = s.x + row * s.ldx_v + t;
    // vectors past the row end (padded team shapes) read as zero and are
    // never stored; they add nothing to the sum of squares
    if (s.res) {
        const uint4 *rr = s.res + row * s.ldres_v + t;
        uint4 xv[VPT], rv[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const bool ok = !GUARD || k * tpr + t < nvec;
            xv[k] = ok ? ld_stream(xr + k * tpr) : make_uint4(0, 0, 0, 0);
            rv[k] = ok ? ld_stream(rr + k * tpr) : make_uint4(0, 0, 0, 0);
        }
        uint4 *orow = s.out_res + row * nvec + t;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            r[k] = add_bf16x8(xv[k], rv[k]);
            if ((SPLIT == 1 || k / NV == part) && (!GUARD || k * tpr + t < nvec) &&
                RMSQ_IN_BOUNDS(s.debug_flag, row < s.M && k * tpr + t < nvec))
                orow[k * tpr] = r[k];
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const bool ok = !GUARD || k * tpr + t < nvec;
            r[k] = ok ? ld_stream(xr + k * tpr) : make_uint4(0, 0, 0, 0);
        }
    }
    if constexpr (LAT) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vk = (part * NV + k) * tpr + t;
            g[k] = (!GUARD || vk < nvec) ? ld_keep(s.gamma + vk) : make_uint4(0, 0, 0, 0);
        }
        row_finish<VPT, TPR, MX, GAMMA_REGS, true, SPLIT>(s, row, t, team, parity, red, r, s.gamma, g, part);
    } else {
        static_assert(SPLIT == 1, "split rows exist in the latency form only");
        row_finish<VPT, TPR, MX, GAMMA_GLOBAL>(s, row, t, team, parity, red, r, s.gamma, g);
    }
}

}  // namespace rmsq
