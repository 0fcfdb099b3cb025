/*
 * rmsq_oracle.c -- plain, slow CPU definition of the fused
 * (residual add +) RMSNorm + per-token-group activation quantisation.
 *
 * TEST INFRASTRUCTURE. This file is the oracle the CUDA path is checked
 * against. Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg load it; the product library never calls it,
 * and the two share no code, header, table or constant.
 *
 * It is written as the UNFUSED composition of the separate kernels the
 * fusion replaces -- residual add, RMSNorm, per-group dynamic quant -- one
 * plain function each, in that order (sglang PR "[AMD] Add fused all-reduce
 * RMSNorm per-group quant for Qwen3.5 FP8": Motivation, Fallback order item 2,
 * and the kernel-count table rows add_rmsnorm_quant_kernel and
 * dynamic_per_group_scaled_quant_kernel).
 *
 * Per row of H bf16 values (bf16 decodes exactly to fp32):
 *   1. add:   r_i = bf16_rne(f32(x_i) + f32(res_i)); r is the residual output
 *             (the "residual" member of the ((fp8, scale), residual) tuple,
 *             same PR, Modifications).
 *   2. norm:  S = sum r_i^2 in fp64 (every square is exact in fp64; Neumaier
 *             compensated summation), inv = f32(1 / sqrt(S / H + eps)) with
 *             fp64 IEEE divide and sqrt and one final rounding to fp32,
 *             y_i = bf16_rne((f32(r_i) * inv) * f32(gamma_i)), two fp32
 *             multiplies in that order, no fused multiply-add. y is the bf16
 *             side output ("keep_bf16", (bf16, fp8, scale), same PR).
 *   3a. FP8 group quant, group G = 128 (one FP8 scale per 128 elements:
 *             page "fused rmsnorm quant fp8 work", Motivation): amax =
 *             max |y_i| over the group, scale = f32(amax / 448) by IEEE
 *             fp32 division, q_i =
 *             e4m3(f32(y_i / scale)) by IEEE fp32 division by the stored
 *             scale followed by the saturating round-to-nearest-even E4M3
 *             encoder (OCP 8-bit floating point, E4M3, largest finite 448).
 *   3b. MXFP4 group quant, group 32 (ATOM PR "Support input_rmsnorm_quant &
 *             qknorm_quant fused for Atom dpsk v2 model", Technical Details:
 *             "fused RMSNorm+MXFP4 quant"): X = clamp(floor(log2(amax)) - 2,
 *             -127, 127), scale byte = X + 127 (E8M0), elements
 *             e2m1_rne_sat(y_i * 2^-X), two per byte, even element in the low
 *             nibble (OCP Microscaling Formats v1.0, MXFP4).
 *   4. consumer GEMM: D = A B^T on MXFP4 operands (activation A from 3b,
 *             weights B), fp64 exact sum, fp32 accumulator reading, bf16
 *             output; see the GEMM section below for its citation.
 *   qknorm:   steps 2 and 3a applied separately to the MLA q_a and kv_a
 *             latents with their own gammas and no residual (page "fused
 *             rmsnorm quant fp8 work", Modifications, "DeepseekV2AttentionMLA
 *             (for q, k_)"; ATOM PR, Technical Details, "qknorm quant").
 *
 * Readings where the pages are silent (each repeated in the design notes):
 *   - the norm uses the bf16-rounded r, the value the add kernel writes;
 *   - the quantiser reads the bf16 y, the value the unfused quant kernel
 *     would read from memory;
 *   - an all-zero group (amax == 0) gets scale 0.0f and codes that keep the
 *     sign of the zero input (the quotient 0/0 is not formed); MXFP4 gives
 *     scale byte 0x00 and zero codes;
 *   - signed zeros keep their sign in both encoders;
 *   - NaN and Inf inputs are outside the workloads; the encoders map NaN to
 *     the E4M3 NaN code and Inf to the largest finite value.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math). pthreads
 * split rows into contiguous ranges; every row is computed the same way
 * whatever the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to bf16, nearest, ties to even; NaN stays a quiet NaN. */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------- encoders */

/* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite 448 (0x7E); subnormals are k * 2^-9. */
uint8_t oracle_e4m3_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(v))
        return (uint8_t)(sign | 0x7f);
    double a = fabs((double)v);
    if (a > 448.0) /* saturate: every value above 448 (and Inf) -> 448 */
        return (uint8_t)(sign | 0x7e);
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: spacing 2^-9; n may round up to 8, the first
         * normal code, which is the right answer there */
        code = (int)nearbyint(a * 512.0);
    } else {
        int e2;
        frexp(a, &e2);        /* a = f * 2^e2, f in [0.5, 1) */
        int e = e2 - 1;       /* floor(log2 a), exact */
        double n = nearbyint(ldexp(a, 3 - e)); /* in [8, 16] */
        code = ((e + 7) << 3) + ((int)n - 8);  /* n == 16 carries into e+1 */
    }
    if (code > 0x7e)
        code = 0x7e;
    return (uint8_t)(sign | code);
}

float oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (e == 0xf && m == 7)
        return s ? -NAN : NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + m, e - 7 - 3);
    return (float)(s ? -v : v);
}

/* OCP E2M1 (MXFP4 element): values 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign bit 3.
 * Round to nearest, ties to the even code, saturate to 6. */
uint8_t oracle_e2m1_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 31) << 3);
    if (isnan(v))
        return (uint8_t)(sign | 0x7);
    double a = fabs((double)v);
    int code;
    if (a >= 6.0) {
        code = 7;
    } else if (a < 1.0) {
        code = (int)nearbyint(2.0 * a);        /* 0, 0.5 or 1.0 -> codes 0..2 */
    } else {
        int e2;
        frexp(a, &e2);
        int e = e2 - 1;                        /* 0, 1 or 2 */
        double n = nearbyint(ldexp(a, 1 - e)); /* in [2, 4] */
        code = 2 * (e + 1) + ((int)n - 2);
        if (code > 7)
            code = 7;
    }
    return (uint8_t)(sign | code);
}

float oracle_e2m1_decode(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (float)(s ? -v : v);
}

/* Shared MX exponent of a group from its amax: X = clamp(floor(log2 amax) - 2,
 * -127, 127), so that amax * 2^-X lies in [4, 8) (E2M1's largest power of
 * two is 4). amax == 0 gives X = -127. Returned as the unbiased exponent. */
int oracle_mx_exponent(float amax)
{
    if (!(amax > 0.0f))
        return -127;
    int e2;
    frexp((double)amax, &e2);
    int X = (e2 - 1) - 2;
    if (X < -127)
        X = -127;
    if (X > 127)
        X = 127;
    return X;
}

/* ------------------------------------------------------- row threading */

typedef void (*row_range_fn)(void *ctx, int64_t m0, int64_t m1);

typedef struct {
    row_range_fn fn;
    void *ctx;
    int64_t m0, m1;
} row_job;

static void *row_job_run(void *p)
{
    row_job *j = (row_job *)p;
    j->fn(j->ctx, j->m0, j->m1);
    return NULL;
}

static void for_rows(row_range_fn fn, void *ctx, int64_t M, int nthreads)
{
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads <= 1 || M < 2) {
        fn(ctx, 0, M);
        return;
    }
    if ((int64_t)nthreads > M)
        nthreads = (int)M;
    pthread_t th[256];
    row_job jobs[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].m0 = M * t / nthreads;
        jobs[t].m1 = M * (t + 1) / nthreads;
        started[t] = pthread_create(&th[t], NULL, row_job_run, &jobs[t]) == 0;
        if (!started[t])
            row_job_run(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t])
            pthread_join(th[t], NULL);
}

/* ----------------------------------------------------- 1. residual add */

typedef struct {
    const uint16_t *x, *res;
    int64_t ldx, ldres, H;
    uint16_t *r;
    int64_t ldr;
} add_ctx;

static void add_rows(void *p, int64_t m0, int64_t m1)
{
    add_ctx *c = (add_ctx *)p;
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t i = 0; i < c->H; ++i) {
            float s = bf16_to_f32(c->x[m * c->ldx + i]) + bf16_to_f32(c->res[m * c->ldres + i]);
            c->r[m * c->ldr + i] = f32_to_bf16_rne(s);
        }
}

/* r = bf16(x + residual), row by row. */
int oracle_add_residual(const uint16_t *x, int64_t ldx, const uint16_t *res, int64_t ldres,
                        int64_t M, int64_t H, uint16_t *r, int64_t ldr, int nthreads)
{
    if (!x || !res || !r || M < 0 || H < 0)
        return -1;
    add_ctx c = {x, res, ldx, ldres, H, r, ldr};
    for_rows(add_rows, &c, M, nthreads);
    return 0;
}

/* ---------------------------------------------------------- 2. RMSNorm */

typedef struct {
    const uint16_t *r, *gamma;
    int64_t ldr, H;
    float eps;
    uint16_t *y;
    int64_t ldy;
    float *inv;
    double *margin;
} norm_ctx;

static void norm_rows(void *p, int64_t m0, int64_t m1)
{
    norm_ctx *c = (norm_ctx *)p;
    for (int64_t m = m0; m < m1; ++m) {
        const uint16_t *row = c->r + m * c->ldr;
        /* Neumaier's compensated sum of the exact squares */
        double sum = 0.0, comp = 0.0;
        for (int64_t i = 0; i < c->H; ++i) {
            double v = (double)bf16_to_f32(row[i]);
            double sq = v * v;
            double t = sum + sq;
            if (fabs(sum) >= fabs(sq))
                comp += (sum - t) + sq;
            else
                comp += (sq - t) + sum;
            sum = t;
        }
        double S = sum + comp;
        double t64 = 1.0 / sqrt(S / (double)c->H + (double)c->eps);
        float inv = (float)t64;
        if (c->inv)
            c->inv[m] = inv;
        if (c->margin) {
            /* relative distance of the fp64 value from the nearest point at
             * which its fp32 rounding would change */
            double up = (double)nextafterf(inv, INFINITY);
            double dn = (double)nextafterf(inv, 0.0f);
            double mid_up = 0.5 * ((double)inv + up);
            double mid_dn = 0.5 * ((double)inv + dn);
            c->margin[m] = fmin(fabs(t64 - mid_up), fabs(t64 - mid_dn)) / t64;
        }
        for (int64_t i = 0; i < c->H; ++i) {
            float a = bf16_to_f32(row[i]) * inv;
            float b = a * bf16_to_f32(c->gamma[i]);
            c->y[m * c->ldy + i] = f32_to_bf16_rne(b);
        }
    }
}

/* y = bf16((r * inv_rms) * gamma); optionally the per-row fp32 inv_rms and
 * the relative margin of its fp64 value to the nearest fp32 rounding
 * boundary. */
int oracle_rmsnorm(const uint16_t *r, int64_t ldr, const uint16_t *gamma, float eps,
                   int64_t M, int64_t H, uint16_t *y, int64_t ldy, float *inv, double *margin,
                   int nthreads)
{
    if (!r || !gamma || !y || M < 0 || H <= 0)
        return -1;
    norm_ctx c = {r, gamma, ldr, H, eps, y, ldy, inv, margin};
    for_rows(norm_rows, &c, M, nthreads);
    return 0;
}

/* ----------------------------------------------- 3a. FP8 group quant */

/* Scale layouts: row-major [M, H/G]; column-major [H/G, M]; column-major with
 * the leading dimension M rounded up to a multiple of 4 (padding untouched). */
enum { ORACLE_SCALE_ROW_MAJOR = 0, ORACLE_SCALE_COL_MAJOR = 1, ORACLE_SCALE_COL_MAJOR_PAD4 = 2 };

typedef struct {
    const uint16_t *y;
    int64_t ldy, M, H, G;
    int layout;
    uint8_t *q;
    int64_t ldq;
    float *scale;
} fp8q_ctx;

static void fp8q_rows(void *p, int64_t m0, int64_t m1)
{
    fp8q_ctx *c = (fp8q_ctx *)p;
    int64_t ngroups = c->H / c->G;
    for (int64_t m = m0; m < m1; ++m) {
        const uint16_t *row = c->y + m * c->ldy;
        for (int64_t g = 0; g < ngroups; ++g) {
            float amax = 0.0f;
            for (int64_t i = g * c->G; i < (g + 1) * c->G; ++i) {
                float a = fabsf(bf16_to_f32(row[i]));
                if (a > amax)
                    amax = a;
            }
            float scale = amax / 448.0f;
            if (c->layout == ORACLE_SCALE_ROW_MAJOR)
                c->scale[m * ngroups + g] = scale;
            else if (c->layout == ORACLE_SCALE_COL_MAJOR)
                c->scale[g * c->M + m] = scale;
            else
                c->scale[g * ((c->M + 3) / 4 * 4) + m] = scale;
            for (int64_t i = g * c->G; i < (g + 1) * c->G; ++i) {
                float v = bf16_to_f32(row[i]);
                float quot = (amax == 0.0f) ? v : v / scale;
                c->q[m * c->ldq + i] = oracle_e4m3_encode(quot);
            }
        }
    }
}

/* Per-group dynamic FP8 quant of the bf16 y: scale = amax/448 stored at
 * [m*(H/G)+g] (row-major) or [g*M+m] (column-major); q = e4m3(y/scale). */
int oracle_group_quant_fp8(const uint16_t *y, int64_t ldy, int64_t M, int64_t H, int64_t G,
                           int layout, uint8_t *q, int64_t ldq, float *scale, int nthreads)
{
    if (!y || !q || !scale || M < 0 || H <= 0 || G <= 0 || H % G != 0)
        return -1;
    if (layout != ORACLE_SCALE_ROW_MAJOR && layout != ORACLE_SCALE_COL_MAJOR &&
        layout != ORACLE_SCALE_COL_MAJOR_PAD4)
        return -1;
    fp8q_ctx c = {y, ldy, M, H, G, layout, q, ldq, scale};
    for_rows(fp8q_rows, &c, M, nthreads);
    return 0;
}

/* ---------------------------------------------- 3b. MXFP4 group quant */

typedef struct {
    const uint16_t *y;
    int64_t ldy, H;
    uint8_t *q;
    int64_t ldq;
    uint8_t *scale;
    int64_t ldscale;
} mxq_ctx;

static void mxq_rows(void *p, int64_t m0, int64_t m1)
{
    mxq_ctx *c = (mxq_ctx *)p;
    const int64_t G = 32;
    for (int64_t m = m0; m < m1; ++m) {
        const uint16_t *row = c->y + m * c->ldy;
        for (int64_t g = 0; g < c->H / G; ++g) {
            float amax = 0.0f;
            for (int64_t i = g * G; i < (g + 1) * G; ++i) {
                float a = fabsf(bf16_to_f32(row[i]));
                if (a > amax)
                    amax = a;
            }
            int X = oracle_mx_exponent(amax);
            c->scale[m * c->ldscale + g] = (uint8_t)(X + 127);
            for (int64_t i = g * G; i < (g + 1) * G; i += 2) {
                uint8_t lo = oracle_e2m1_encode(ldexpf(bf16_to_f32(row[i]), -X));
                uint8_t hi = oracle_e2m1_encode(ldexpf(bf16_to_f32(row[i + 1]), -X));
                c->q[m * c->ldq + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* MXFP4 quant of the bf16 y: q [M, H/2] packed e2m1 pairs, scale [M, H/32]
 * E8M0 bytes (row-major). */
int oracle_group_quant_mxfp4(const uint16_t *y, int64_t ldy, int64_t M, int64_t H,
                             uint8_t *q, int64_t ldq, uint8_t *scale, int64_t ldscale,
                             int nthreads)
{
    if (!y || !q || !scale || M < 0 || H <= 0 || H % 32 != 0)
        return -1;
    mxq_ctx c = {y, ldy, H, q, ldq, scale, ldscale};
    for_rows(mxq_rows, &c, M, nthreads);
    return 0;
}

/* ------------------------------------ MXFP4 scales in MMA tile layout */

/* Re-lays a row-major [M, G] matrix of E8M0 scale bytes into the layout that
 * Blackwell's block-scaled MMA reads scale factors from (NVIDIA PTX ISA,
 * tcgen05 block scaling; cuBLAS, "1D block scaling factors layout"): tiles of
 * 128 rows x 4 groups (512 bytes), stored row-tile major with ceil(G/4)
 * tiles per row tile; inside a tile, row r and group c at
 * (r % 32) * 16 + (r / 32) * 4 + c. Padding bytes of partial tiles are left
 * as they are. */
int oracle_mx_scale_tiles(const uint8_t *s, int64_t M, int64_t G, uint8_t *out)
{
    if (!s || !out || M < 0 || G <= 0)
        return -1;
    int64_t ktiles = (G + 3) / 4;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t g = 0; g < G; ++g) {
            int64_t tile = (m / 128) * ktiles + g / 4;
            int64_t r = m % 128, c = g % 4;
            out[tile * 512 + (r % 32) * 16 + (r / 32) * 4 + c] = s[m * G + g];
        }
    return 0;
}

/* ------------------------------------- 4. consumer GEMM on MXFP4 data */

/* The GEMM that consumes the quantised activations: the MLA / MoE
 * projections of the DeepSeek models run as "A16W-FP4" GEMMs whose
 * activation operand is quantised to MXFP4 either by the fused norm + quant
 * kernel before the GEMM or in the GEMM itself ("prequant"; ATOM PR
 * "Triton fusion/GEMM optimizations for DS FP4 and FP8": the required AITER
 * PR list, "Triton A16WFP4 GEMM prequant", and the environment-variable
 * notes that pick one placement or the other by concurrency).
 *
 * Both operands are MXFP4 along K (OCP Microscaling Formats v1.0: blocks of
 * 32 E2M1 elements sharing one E8M0 scale 2^(byte - 127)); a [M, K/2] and
 * b [N, K/2] are row-major packed codes (even element in the low nibble),
 * sa [M, K/32] and sb [N, K/32] row-major scale bytes. The result is
 *   D[m][n] = sum_k dec(a[m][k]) 2^(sa[m][k/32]-127) dec(b[n][k]) 2^(sb[n][k/32]-127),
 * i.e. a times b transposed, both "K-major" as the weights of a linear layer
 * are stored. Every term is exact in fp64 (E2M1 values have two significant
 * bits); the sum is Neumaier-compensated, so d64 is the exact sum rounded
 * once to fp64 unless the terms span more than ~100 binades. Reading adopted
 * where the pages give no precision: an fp32 accumulator, so the bf16 output
 * is bf16_rne(f32(d64)). abs64 receives sum_k |term| (the scale of the
 * accumulation error any fp32 summation order can make). d64, abs64 and
 * dbf16 may each be NULL. */
typedef struct {
    const uint8_t *a, *sa, *b, *sb;
    int64_t N, K;
    double *d64, *abs64;
    uint16_t *dbf16;
} gemm_ctx;

static double mx_element(const uint8_t *q, const uint8_t *s, int64_t k)
{
    uint8_t byte = q[k / 2];
    uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return ldexp((double)oracle_e2m1_decode(code), (int)s[k / 32] - 127);
}

static void gemm_rows(void *p, int64_t m0, int64_t m1)
{
    gemm_ctx *c = (gemm_ctx *)p;
    const int64_t K = c->K;
    for (int64_t m = m0; m < m1; ++m) {
        const uint8_t *arow = c->a + m * (K / 2), *asc = c->sa + m * (K / 32);
        for (int64_t n = 0; n < c->N; ++n) {
            const uint8_t *brow = c->b + n * (K / 2), *bsc = c->sb + n * (K / 32);
            double sum = 0.0, comp = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double term = mx_element(arow, asc, k) * mx_element(brow, bsc, k);
                double t = sum + term;
                if (fabs(sum) >= fabs(term))
                    comp += (sum - t) + term;
                else
                    comp += (term - t) + sum;
                sum = t;
                mag += fabs(term);
            }
            double d = sum + comp;
            int64_t o = m * c->N + n;
            if (c->d64)
                c->d64[o] = d;
            if (c->abs64)
                c->abs64[o] = mag;
            if (c->dbf16)
                c->dbf16[o] = f32_to_bf16_rne((float)d);
        }
    }
}

int oracle_mxfp4_gemm(const uint8_t *a, const uint8_t *sa, const uint8_t *b, const uint8_t *sb,
                      int64_t M, int64_t N, int64_t K, double *d64, double *abs64, uint16_t *dbf16,
                      int nthreads)
{
    if (!a || !sa || !b || !sb || M < 0 || N < 0 || K <= 0 || K % 32 != 0)
        return -1;
    gemm_ctx c = {a, sa, b, sb, N, K, d64, abs64, dbf16};
    for_rows(gemm_rows, &c, M, nthreads);
    return 0;
}

/* ------------------------------------------------ elementwise helpers */

void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

void oracle_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_e2m1_decode_array(const uint8_t *c, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_decode(c[i]);
}

void oracle_mx_exponent_array(const float *amax, int64_t n, int32_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_mx_exponent(amax[i]);
}

void oracle_bf16_round_array(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne(v[i]);
}
