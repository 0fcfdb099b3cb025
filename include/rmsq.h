/*
 * rmsq.h -- C ABI of librmsq: fused (residual add +) RMSNorm + dynamic
 * per-token-group activation quantisation on NVIDIA GB300 (sm_103a).
 *
 * What a call computes, per row m of an [M, H] bf16 activation:
 *
 *   r = bf16(x + residual)            written to out_residual (when a
 *                                     residual is given; otherwise r = x)
 *   inv = f32(1 / sqrt(mean(r^2) + eps))
 *   y = bf16((r * inv) * gamma)       written to out_bf16 when non-NULL
 *   FP8:   per 1x128 group  scale = amax|y| / 448 (fp32),
 *          q = e4m3_saturate(y / scale)   (OCP E4M3, round to nearest even)
 *   MXFP4: per 1x32 group   X = clamp(floor(log2 amax|y|) - 2, -127, 127),
 *          scale byte = X + 127 (E8M0), q = e2m1_saturate(y * 2^-X),
 *          two codes per byte, element 2k in the low nibble (OCP MX v1.0)
 *
 * Sources: the RMSNorm + group_size=128 FP8 fusion (page "fused rmsnorm
 * quant fp8 work", Motivation); the ((fp8, scale), residual) and
 * ((bf16, fp8, scale), residual) outputs and the keep_bf16 switch (sglang PR
 * "[AMD] Add fused all-reduce RMSNorm per-group quant for Qwen3.5 FP8",
 * Motivation and Modifications); the MLA q/kv latent norm and the RMSNorm +
 * MXFP4 fusion (ATOM PR "Support input_rmsnorm_quant & qknorm_quant fused
 * for Atom dpsk v2 model", Technical Details). An all-zero group gets scale
 * 0 (E8M0 byte 0x00) and zero codes that keep the sign of the input.
 *
 * Conventions for every compute entry point:
 *  - Pointers are DEVICE pointers owned by the caller; the library allocates
 *    nothing and keeps no state between calls. bf16 tensors are passed as
 *    raw 16-bit storage.
 *  - Inputs x / residual / q_a / kv_a are row-major with a leading dimension
 *    (ld_*, in elements, >= the row length); outputs are dense row-major.
 *  - Requirements checked on the host before anything is launched: non-NULL
 *    required pointers; H a positive multiple of the group; 16-byte aligned
 *    bf16 base pointers and leading dimensions that are multiples of 8; 16-
 *    byte aligned q / y outputs; 4-byte aligned fp32 scales; eps finite and
 *    >= 0; no output overlapping an input or another output, except that
 *    out_residual may be exactly residual (in-place update, which needs
 *    ld_res == H). A failed check returns RMSQ_ERR_INVALID_ARG,
 *    RMSQ_ERR_MISALIGNED or RMSQ_ERR_UNSUPPORTED and launches nothing.
 *  - M == 0 returns RMSQ_OK without launching.
 *  - The work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and the call returns without waiting. A launch failure
 *    returns RMSQ_ERR_CUDA; rmsq_last_error() then holds the CUDA message.
 *  - Stream order is kept. The norm + quant kernels are launched as
 *    programmatic dependents of the kernel before them on the stream: their
 *    blocks may be scheduled while it finishes, but every block waits
 *    (griddepcontrol.wait) for it to complete, and its writes to be visible,
 *    before reading or writing any global memory. Only then does the kernel
 *    allow the next kernel on the stream to be scheduled early, if that one
 *    is itself launched as a programmatic dependent (the GEMMs below are);
 *    such a kernel must wait in the same way before it reads these outputs.
 *    Kernels launched without the attribute are unaffected.
 */
#ifndef RMSQ_H
#define RMSQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rmsq_status {
    RMSQ_OK = 0,
    RMSQ_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, bad enum, overlap */
    RMSQ_ERR_MISALIGNED = 2,    /* pointer or leading dimension alignment */
    RMSQ_ERR_UNSUPPORTED = 3,   /* valid but not implemented (e.g. group != 128 for FP8) */
    RMSQ_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    RMSQ_ERR_TIMEOUT = 5,       /* a bounded device wait gave up (rmsq_sync_status) */
    RMSQ_ERR_BOUNDS = 6         /* debug build only: a store's index check failed (rmsq_sync_status) */
} rmsq_status;

typedef enum rmsq_scale_layout {
    RMSQ_SCALE_ROW_MAJOR = 0,     /* scale[m * (H/128) + g]  ([M, H/128]) */
    RMSQ_SCALE_COL_MAJOR = 1,     /* scale[g * M + m]        ([H/128, M], no padding) */
    RMSQ_SCALE_COL_MAJOR_PAD4 = 2 /* scale[g * Mp + m], Mp = M rounded up to a multiple of 4, so
                                     every column starts on 16 bytes (a blockwise-FP8 GEMM's TMA
                                     load); out_scale must be 16-byte aligned; the padding
                                     entries are not written */
} rmsq_scale_layout;

/*
 * Fused residual add + RMSNorm + 1x128 FP8 (E4M3) quantisation.
 *
 *   x            [M, ld_x] bf16, row m at x + m*ld_x
 *   residual     [M, ld_res] bf16, or NULL for no residual add
 *   gamma        [H] bf16
 *   eps          added to mean(r^2)
 *   group        quantisation group; must be 128
 *   out_q        [M, H] E4M3 bytes
 *   out_scale    fp32, [M, H/128] or [H/128, M] per scale_layout
 *   out_residual [M, H] bf16 = bf16(x + residual); required iff residual
 *   out_bf16     [M, H] bf16 normalised y, or NULL ("keep_bf16" off)
 *   stream       cudaStream_t
 */
rmsq_status rmsq_add_rmsnorm_quant_group_fp8(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, int32_t group, void *out_q, float *out_scale,
    int32_t scale_layout, void *out_residual, void *out_bf16, void *stream);

/*
 * One launch normalising and FP8-quantising the two MLA attention latents
 * (q_a of width Hq, kv_a of width Hkv) with their own gammas; no residual.
 * Each latent gets exactly what rmsq_add_rmsnorm_quant_group_fp8 with
 * residual == NULL would give it.
 *
 *   q_a [M, ld_q], kv_a [M, ld_kv] bf16 (kv_a may be a column slice of a
 *   wider projection output); gamma_q [Hq], gamma_kv [Hkv] bf16;
 *   out_q_q [M, Hq] and out_kv_q [M, Hkv] E4M3; out_q_scale / out_kv_scale
 *   fp32 in scale_layout; out_q_bf16 / out_kv_bf16 optional bf16 y.
 */
rmsq_status rmsq_qknorm_quant_fp8(
    const void *q_a, int64_t ld_q, const void *kv_a, int64_t ld_kv, const void *gamma_q,
    const void *gamma_kv, float eps, int64_t M, int64_t Hq, int64_t Hkv, int32_t group,
    void *out_q_q, float *out_q_scale, void *out_kv_q, float *out_kv_scale,
    int32_t scale_layout, void *out_q_bf16, void *out_kv_bf16, void *stream);

/*
 * Fused residual add + RMSNorm + MXFP4 quantisation (group 32).
 *
 *   out_q      [M, H/2] bytes, element 2k in the low nibble of byte k
 *   out_scale  [M, H/32] E8M0 bytes (X + 127), row-major
 *   other arguments as for the FP8 call; H must be a multiple of 32.
 */
rmsq_status rmsq_add_rmsnorm_quant_mxfp4(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale, void *out_residual,
    void *out_bf16, void *stream);

/*
 * The MLA latent pair in one launch, MXFP4 flavour (the pages' "FP4 qknorm"):
 * each latent gets exactly what rmsq_add_rmsnorm_quant_mxfp4 with
 * residual == NULL would give it. Hq and Hkv are multiples of 32.
 *
 *   out_q_q [M, Hq/2], out_kv_q [M, Hkv/2] packed E2M1 bytes;
 *   out_q_scale [M, Hq/32], out_kv_scale [M, Hkv/32] E8M0 bytes (row-major);
 *   out_q_bf16 / out_kv_bf16 optional bf16 y.
 */
rmsq_status rmsq_qknorm_quant_mxfp4(
    const void *q_a, int64_t ld_q, const void *kv_a, int64_t ld_kv, const void *gamma_q,
    const void *gamma_kv, float eps, int64_t M, int64_t Hq, int64_t Hkv, uint8_t *out_q_q,
    uint8_t *out_q_scale, uint8_t *out_kv_q, uint8_t *out_kv_scale, void *out_q_bf16,
    void *out_kv_bf16, void *stream);

/*
 * As rmsq_add_rmsnorm_quant_mxfp4, with the E8M0 scales written directly in
 * the layout Blackwell's block-scaled MMA reads its scale factors from
 * (the GB300 counterpart of the pages' GEMM-specific "preshuffle" scale
 * layouts): the [M, H/32] scale matrix is cut into tiles of 128 rows x 4
 * groups, 512 bytes each, stored row-tile major (ceil(H/128) tiles per row
 * tile); inside a tile, row r and group c are at byte
 * (r % 32) * 16 + (r / 32) * 4 + c. Scale (m, g) is therefore at
 *   ((m / 128) * ceil(H/128) + g / 4) * 512 + (m % 32) * 16 + ((m % 128) / 32) * 4 + g % 4.
 * out_scale_tiles holds ceil(M/128) * ceil(H/128) * 512 bytes, 16-byte aligned;
 * entries for rows >= M or groups >= H/32 (tile padding) are not written.
 */
rmsq_status rmsq_add_rmsnorm_quant_mxfp4_mma_scales(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale_tiles, void *out_residual,
    void *out_bf16, void *stream);

/*
 * Residual add + RMSNorm alone: r and y as above, no quantisation. This is
 * the norm of the unfused placement in which the quant moves into the
 * consumer GEMM (ATOM PR "Triton fusion/GEMM optimizations for DS FP4 and
 * FP8": "AR_RMS + Quant_GEMM" at concurrency 4, with the "Triton A16WFP4
 * GEMM prequant" kernel); y goes to rmsq_a16wfp4_gemm. out_bf16 is required;
 * H must be a multiple of 32. Same conventions and checks as the fused calls.
 */
rmsq_status rmsq_add_rmsnorm(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, void *out_residual, void *out_bf16, void *stream);

/* ------------------------------------------------------- consumer GEMM */

/*
 * The GEMM that consumes the quantised activation, on the block-scaled
 * tensor cores (tcgen05.mma kind::mxf4), in the two placements the ATOM PR
 * "Triton fusion/GEMM optimizations for DS FP4 and FP8" chooses between by
 * concurrency (its environment-variable notes and the AITER PR list:
 * "Triton A16WFP4 GEMM prequant"):
 *
 *   D[M, N] = A[M, K] * B[N, K]^T,   D bf16 (fp32 accumulation, rounded to
 *                                    nearest even once), row-major, ld_d
 *
 * A and B are MXFP4 along K: E2M1 codes two per byte (element 2k in the low
 * nibble; [rows, K/2] row-major with a leading dimension in BYTES) and one
 * E8M0 scale per 32 elements, given in the MMA tile layout of
 * rmsq_add_rmsnorm_quant_mxfp4_mma_scales (ceil(rows/128) * K/128 tiles of
 * 512 bytes; rmsq_mx_scale_tiles converts a row-major scale matrix). B is
 * the weight of a linear layer, [out_features, in_features].
 *
 * rmsq_mxfp4_gemm takes A quantised (the fused norm + quant placement);
 * rmsq_a16wfp4_gemm takes A in bf16 ([M, K], ld_a in elements) and
 * quantises it inside the GEMM with exactly the rule of
 * rmsq_add_rmsnorm_quant_mxfp4 (the prequant placement), so both give
 * bit-identical D for the same activation.
 *
 * Requirements (checked on the host; nothing is launched on failure):
 * K a positive multiple of 256 and N a multiple of 8 (RMSQ_ERR_UNSUPPORTED
 * otherwise); 16-byte aligned a_q / a / b_q / scale tiles / d; ld_a, ld_b
 * multiples of 16 bytes (bf16 ld_a: multiple of 8 elements) and at least a
 * row; ld_d a multiple of 8 elements, >= N; d must not overlap an input.
 * M == 0 or N == 0 returns RMSQ_OK. Tiles of D with rows >= M or columns >=
 * N are not written.
 */
rmsq_status rmsq_mxfp4_gemm(
    const void *a_q, int64_t ld_a, const void *a_scale_tiles, const void *b_q, int64_t ld_b,
    const void *b_scale_tiles, void *d, int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream);
/*
 * Every wait inside the GEMM kernels (a CTA waiting for its operand copies,
 * for the tensor cores, or for its cluster peers) is bounded, 2 s by default
 * (rmsq_gemm_opts.wait_limit_ns). A CTA whose wait runs out stops, drains its
 * copies, frees its tensor memory and sets the status word; the call itself
 * has already returned RMSQ_OK at launch. D is then incomplete, and only
 * rmsq_sync_status reports it (RMSQ_ERR_TIMEOUT): a caller that cannot rule
 * out a stalled GPU (time-slicing with other work, a debugger) checks
 * rmsq_sync_status before trusting D. The limit is more than a thousand
 * times the slowest launch measured on GB300 (the quantising GEMM at
 * M = 16384, N = 2112, K = 7168: about a millisecond; the GEMM on quantised
 * A: about 0.1 ms).
 *
 * Overlap with the norm + quant: the one-CTA-per-tile GEMM (the schedule the
 * library picks below about 2048 tokens) is launched as a programmatic
 * dependent of the kernel before it on the stream, and the norm + quant
 * kernels let their dependents start early. Right after a norm + quant (or
 * rmsq_add_rmsnorm) call on the same stream, the GEMM therefore sets up and
 * loads B and its scale tiles while that call is still running, and waits
 * for it to finish before it reads A (or the bf16 activation) and before it
 * writes D. B and b_scale_tiles must not be outputs of that immediately
 * preceding call. After any other kernel, the GEMM starts when that kernel
 * has finished, as usual.
 */

rmsq_status rmsq_a16wfp4_gemm(
    const void *a, int64_t ld_a, const void *b_q, int64_t ld_b, const void *b_scale_tiles, void *d,
    int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * Row-major [R, G] E8M0 scale bytes (leading dimension ld) -> the MMA tile
 * layout above: out receives ceil(R/128) * ceil(G/4) * 512 bytes, padding
 * (rows >= R, groups >= G) set to `fill`. For preparing weight scales.
 */
rmsq_status rmsq_mx_scale_tiles(const uint8_t *scale, int64_t ld, int64_t R, int64_t G, uint8_t *out,
                                uint8_t fill, void *stream);

/* ------------------------------------------------------------ utilities */

/*
 * Copies `bytes` bytes from src to dst (device pointers, 16-byte aligned,
 * not overlapping, bytes a multiple of 16) with a plain streaming kernel:
 * every byte is read from and written to HBM once. This is not an operation
 * of the source pages; it is the read + write copy whose rate serves as the
 * HBM roofline's peak where no separately measured peak is available.
 * Enqueued on `stream`; RMSQ_ERR_INVALID_ARG for bad arguments.
 */
rmsq_status rmsq_copy(const void *src, void *dst, int64_t bytes, void *stream);

/* Static description of a status code. */
const char *rmsq_status_string(rmsq_status s);

/* Message of the last failing call on this host thread ("" if none). */
const char *rmsq_last_error(void);

/*
 * Waits for `stream`, then reads and clears the library's device status
 * word on the current device. Returns RMSQ_ERR_TIMEOUT if a kernel launched
 * since the last read gave up a bounded wait (its outputs are then
 * incomplete), RMSQ_ERR_BOUNDS if, in a library built with RMSQ_DEBUG, an
 * index check before a store failed (the store was skipped),
 * RMSQ_ERR_CUDA if the synchronisation failed or a GEMM kernel found its
 * shared memory not 1024-byte aligned (it then wrote nothing; its layout
 * relies on the alignment the hardware gives), else RMSQ_OK.
 *
 * The word is one per device and per process, shared by every stream and
 * host thread: a call reports (and clears) what any kernel of the library on
 * this device recorded since the previous call, whichever stream launched
 * it, and only `stream` is waited for. The bits read are cleared with an
 * atomic operation enqueued on `stream`, so a bit that a kernel on another
 * stream sets between the read and the clear is kept for the next call.
 */
rmsq_status rmsq_sync_status(void *stream);

/* ------------------------------------------------- launch control & tests */

typedef enum rmsq_kernel {
    RMSQ_KERNEL_AUTO = 0,        /* library's choice */
    RMSQ_KERNEL_ROWS = 1,        /* one team per row, rows loaded into registers */
    RMSQ_KERNEL_PERSISTENT = 2   /* grid of resident blocks looping over rows, x / residual
                                    rows double-buffered in shared memory by bulk copies */
} rmsq_kernel;

typedef enum rmsq_form {
    RMSQ_FORM_AUTO = 0,          /* latency form when the row kernel's launch has at most one
                                    block per SM, else the throughput form */
    RMSQ_FORM_THROUGHPUT = 1,    /* gamma read as the row is normalised; the team's first warp
                                    finalises inv_rms and broadcasts it (a second barrier) */
    RMSQ_FORM_LATENCY = 2        /* gamma loaded together with the row; every warp finalises
                                    inv_rms itself after the one barrier */
} rmsq_form;

/*
 * Optional launch control for the _ex entry points (NULL = defaults). Kernels
 * and rows-per-block choices with the same team shape give bit-identical
 * outputs; different team shapes sum the squares in a different order and
 * can differ only in rows whose inv_rms is within ~2^-44 of an fp32 rounding
 * boundary. These exist for tests and tuning.
 *   kernel          rmsq_kernel
 *   vpt             16-byte vectors (8 bf16) per thread, 1..8; 0 = auto. The
 *                   team (threads per row) is the smallest size that holds
 *                   H/8 vectors at vpt each and is either a power-of-two
 *                   multiple of the group's vector count up to 32 or a
 *                   multiple of 32, at most 512; vectors past the row end
 *                   are idle (whole groups).
 *   rows_per_block  0 = auto: 256 threads' worth of teams, or in the latency
 *                   form as few rows per block (whole warps) as keep the
 *                   launch within one block per SM
 *   grid            persistent kernel: number of blocks, 0 = auto
 *   debug_skip_row  persistent kernel: the copy of this row is never issued,
 *                   so its wait runs out (test of the bounded wait); -1 = off
 *   wait_limit_ns   persistent kernel: limit of every wait, 0 = 2 s
 *   form            row kernel: rmsq_form. Both forms give bit-identical
 *                   outputs (same order of every addition); the latency form
 *                   exists for the compiled team shapes (H = 7168, 8192, 5120,
 *                   4096, 2048, 1536, 512, 256 at their default vpt) and is
 *                   ignored for other shapes.
 *   split           latency form with one row per block: the blocks that
 *                   share each row's outputs, 1, 2 or 4 (dividing vpt);
 *                   each loads and reduces the whole row, so all compute the
 *                   same inv_rms, and normalises, quantises and stores its
 *                   part. 0 = auto: the largest of 4 and 2 that keeps the
 *                   launch within one block per SM, else 1. A residual
 *                   updated in place (out_residual == residual) is never
 *                   split: a block would write back its part while another
 *                   block of the row may still be reading it. Auto then
 *                   takes 1, and split > 1 is refused (RMSQ_ERR_UNSUPPORTED).
 */
typedef struct rmsq_launch_opts {
    int32_t kernel;
    int32_t vpt;
    int32_t rows_per_block;
    int32_t grid;
    int64_t debug_skip_row;
    int64_t wait_limit_ns;
    int32_t form;
    int32_t split;
} rmsq_launch_opts;

rmsq_status rmsq_add_rmsnorm_quant_group_fp8_ex(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, int32_t group, void *out_q, float *out_scale,
    int32_t scale_layout, void *out_residual, void *out_bf16, void *stream,
    const rmsq_launch_opts *opts);

rmsq_status rmsq_add_rmsnorm_quant_mxfp4_ex(
    const void *x, int64_t ld_x, const void *residual, int64_t ld_res, const void *gamma,
    float eps, int64_t M, int64_t H, uint8_t *out_q, uint8_t *out_scale, void *out_residual,
    void *out_bf16, void *stream, const rmsq_launch_opts *opts);

/*
 * Optional control of the GEMM launch (NULL = defaults), for tests and
 * tuning; results do not depend on it.
 *   bn             rows of B per CTA tile: 64, 128 or 256, or 192 with the
 *                  CTA-pair schedule only (then rows of B per pair tile);
 *                  0 = auto (for the prequant GEMM, which quantises A once
 *                  per B tile: 64 up to 16 rows of A, 128 with exactly two
 *                  128-row tiles of A, else 256; for the plain GEMM 256 once
 *                  that gives half the SMs a tile, else 128 with two or more
 *                  128-row tiles of A, else 64; CTA pairs take 256 or 192,
 *                  whichever leaves the busiest pair the least work)
 *   ksplit         CTAs, launched as one thread-block cluster, that split K
 *                  for each tile and add their fp32 partial sums through
 *                  distributed shared memory (rank order, so deterministic):
 *                  1..8 and at most K/256; 0 = auto (enough to give every SM
 *                  a CTA when there are fewer tiles than SMs). Splitting K
 *                  changes the order of the fp32 additions, so results can
 *                  differ between ksplit values in the last bits (both
 *                  placements agree bit for bit at equal ksplit and bn).
 *   wait_limit_ns  limit of every wait inside the kernel, 0 = 2 s
 *   debug_stall_stage  test hook, 0 = off (so zero-initialised options are
 *                  the defaults): with s > 0 every CTA leaves the loads of its
 *                  K stage s - 1 (counted within the CTA's share of K)
 *                  unissued, so a wait runs out; the kernel then stops,
 *                  drains, frees its tensor memory and sets the status word
 *                  (rmsq_sync_status returns RMSQ_ERR_TIMEOUT, D is
 *                  incomplete). With the persistent schedule the stage is
 *                  counted over the CTA's tiles.
 *   schedule       0 = auto (CTA pairs when quantised A takes 256-row B
 *                  tiles without a K split; else persistent when there are
 *                  more tiles than SMs), 1 = one tile per CTA, 2 =
 *                  persistent: one CTA per SM walks the tiles, so a tile's
 *                  set-up, first loads and epilogue overlap its neighbours'
 *                  work (quantised A and ksplit 1 only), 3 = persistent CTA
 *                  pairs: a cluster of two CTAs computes 256 x 256 (or
 *                  256 x 192, two accumulators) tiles with the tensor cores
 *                  of both SMs (quantised A, bn 0, 192 or 256, ksplit 0 or
 *                  1). Results do not depend on it.
 */
typedef struct rmsq_gemm_opts {
    int32_t bn;
    int32_t ksplit;
    int64_t wait_limit_ns;
    int32_t debug_stall_stage;
    int32_t schedule;
} rmsq_gemm_opts;

rmsq_status rmsq_mxfp4_gemm_ex(
    const void *a_q, int64_t ld_a, const void *a_scale_tiles, const void *b_q, int64_t ld_b,
    const void *b_scale_tiles, void *d, int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream,
    const rmsq_gemm_opts *opts);

rmsq_status rmsq_a16wfp4_gemm_ex(
    const void *a, int64_t ld_a, const void *b_q, int64_t ld_b, const void *b_scale_tiles, void *d,
    int64_t ld_d, int64_t M, int64_t N, int64_t K, void *stream, const rmsq_gemm_opts *opts);

/*
 * The launch rmsq_mxfp4_gemm_ex (prequant = 0) or rmsq_a16wfp4_gemm_ex
 * (prequant != 0) makes for an M x N x K product with these options (NULL =
 * defaults), on a device with `sms` SMs on which `pairs_256` / `pairs_192`
 * CTA pairs of the 256- / 192-wide pair kernel fit at once (the GEMM entry
 * points ask the current device for the three numbers; here the caller gives
 * them). This is the library's own launch choice, not an operation of the
 * source pages. Pure host arithmetic: no CUDA call, no device needed. The
 * choice is the one the GEMM calls make, so it applies their option and shape
 * checks and returns the same status for the same arguments (pointer, pitch
 * and alignment checks aside); a pair capacity is needed only when the
 * library picks the pair width, and a non-positive one then gives
 * RMSQ_ERR_INVALID_ARG.
 *   plan->bn               B-tile width (rows of B per CTA, or per CTA pair)
 *   plan->ksplit           CTAs of one cluster that split each tile's K (1: none)
 *   plan->schedule         1 one tile per CTA (or per cluster), 2 persistent,
 *                          3 CTA pairs
 *   plan->persistent_ctas  CTAs of the persistent grid (schedule 2), else 0
 * With M = 0 or N = 0 nothing is launched and *plan is all zeros. *plan is
 * zeroed first, so it is all zeros after any error. plan is required
 * (caller-owned host memory).
 */
typedef struct rmsq_gemm_plan {
    int32_t bn;
    int32_t ksplit;
    int32_t schedule;
    int32_t persistent_ctas;
} rmsq_gemm_plan;

rmsq_status rmsq_gemm_plan_for(
    int32_t prequant, int64_t M, int64_t N, int64_t K, const rmsq_gemm_opts *opts, int32_t sms,
    int32_t pairs_256, int32_t pairs_192, rmsq_gemm_plan *plan);

/*
 * The device encoders the kernels use, applied elementwise to n fp32 values
 * (device pointers): E4M3 bytes (round to nearest even, saturating; NaN ->
 * 0x7F/0xFF), and E2M1 codes, one 4-bit code per output byte. They exist so
 * that the hardware conversions can be checked against an independent
 * definition.
 */
rmsq_status rmsq_encode_e4m3(const float *in, uint8_t *out, int64_t n, void *stream);
rmsq_status rmsq_encode_e2m1(const float *in, uint8_t *out, int64_t n, void *stream);

/*
 * Exhaustive self-check of the FP8 quantiser's division: for every positive
 * finite bf16 amax and every bf16 y with |y| <= amax (both signs), the E4M3
 * code the kernels produce for y / (amax/448) is compared with the code of
 * IEEE fp32 division, and the kernels' scale amax/448 with the IEEE
 * quotient. `counts` is a caller-zeroed device array of five unsigned
 * 64-bit counters, incremented by: code mismatches, fp32 quotient mismatches,
 * (amax, y) pairs checked, scale mismatches, quotient mismatches with
 * |y| >= 2^-100 (informational: the kernels use only the code, whose count
 * must be zero). Enqueued on `stream`.
 */
rmsq_status rmsq_check_group_division(unsigned long long *counts, void *stream);

/*
 * Positive control of the debug build's store checks: in a library built
 * with RMSQ_DEBUG, enqueues a one-thread kernel whose single check fails on
 * purpose (nothing is stored), so that the next rmsq_sync_status returns
 * RMSQ_ERR_BOUNDS. In release builds it returns RMSQ_ERR_UNSUPPORTED and
 * launches nothing.
 */
rmsq_status rmsq_debug_bounds_selftest(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* RMSQ_H */
