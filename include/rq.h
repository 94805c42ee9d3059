/*
 * rq.h -- C ABI of the rotation-based W4A4 inference kernels (GB300, sm_103a).
 *
 * The online hot path of rotation-based 4-bit inference, and the operations
 * around it:
 *
 *   rq_fwht_quant       randomized fast Walsh-Hadamard transform of each row,
 *                       fused with per-row symmetric INT4 quantization and
 *                       nibble packing;
 *   rq_w4a4_gemm        the W4A4 linear layer: exact integer product of packed
 *                       INT4 activations and packed INT4 (rotation-folded)
 *                       weights, with a per-token x per-channel scale epilogue;
 *   rq_kv_rotate_quant  head-wise Hadamard rotation and INT4 quantization of K
 *                       and V before they are written to the cache.
 *   rq_fwht_quant_gemm  decode-sized fusion of rq_fwht_quant and rq_w4a4_gemm:
 *                       rotation, quantization and the W4A4 product in one
 *                       launch, the rotated activations never reaching HBM.
 *   rq_attn_decode      attention of decode queries over the rotated INT4 KV
 *                       cache that rq_kv_rotate_quant writes;
 *   rq_w4a8_gemm        the W4A8 variant of the linear layer (INT8 activations),
 *                       with per-channel or per-group weight scales.
 *
 * Sources (page title, then section / equation):
 *   [ROT] "Rotational Quantization: How Orthogonal Transforms and Hadamard
 *         Incoherence Enable Outlier-Free Low-Bit Inference" (llms.blog)
 *   [QR]  aicassindra.com quantization series, "QuaRot" page
 *   [SQ]  aicassindra.com quantization series, "SpinQuant" page
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every data pointer is a DEVICE pointer (memory the current CUDA
 *   device can read/write: cudaMalloc / PyTorch CUDA tensors / managed memory).
 *   The caller owns all buffers.  The library allocates no device memory and
 *   keeps no state between calls except one device-resident error word used by
 *   bounded waits (see rq_sync_status).
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Calls only enqueue work and return; results are ready once the
 *   stream reaches that point.  Calls on different streams may run concurrently
 *   as long as their output buffers do not overlap.
 * Alignment.  Every pointer must be 16-byte aligned and every row stride a
 *   multiple of 16 bytes; otherwise RQ_ERR_MISALIGNED.
 * Errors.  Arguments are checked on the host before anything is enqueued; a
 *   failing check returns a non-zero rq_status and enqueues nothing.  A failed
 *   kernel launch returns RQ_ERR_CUDA.  Nothing is ever printed or aborted.
 * Rotation.  R is the randomized Hadamard rotation of [ROT] §Incoherence
 *   Processing via Randomized Hadamard Transforms: H_n is the normalized
 *   Sylvester matrix of the page's recursion H_1 = [1],
 *   H_2k = (1/sqrt2)[[H_k, H_k], [H_k, -H_k]] (natural order, entries
 *   +-1/sqrt(n)), and s in {-1,+1}^n is a Rademacher vector drawn from `seed`:
 *   s_i = +1 when the top bit of output i (0-based) of SplitMix64 seeded with
 *   `seed` is 0, else -1.  flags bit 0 (RQ_SIGNS_FIRST) selects the form:
 *     RQ_SIGNS_FIRST set:   y = (x diag(s)) H_n     (the signs act first)
 *     RQ_SIGNS_FIRST clear: y = (x H_n) diag(s)     (R = H_d·diag(s), [ROT] eq.)
 *   The two forms are transposes of each other; use the same flags for the
 *   activations and for the offline weight fold.
 * Quantization.  Per row (token, or (token, head)): scale = max_j |y_j| / 7,
 *   q_j = clamp(round_half_even(y_j / scale), -8, 7); an all-zero row gets
 *   scale 0 and all-zero codes.  The scale is stored as fp32.  The GPU decides
 *   the rounding in fp32: a code may differ by one from an exact (fp64)
 *   computation only where y_j/scale lies within about 1e-6 of a half-integer.
 * Packing.  A row of n codes is n/2 bytes; byte j holds code 2j in bits 3..0
 *   and code 2j+1 in bits 7..4, each a 4-bit two's-complement value.
 */
#ifndef RQ_H
#define RQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RQ_OK = 0,
    RQ_ERR_INVALID_ARG = 1, /* a size is negative/zero where not allowed, a required pointer is NULL */
    RQ_ERR_UNSUPPORTED = 2, /* a size outside what the kernels implement (e.g. n = 24) */
    RQ_ERR_MISALIGNED = 3,  /* a pointer or stride breaks the 16-byte rule */
    RQ_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    RQ_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see rq_sync_status) */
} rq_status;

typedef enum {
    RQ_F32 = 0,  /* float */
    RQ_BF16 = 1, /* bfloat16 */
    RQ_F16 = 2,  /* IEEE half */
    RQ_I32 = 3   /* int32 (GEMM raw accumulators only) */
} rq_dtype;

enum { RQ_SIGNS_FIRST = 1u };
/* rq_attn_decode: leave the output in the rotated basis (o~ instead of o~ R^T). */
enum { RQ_ATTN_ROTATED_OUT = 2u };
/* rq_fwht_quant (n = m 2^k, or a power of two from 256 to 8192): INT8 codes per row (activations of the W4A8 layer),
 * or INT4 codes with one scale per group of 128 elements (weights with per-group
 * scales); rq_w4a4_gemm: w_scales are per group of 128 (with RQ_A_E4M3). */
enum { RQ_INT8_CODES = 4u, RQ_GROUP_SCALES = 8u };
/* rq_fwht_quant (powers of two from 256 to 8192): the INT4 codes written as the
 * W4A4 product's operand, one byte per code (see rq_fwht_quant); rq_w4a4_gemm:
 * the activation codes a_q are given in that form. */
enum { RQ_E4M3_CODES = 16u, RQ_A_E4M3 = 16u };

/* rq_fwht_quant code mode: the default INT4 codes, one int8 byte each. */
enum { RQ_INT4_BYTES = 32u };

/* Smallest / largest supported Hadamard size (row length n, head_dim). */
#define RQ_MIN_N 32
#define RQ_MAX_N 8192

/*
 * rq_fwht_quant -- rotate each row by R and quantize it to packed INT4.
 *
 *   [ROT] §Weight Absorption and Online Fast Walsh-Hadamard Transforms,
 *   2. Online FWHT (n log2 n additions/subtractions, one global 1/sqrt(n)
 *   scale); [ROT] §Incoherence (R = H_d·diag(s)); [QR] §End-to-end flow (the
 *   activation is rotated on the fly by a Hadamard transform, then quantized to
 *   INT4).  The same call performs the offline
 *   weight fold W~ = R^T W of [ROT] §Weight Absorption, 1. when given the rows
 *   of W^T (one output channel per row): each output channel is then quantized
 *   with its own scale.
 *
 *   x        [rows][ld_x] elements of x_dtype (RQ_F32, RQ_BF16 or RQ_F16);
 *            row r is x + r*ld_x, its first n elements are used.
 *   rows     number of rows, >= 0 (0: nothing is enqueued).
 *   n        row length: a power of two in [RQ_MIN_N, RQ_MAX_N], or m 2^k with
 *            m in {12, 20, 28} and 2^k in [32, 1024] (e.g. 3072, 5120, 14336,
 *            28672).  For the latter, H_n is H_m (x) H_{2^k} with H_m a Paley
 *            Hadamard matrix ([ROT] §The Computational Cost of Arbitrary
 *            Rotations and §SpinQuant: sizes that are not powers of two, via
 *            products of Sylvester-compatible sizes):
 *              chi = quadratic character mod q, Q[i][j] = chi(j - i);
 *              m = 12, 20 (q = 11, 19): H = I + [[0, 1^T], [-1, Q]];
 *              m = 28 (q = 13): S = [[0, 1^T], [1, Q]],
 *                H = S (x) [[1, 1], [1, -1]] + I (x) [[1, -1], [-1, -1]];
 *            element a 2^k + j of a row is segment a, offset j, and
 *            y = x diag(s) (H_m (x) H_{2^k}) / sqrt(n) (or diag(s) after).
 *   ld_x     row stride in elements, >= n, ld_x * sizeof(x_dtype) % 16 == 0.
 *   seed     sign-vector seed.
 *   flags    RQ_SIGNS_FIRST or 0, plus at most one of (n = m 2^k, n = 128,
 *            or a power of two from 256 to 8192; RQ_ERR_UNSUPPORTED for
 *            n < 128; at n = 128 the one group of RQ_GROUP_SCALES is the row):
 *            RQ_INT8_CODES: per-row INT8 codes for the W4A8 layer's
 *              activations ([SQ] §End-to-end flow): q is [rows][n] int8,
 *              scale = max|y| / 127, q = clamp(round_half_even(y / scale),
 *              -128, 127), scales [rows] fp32 as above;
 *            RQ_GROUP_SCALES: INT4 codes with one scale per group of 128
 *              consecutive elements ([SQ] §The architecture, per-group scales;
 *              the weight fold of the W4A8 layer): q as above, scales
 *              [rows][n/128] fp32.
 *            RQ_E4M3_CODES (n = 128 and powers of two from 256 to 8192): the same
 *              INT4 codes and scales as the default, each code stored as the
 *              tensor-core operand of rq_w4a4_gemm (RQ_A_E4M3): q is
 *              [rows][n] bytes; the byte of code q is q for q >= 0 and
 *              0x80 | -q for q < 0 (the FP8 E4M3 encoding of q * 2^-9), and
 *              within each group of 8 codes the bytes hold codes
 *              0, 2, 4, 6, 1, 3, 5, 7 of the group.  scales is [rows][2]
 *              fp32: the row's scale (max|y|/7, as the default) and the sum
 *              of its n codes (an integer, exact in fp32), the product's
 *              offset term.  Twice the bytes of the packed form; the product
 *              then widens only the weights.
 *            RQ_INT4_BYTES: the default INT4 codes and scales (max|y|/7),
 *              each code stored as one int8 byte: q is [rows][n] int8.  This
 *              is the activation operand of rq_w4a8_gemm, which then computes
 *              the W4A4 product with per-channel or per-group (128) weight
 *              scales ([SQ] §The architecture, per-group scales).
 *   q        out: [rows][n/2] bytes, packed codes (row stride n/2).
 *   scales   out: [rows] fp32 scales, max|y|/7 of each rotated row (the
 *            shapes above for RQ_GROUP_SCALES and RQ_E4M3_CODES).
 *   y        out, may be NULL: [rows][n] fp32 rotated rows y = xR (parity
 *            checks only; writing it adds 4n bytes of traffic per row).
 */
rq_status rq_fwht_quant(const void *x, rq_dtype x_dtype, int64_t rows, int64_t n, int64_t ld_x,
                        uint64_t seed, uint32_t flags, uint8_t *q, float *scales, float *y,
                        void *stream);

/*
 * rq_w4a4_gemm -- y = dequant(Q(XR) · Q(R^T W)).
 *
 *   acc[m][c] = sum_k qa[m][k] * qw[c][k]   (exact, int32)
 *   y[m][c]   = acc[m][c] * a_scales[m] * w_scales[c]   (fp32 math)
 *   [ROT] §The Principle of Computational Invariance (Y = (XR)(R^T W));
 *   [ROT] §Learned Orthogonal Rotations (the product Q(XR)·Q(R^T W));
 *   [ROT] §Hardware Execution, 1. True INT4 Tensor Core Utilization;
 *   [QR] §End-to-end flow.
 *
 *   a_q       [M][K/2] packed activation codes (row stride K/2), e.g. from
 *             rq_fwht_quant on X.
 *   a_scales  [M] per-token fp32 scales.
 *   w_q       [N][K/2] packed weight codes, one output channel per row, e.g.
 *             from rq_fwht_quant on the rows of W^T (the offline fold).
 *   w_scales  [N] per-channel fp32 scales, or with RQ_GROUP_SCALES [N][K/128]
 *             per-group scales (rq_fwht_quant with RQ_GROUP_SCALES on the rows
 *             of W^T).
 *   M, N, K   M >= 0, N >= 0 (0: nothing is enqueued), K a positive multiple
 *             of 128 and at most 65536.
 *   seed      accepted for a uniform signature and ignored: the rotation is
 *             already folded into w_q.
 *   flags     0, or RQ_A_E4M3: a_q is [M][K] bytes, the activation codes in
 *             the operand form rq_fwht_quant writes with RQ_E4M3_CODES (M > 64
 *             only; RQ_ERR_UNSUPPORTED otherwise), and a_scales is [M][2]
 *             (scale, sum of the row's codes) as it writes them; a_scales is
 *             then required for RQ_I32 too.
 *             RQ_A_E4M3 | RQ_GROUP_SCALES: per-group (128) weight scales
 *             ([SQ] §The architecture, per-group scales):
 *               y[m][c] = a_scales[m][0] * sum_g w_scales[c][g] * acc_g[m][c],
 *             acc_g the exact sum over the 128 codes of group g, scaled and
 *             summed in fp32 in group order.  M > 64, N a multiple of 128,
 *             K <= 8192, RQ_F16 or RQ_F32 output; RQ_ERR_UNSUPPORTED otherwise
 *             (rq_w4a8_gemm on RQ_INT4_BYTES codes covers the other shapes).
 *   y         out: [M][N] row-major, of y_dtype:
 *             RQ_F16  the dequantized product rounded to fp16;
 *             RQ_F32  the dequantized product in fp32;
 *             RQ_I32  the raw int32 accumulators (scales unused, may be NULL,
 *                     but for the code sums of RQ_A_E4M3).
 *             N * sizeof(y_dtype) must be a multiple of 16 bytes.
 *   Kernels (all on tensor cores, the integer sums exact in each):
 *     M > 64: persistent CTA pairs, 256 x 256 tiles, codes widened to FP8
 *       (tcgen05 kind::f8f6f4), tiles walked M-fastest for L2 reuse of W;
 *     M <= 64, N a multiple of 128, K <= 8192: weights in tensor memory as
 *       the MMA's 128-row side, tokens as its N side, K split over thread-block
 *       clusters of up to 8 CTAs reduced in distributed shared memory;
 *     other shapes: legacy FP8 mma.sync, CTAs of 16 channels x 64 tokens;
 *     per-group scales: CTA pairs, 256 x 128 tiles, one tensor-memory partial
 *       per group, scaled and summed by the epilogue warps in registers.
 */
rq_status rq_w4a4_gemm(const uint8_t *a_q, const float *a_scales, const uint8_t *w_q,
                       const float *w_scales, int64_t M, int64_t N, int64_t K, uint64_t seed,
                       uint32_t flags, void *y, rq_dtype y_dtype, void *stream);

/*
 * rq_kv_rotate_quant -- rotate each (token, head) vector of K and V by the
 * randomized Hadamard of size head_dim and quantize it per (token, head).
 *
 *   [QR] §The architecture (the KV-cache rotation box: each token's keys and
 *   values are rotated, then quantized, before they are stored) and
 *   §End-to-end flow, "The KV cache"; [ROT] §Hardware Execution, 2. End-to-End
 *   KV Cache Footprint Reduction.  One sign vector of length head_dim (from
 *   `seed`) is shared by every head and by K and V.
 *
 *   k, v       [tokens][heads][head_dim] contiguous, of dtype (RQ_BF16, RQ_F16
 *              or RQ_F32).  Either may be NULL, not both; a NULL input skips
 *              its outputs (which may then be NULL too).
 *   tokens     >= 0 (0: nothing is enqueued); heads >= 1.
 *   head_dim   a power of two in [RQ_MIN_N, 256].
 *   kq, vq     out: [tokens][heads][head_dim/2] packed codes.
 *   ks, vs     out: [tokens][heads] fp32 scales.
 */
rq_status rq_kv_rotate_quant(const void *k, const void *v, rq_dtype dtype, int64_t tokens,
                             int64_t heads, int64_t head_dim, uint64_t seed, uint32_t flags,
                             uint8_t *kq, float *ks, uint8_t *vq, float *vs, void *stream);

/*
 * rq_fwht_quant_gemm -- y = dequant(Q(x R) . w_q) for a few tokens, in one launch.
 *
 *   The rotation and quantization of rq_fwht_quant ([ROT] §Incoherence
 *   Processing via Randomized Hadamard Transforms; §Weight Absorption and
 *   Online Fast Walsh-Hadamard Transforms, 2.) fused with the product of
 *   rq_w4a4_gemm ([ROT] §Hardware Execution and Serving Economics, 1.): the
 *   codes of x R are formed in on-chip memory and consumed there.  The result
 *   equals rq_fwht_quant followed by rq_w4a4_gemm on the same inputs (the same
 *   codes and scales, bit for bit).
 *
 *   x         [M][ld_x] activation rows, bf16 or fp16 (x_dtype), ld_x >= K.
 *   M         1 <= M <= 16 (decode batches).
 *   K         the row length: 1024, 2048, 4096 or 8192 (RQ_ERR_UNSUPPORTED
 *             otherwise).
 *   seed, flags   as for rq_fwht_quant; must match the fold of w_q.
 *   w_q, w_scales, N   as for rq_w4a4_gemm; N a multiple of 128.
 *   y, y_dtype as for rq_w4a4_gemm (RQ_F16, RQ_F32, or RQ_I32 raw accumulators).
 *   a_q, a_scales  optional (NULL to skip): receive the activation codes
 *              [M][K/2] and scales [M], as rq_fwht_quant would write them.
 *   Errors: as for rq_fwht_quant and rq_w4a4_gemm (RQ_ERR_INVALID_ARG,
 *   RQ_ERR_UNSUPPORTED for a shape or dtype outside the above,
 *   RQ_ERR_MISALIGNED for pointers or a row stride off their 16-byte rules);
 *   M == 0 or N == 0 returns RQ_OK without a launch.  The launch has N/128
 *   thread-block clusters of S = 1, 2, 4 or 8 CTAs (S >= K/1024), one CTA per
 *   SM: the CTAs of a cluster split K, rotate the tokens between them and
 *   exchange the codes in distributed shared memory; the product runs on the
 *   5th-generation tensor cores (weights in tensor memory).  A bounded wait that
 *   gives up sets the error word that rq_sync_status reads.
 */
rq_status rq_fwht_quant_gemm(const void *x, rq_dtype x_dtype, int64_t M, int64_t K, int64_t ld_x,
                             uint64_t seed, uint32_t flags, const uint8_t *w_q, const float *w_scales,
                             int64_t N, void *y, rq_dtype y_dtype, uint8_t *a_q, float *a_scales,
                             void *stream);

/*
 * rq_attn_decode -- attention of decode queries over the rotated INT4 KV cache.
 *
 *   [QR] §End-to-end flow, "The KV cache": a later token's attention reads the
 *   four-bit rotated cache, and rotation invariance keeps the scores those of
 *   the full-precision computation; [QR] §The architecture (the invariance box:
 *   a rotation is cancelled by its transpose, folded into the next weight or
 *   applied as its own Hadamard).  For query row m and head h:
 *     q~   = q[m][h] R                        (R as the cache write: seed, flags)
 *     e_t  = softmax_scale * (q~ . k^_t)      k^_t = codes(kq[t][h]) * ks[t][h]
 *     p    = softmax over t of e
 *     out  = (sum_t p_t v^_t) R^T             v^_t = codes(vq[t][h]) * vs[t][h]
 *   or the sum itself with RQ_ATTN_ROTATED_OUT (for an output weight with R
 *   folded in).  Every query row attends to every cached token (no mask).
 *
 *   q          [M][heads][head_dim] activations, fp32, bf16 or fp16 (q_dtype),
 *              contiguous.
 *   kq, vq     [tokens][heads][head_dim/2] packed codes; ks, vs [tokens][heads]
 *              fp32 scales: the layout rq_kv_rotate_quant writes.
 *   tokens     >= 1 cached tokens.
 *   head_dim   32, 64, 128 or 256 (RQ_ERR_UNSUPPORTED otherwise).
 *   seed       the cache's sign seed.
 *   flags      RQ_SIGNS_FIRST (as the cache was written) | RQ_ATTN_ROTATED_OUT.
 *   softmax_scale  multiplies the scores (usually 1/sqrt(head_dim)).
 *   out        [M][heads][head_dim] fp32.
 *   Errors: RQ_ERR_INVALID_ARG (negative sizes, tokens < 1 with work to do,
 *   unknown flags, NULL pointers), RQ_ERR_UNSUPPORTED (dtype, head_dim),
 *   RQ_ERR_MISALIGNED (q, kq, vq, out not 16-byte aligned; ks, vs not 4-byte
 *   aligned).  M == 0 or heads == 0 returns RQ_OK without a launch.  One
 *   cluster of 8 CTAs per (row, head), each reading an eighth of the tokens;
 *   no global scratch.
 */
rq_status rq_attn_decode(const void *q, rq_dtype q_dtype, int64_t M, int64_t heads, int64_t head_dim,
                         const uint8_t *kq, const float *ks, const uint8_t *vq, const float *vs, int64_t tokens,
                         uint64_t seed, uint32_t flags, float softmax_scale, float *out, void *stream);

/*
 * rq_w4a8_gemm -- the W4A8 linear layer with per-channel or per-group weight scales.
 *
 *   [SQ] §The architecture (INT4 weights, INT8 activations, per-channel or
 *   per-group scales), §End-to-end flow (the rotated activation quantized to
 *   INT8 and multiplied against the INT4 rotated weights):
 *     acc_g[m][c] = sum_{k in group g} a_q[m][k] * w_q[c][k]   (exact integers)
 *     y[m][c]     = a_scales[m] * sum_g w_scales[c][g] * acc_g[m][c]
 *
 *   a_q       [M][K] int8 codes (rq_fwht_quant with RQ_INT8_CODES).
 *   a_scales  [M] fp32.
 *   w_q       [N][K/2] packed INT4 codes, one output channel per row.
 *   w_scales  [N] fp32 (group == K) or [N][K/128] fp32 (group == 128,
 *             rq_fwht_quant with RQ_GROUP_SCALES on the rows of W^T).
 *   K         a multiple of 128.  group: 128 or K.
 *   y, y_dtype  [M][N]: RQ_F16, RQ_F32, or RQ_I32 (raw exact sums, group == K
 *             only).
 *   Kernels: per-channel scales with M > 64, K <= 65536 and rows of y a
 *   multiple of 16 bytes run on the 5th-generation tensor cores (each INT8 code
 *   split exactly into two 4-bit halves, a = 16 (a >> 4) + (a & 15), both
 *   multiplied as FP8 into separate exact accumulators, CTA pairs, 128 x 256
 *   output tiles).  Per-group scales with M > 64, N a multiple of 128 and
 *   K <= 8192 also run on the tensor cores: one exact partial per group in
 *   tensor memory, scaled and summed in fp32 by the epilogue (128 x 128 tiles).
 *   Everything else goes through legacy tensor-core MMAs (int8 x int8 ->
 *   int32), CTAs of 16 channels x 32 tokens.  The integer sums of a group are
 *   exact in every kernel.
 *   Errors: RQ_ERR_INVALID_ARG (negative sizes, NULL pointers),
 *   RQ_ERR_UNSUPPORTED (K, group, y_dtype), RQ_ERR_MISALIGNED (a_q, w_q, y not
 *   16-byte aligned; scales not 4-byte aligned).  M == 0 or N == 0 returns
 *   RQ_OK without a launch.
 */
rq_status rq_w4a8_gemm(const int8_t *a_q, const float *a_scales, const uint8_t *w_q, const float *w_scales,
                       int64_t M, int64_t N, int64_t K, int64_t group, void *y, rq_dtype y_dtype, void *stream);

/*
 * rq_sync_status -- wait for `stream` to drain, then report and clear the
 * device error word that bounded waits set when they give up (RQ_ERR_TIMEOUT),
 * or RQ_ERR_CUDA if the stream itself reports an error.  RQ_OK otherwise.
 */
rq_status rq_sync_status(void *stream);

/*
 * rq_selftest_wait_timeout -- exercise the failure-detection path on the device.
 *
 *   Launches one thread that waits, through the same bounded mbarrier wait the
 *   rotation kernels use for their bulk copies, on a barrier that nothing
 *   arrives on.  After `limit_cycles` SM clock cycles the wait gives up, raises
 *   the device error word and the kernel returns; no memory is touched and the
 *   context stays usable.  The next rq_sync_status(stream) returns
 *   RQ_ERR_TIMEOUT (and clears the word).
 *   limit_cycles  1000 .. 4e9 (the production kernels use ~4e9, about 2 s).
 *   Errors: RQ_ERR_INVALID_ARG (limit out of range), RQ_ERR_CUDA (launch).
 */
rq_status rq_selftest_wait_timeout(int64_t limit_cycles, void *stream);

/*
 * rq_probe_f8_mma -- measure the tensor pipe that the W4A4 products run on.
 *
 *   Not an operation of the method (the pages have no counterpart): a
 *   measurement aid for reporting the GEMMs against their own pipe.  One CTA per
 *   SM issues `mmas_per_sm` back-to-back tcgen05.mma kind::f8f6f4 instructions
 *   of shape M128 N256 K32 (E4M3 operands of zeros in shared memory, fp32
 *   accumulator in tensor memory), each 2 * 128 * 256 * 32 = 2,097,152
 *   floating-point operations, then waits (bounded) for them.  Time the call on
 *   `stream` with events: rate = 2097152 * mmas_per_sm * (*ctas) / time.
 *   mmas_per_sm  1 .. 2^30.
 *   ctas         out (may be NULL): CTAs launched (the SM count).
 *   Errors: RQ_ERR_INVALID_ARG (count out of range), RQ_ERR_CUDA (launch); a
 *   wait that gives up sets the error word that rq_sync_status reads.
 */
rq_status rq_probe_f8_mma(int64_t mmas_per_sm, int32_t *ctas, void *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *rq_status_string(rq_status status);

/* Library ABI version: (major << 16) | minor. */
uint32_t rq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RQ_H */
