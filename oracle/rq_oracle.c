/*
 * rq_oracle.c -- plain, slow, single-threaded fp64 oracle for the rotation-based
 * W4A4 hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * constant with the CUDA library, and it never reads anything the CUDA library
 * produced.
 *
 * Sources (page title, then section / equation):
 *   [ROT]  "Rotational Quantization: How Orthogonal Transforms and Hadamard
 *          Incoherence Enable Outlier-Free Low-Bit Inference" (llms.blog)
 *   [QR]   aicassindra.com, quantization series, "QuaRot" page
 *   [SQ]   aicassindra.com, quantization series, "SpinQuant" page
 *
 * Every function states the passage it follows.  Where the pages are silent the
 * reading taken is stated at the function ("reading: ...").
 *
 * Parity status: every function below is pinned by the CPU tests (closed forms,
 * library routines, brute force, published test vectors); none is "parity
 * unpinned".
 *
 * Compile with -ffp-contract=off so that no multiply-add is fused: the results
 * are then the same on x86-64 and aarch64 hosts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define RQO_OK 0
#define RQO_ERR_ARG 1
#define RQO_ERR_OVERFLOW 2
#define RQO_ERR_NOMEM 3

/* flags bit 0: rotation form.
 *   0: y = (x H_n) diag(s)    -- R = H_d diag(s)            [ROT] §Incoherence, eq. R = H_d·diag(s)
 *   1: y = (x diag(s)) H_n    -- sign flip then transform   (the "x·diag(±1)·H_n/√n" form)
 * Both are orthogonal and each is the transpose of the other (H_n is symmetric). */
#define RQO_SIGNS_FIRST 1u

/* ------------------------------------------------------------------------- */
/* Random signs.                                                              */
/* ------------------------------------------------------------------------- */

/* SplitMix64, as published by Steele, Lea and Flood ("Fast splittable
 * pseudorandom number generators", OOPSLA 2014) and in Vigna's reference
 * splitmix64.c: the state advances by the golden-ratio increment before each
 * output, and each output is the state passed through two xor-shift-multiply
 * rounds and a final xor-shift.  Returns output number i (0-based) of the
 * stream seeded with `seed`, i.e. the mix of seed + (i+1)*increment. */
uint64_t rqo_splitmix64(uint64_t seed, uint64_t i)
{
    const uint64_t golden_gamma = 0x9e3779b97f4a7c15ULL;
    uint64_t z = seed + (i + 1u) * golden_gamma;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* Rademacher vector s in {-1,+1}^n: [ROT] §Incoherence (each sign drawn at
 * random, +1 or -1 alike).  Reading: s_i = +1 when the top bit of SplitMix64 output i is 0,
 * else -1.  The pages fix no generator; this one is ours. */
void rqo_signs(uint64_t seed, int64_t n, int8_t *s)
{
    for (int64_t i = 0; i < n; ++i)
        s[i] = (rqo_splitmix64(seed, (uint64_t)i) >> 63) ? (int8_t)-1 : (int8_t)1;
}

/* ------------------------------------------------------------------------- */
/* Hadamard transform.                                                        */
/* ------------------------------------------------------------------------- */

/* x <- H_n x for the normalized Sylvester Hadamard matrix, written as the
 * recursion of [ROT] §Incoherence: H_1 = [1] and
 *     H_2k = (1/sqrt 2) [[H_k, H_k], [H_k, -H_k]].
 * Applying the block form to x = [top; bottom] gives
 *     H_2k x = (1/sqrt 2) [H_k top + H_k bottom; H_k top - H_k bottom],
 * so the routine transforms each half recursively and then combines.
 * H_n is symmetric, so the same routine computes the row-vector product x H_n. */
static void hadamard_rec(double *x, int64_t n)
{
    if (n == 1)
        return;
    const int64_t h = n / 2;
    hadamard_rec(x, h);
    hadamard_rec(x + h, h);
    const double r = 1.0 / sqrt(2.0);
    for (int64_t i = 0; i < h; ++i) {
        const double a = x[i];
        const double b = x[i + h];
        x[i] = (a + b) * r;
        x[i + h] = (a - b) * r;
    }
}

static int is_pow2(int64_t n) { return n >= 1 && (n & (n - 1)) == 0; }

/* ------------------------------------------------------------------------- */
/* Sizes that are not powers of two: n = m 2^k with a Hadamard block H_m.      */
/* ------------------------------------------------------------------------- */

/* Quadratic character of x modulo the prime q: 0 for x = 0, +1 for a nonzero
 * square, -1 otherwise (found by listing the squares). */
static int qchar(int64_t x, int q)
{
    x %= q;
    if (x < 0)
        x += q;
    if (x == 0)
        return 0;
    for (int64_t y = 1; y < q; ++y)
        if ((y * y) % q == x)
            return 1;
    return -1;
}

/* Hadamard matrix of order m in {12, 20, 28} (row-major int8, entries +-1).
 * [ROT] §The Computational Cost of Arbitrary Rotations / §SpinQuant mention sizes
 * that are not powers of two (padding, or products of Sylvester-compatible
 * sizes); reading: n = m 2^k with R = (H_m (x) H_{2^k}) / sqrt(n) and H_m from
 * Paley's constructions over the prime field GF(q):
 *   Jacobsthal matrix Q[i][j] = qchar(j - i), i, j < q;
 *   m = 12, 20 (Paley I, q = 11, 19, q = 3 mod 4): S = [[0, 1^T], [-1, Q]],
 *     H = I + S;
 *   m = 28 (Paley II, q = 13, q = 1 mod 4): S = [[0, 1^T], [1, Q]],
 *     H = S (x) [[1, 1], [1, -1]] + I (x) [[1, -1], [-1, -1]].
 * Returns RQO_ERR_ARG for any other m. */
int rqo_paley(int m, int8_t *H)
{
    int q, two;
    if (m == 12) {
        q = 11;
        two = 0;
    } else if (m == 20) {
        q = 19;
        two = 0;
    } else if (m == 28) {
        q = 13;
        two = 1;
    } else {
        return RQO_ERR_ARG;
    }
    const int o = q + 1;
    int S[32][32];
    for (int i = 0; i < o; ++i)
        for (int j = 0; j < o; ++j) {
            if (i == 0 && j == 0)
                S[i][j] = 0;
            else if (i == 0)
                S[i][j] = 1;
            else if (j == 0)
                S[i][j] = two ? 1 : -1;
            else
                S[i][j] = qchar((int64_t)(j - 1) - (int64_t)(i - 1), q);
        }
    if (!two) {
        for (int i = 0; i < o; ++i)
            for (int j = 0; j < o; ++j)
                H[i * m + j] = (int8_t)(S[i][j] + (i == j ? 1 : 0));
    } else {
        const int A[2][2] = {{1, 1}, {1, -1}};
        const int B[2][2] = {{1, -1}, {-1, -1}};
        for (int i = 0; i < o; ++i)
            for (int j = 0; j < o; ++j)
                for (int u = 0; u < 2; ++u)
                    for (int v = 0; v < 2; ++v)
                        H[(2 * i + u) * m + (2 * j + v)] =
                            (int8_t)(S[i][j] * A[u][v] + (i == j ? B[u][v] : 0));
    }
    return RQO_OK;
}

/* n = m 2^k with m in {1, 12, 20, 28} (m = 1: a power of two).  Returns m, or 0
 * when n has no such form. */
static int rot_block(int64_t n)
{
    if (is_pow2(n))
        return 1;
    const int ms[3] = {12, 20, 28};
    for (int i = 0; i < 3; ++i)
        if (n % ms[i] == 0 && is_pow2(n / ms[i]))
            return ms[i];
    return 0;
}

int rqo_hadamard(double *x, int64_t n)
{
    if (!is_pow2(n))
        return RQO_ERR_ARG;
    hadamard_rec(x, n);
    return RQO_OK;
}

/* y = x (H_m (x) H_b) / sqrt(m) for n = m b, b a power of two: the normalized
 * Sylvester transform of every length-b segment a (elements a b .. a b + b - 1),
 * then, for every offset j, the row-vector product of the m values x[a b + j]
 * with H_m / sqrt(m): out[a' b + j] = sum_a x[a b + j] H_m[a][a'] / sqrt(m). */
static int kron_rotate(double *y, int64_t n, int m)
{
    const int64_t b = n / m;
    for (int a = 0; a < m; ++a)
        hadamard_rec(y + a * b, b);
    if (m == 1)
        return RQO_OK;
    int8_t H[28 * 28];
    double col[28];
    rqo_paley(m, H);
    const double r = 1.0 / sqrt((double)m);
    for (int64_t j = 0; j < b; ++j) {
        for (int a = 0; a < m; ++a)
            col[a] = y[a * b + j];
        for (int a2 = 0; a2 < m; ++a2) {
            double acc = 0.0;
            for (int a = 0; a < m; ++a)
                acc += col[a] * (double)H[a * m + a2];
            y[a2 * b + j] = acc * r;
        }
    }
    return RQO_OK;
}

/* One rotated row y = x R for the randomized Hadamard R, in the form chosen by
 * flags bit 0 (see RQO_SIGNS_FIRST).  [ROT] §Incoherence, eq. R = H_d·diag(s)
 * and eq. x~ = x R.  For n = m 2^k (m in {12, 20, 28}) H_d is H_m (x) H_{2^k}
 * (see rqo_paley). */
int rqo_rotate_row(const double *x, int64_t n, const int8_t *s, uint32_t flags, double *y)
{
    const int m = rot_block(n);
    if (m == 0)
        return RQO_ERR_ARG;
    if (flags & RQO_SIGNS_FIRST) {
        for (int64_t i = 0; i < n; ++i)
            y[i] = x[i] * (double)s[i];
        kron_rotate(y, n, m);
    } else {
        memcpy(y, x, (size_t)n * sizeof(double));
        kron_rotate(y, n, m);
        for (int64_t i = 0; i < n; ++i)
            y[i] = y[i] * (double)s[i];
    }
    return RQO_OK;
}

/* ------------------------------------------------------------------------- */
/* Symmetric INT4 quantization and packing.                                   */
/* ------------------------------------------------------------------------- */

/* Per-row symmetric INT4: scale = max|y| / 7, q = clamp(round_half_even(y / scale),
 * -8, 7).  The pages name an "INT4 quantizer" with per-channel scales ([QR]
 * §The architecture; [SQ] §The architecture) and the asymmetric step
 * (max-min)/(2^b-1) ([ROT] §The Activation Outlier Bottleneck); the symmetric
 * absmax/7 form with round-half-even and the [-8,7] clamp is the reading taken.
 * Reading for an all-zero row: scale = 0 and every code 0.
 * nearbyint() rounds in the default mode, which is round-half-to-even.
 * `ratio` (nullable) receives y/scale, used by the tests' tie-window count. */
void rqo_quant_row(const double *y, int64_t n, int8_t *q, double *scale, double *ratio)
{
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double a = fabs(y[i]);
        if (a > amax)
            amax = a;
    }
    if (amax == 0.0) {
        *scale = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            q[i] = 0;
            if (ratio)
                ratio[i] = 0.0;
        }
        return;
    }
    const double sc = amax / 7.0;
    *scale = sc;
    for (int64_t i = 0; i < n; ++i) {
        const double r = y[i] / sc;
        double c = nearbyint(r);
        if (c < -8.0)
            c = -8.0;
        if (c > 7.0)
            c = 7.0;
        q[i] = (int8_t)c;
        if (ratio)
            ratio[i] = r;
    }
}

/* Nibble packing (reading; the pages fix no layout): byte j holds element 2j in
 * bits 3..0 and element 2j+1 in bits 7..4, each as a 4-bit two's-complement
 * code.  n must be even. */
void rqo_pack_row(const int8_t *q, int64_t n, uint8_t *out)
{
    for (int64_t j = 0; j < n / 2; ++j) {
        const unsigned lo = (unsigned)q[2 * j] & 0xFu;
        const unsigned hi = (unsigned)q[2 * j + 1] & 0xFu;
        out[j] = (uint8_t)(lo | (hi << 4));
    }
}

static int8_t nibble_to_int(unsigned v)
{
    v &= 0xFu;
    return (int8_t)(v >= 8u ? (int)v - 16 : (int)v);
}

void rqo_unpack_row(const uint8_t *in, int64_t n, int8_t *q)
{
    for (int64_t j = 0; j < n / 2; ++j) {
        q[2 * j] = nibble_to_int(in[j]);
        q[2 * j + 1] = nibble_to_int((unsigned)in[j] >> 4);
    }
}

/* ------------------------------------------------------------------------- */
/* Online rotation + quantization of a row-major matrix.                      */
/* ------------------------------------------------------------------------- */

/* For each row r of x (rows x n, row stride ld_x, fp64): y = x_r R, then the
 * per-row INT4 quantizer and packing.  Outputs: q (rows x n/2 bytes, row stride
 * n/2), scales (rows, fp32, rounded from the fp64 scale), and optionally the
 * fp64 rotated rows y (rows x n) and the ratios y/scale (rows x n).
 * [QR] §End-to-end flow (the activation is rotated on the fly by a Hadamard
 * transform, then quantized to INT4); [ROT] §Weight Absorption,
 * 2. Online Fast Walsh-Hadamard Transform. */
int rqo_fwht_quant(const double *x, int64_t rows, int64_t n, int64_t ld_x, uint64_t seed,
                   uint32_t flags, uint8_t *q, float *scales, double *y_out, double *ratio_out)
{
    if (rot_block(n) == 0 || n < 2 || (n & 1) || rows < 0 || ld_x < n)
        return RQO_ERR_ARG;
    int8_t *s = (int8_t *)malloc((size_t)n);
    double *y = (double *)malloc((size_t)n * sizeof(double));
    int8_t *codes = (int8_t *)malloc((size_t)n);
    if (!s || !y || !codes) {
        free(s);
        free(y);
        free(codes);
        return RQO_ERR_NOMEM;
    }
    rqo_signs(seed, n, s);
    for (int64_t r = 0; r < rows; ++r) {
        double sc = 0.0;
        rqo_rotate_row(x + r * ld_x, n, s, flags, y);
        rqo_quant_row(y, n, codes, &sc, ratio_out ? ratio_out + r * n : NULL);
        rqo_pack_row(codes, n, q + r * (n / 2));
        scales[r] = (float)sc;
        if (y_out)
            memcpy(y_out + r * n, y, (size_t)n * sizeof(double));
    }
    free(s);
    free(y);
    free(codes);
    return RQO_OK;
}

/* ------------------------------------------------------------------------- */
/* W4A4 linear layer.                                                         */
/* ------------------------------------------------------------------------- */

/* acc[m][c] = sum_k qa[m][k] * qw[c][k] in exact integer arithmetic, and
 * y[m][c] = acc[m][c] * sa[m] * sw[c] (scales widened from fp32 to fp64).
 * A is M x K (packed, M x K/2 bytes), W is N x K (packed, N x K/2 bytes): both
 * K-major, W holding one output channel per row.  The integer form of the
 * rotated product Q(XR)·Q(R^T W) of [ROT] §Learned Orthogonal Rotations
 * (loss L(S)) and §The Principle of Computational Invariance (Y = (XR)(R^T W));
 * [QR] §End-to-end flow (the INT4 activation meets the INT4 weights that carry
 * the folded rotation).
 * Either output may be NULL.  Returns RQO_ERR_OVERFLOW if an accumulator
 * leaves the int32 range. */
int rqo_w4a4_gemm(const uint8_t *aq, const float *sa, const uint8_t *wq, const float *sw,
                  int64_t M, int64_t N, int64_t K, int64_t *acc, double *y)
{
    if (M < 0 || N < 0 || K < 0 || (K & 1))
        return RQO_ERR_ARG;
    int8_t *a = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1) * (size_t)(N > 0 ? N : 1));
    if (!a || !w) {
        free(a);
        free(w);
        return RQO_ERR_NOMEM;
    }
    for (int64_t c = 0; c < N; ++c)
        rqo_unpack_row(wq + c * (K / 2), K, w + c * K);
    int status = RQO_OK;
    for (int64_t m = 0; m < M; ++m) {
        rqo_unpack_row(aq + m * (K / 2), K, a);
        for (int64_t c = 0; c < N; ++c) {
            int64_t s = 0;
            const int8_t *wc = w + c * K;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)a[k] * (int64_t)wc[k];
            if (s > INT32_MAX || s < INT32_MIN)
                status = RQO_ERR_OVERFLOW;
            if (acc)
                acc[m * N + c] = s;
            if (y)
                y[m * N + c] = (double)s * (double)sa[m] * (double)sw[c];
        }
    }
    free(a);
    free(w);
    return status;
}

/* The same products for a list of (m, c) output positions only, for checks at
 * sizes where the full product would take too long on one core. */
int rqo_w4a4_gemm_entries(const uint8_t *aq, const float *sa, const uint8_t *wq, const float *sw,
                          int64_t K, int64_t count, const int64_t *ms, const int64_t *cs,
                          int64_t *acc, double *y)
{
    if (K < 0 || (K & 1) || count < 0)
        return RQO_ERR_ARG;
    int8_t *a = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    if (!a || !w) {
        free(a);
        free(w);
        return RQO_ERR_NOMEM;
    }
    int status = RQO_OK;
    for (int64_t e = 0; e < count; ++e) {
        rqo_unpack_row(aq + ms[e] * (K / 2), K, a);
        rqo_unpack_row(wq + cs[e] * (K / 2), K, w);
        int64_t s = 0;
        for (int64_t k = 0; k < K; ++k)
            s += (int64_t)a[k] * (int64_t)w[k];
        if (s > INT32_MAX || s < INT32_MIN)
            status = RQO_ERR_OVERFLOW;
        if (acc)
            acc[e] = s;
        if (y)
            y[e] = (double)s * (double)sa[ms[e]] * (double)sw[cs[e]];
    }
    free(a);
    free(w);
    return status;
}

/* ------------------------------------------------------------------------- */
/* KV cache write: head-wise rotation + quantization.                         */
/* ------------------------------------------------------------------------- */

/* K and V, each [tokens][heads][head_dim] (fp64 here), are rotated per (token,
 * head) vector by the randomized Hadamard of size head_dim and quantized per
 * (token, head): [QR] §The architecture (the KV-cache rotation box: each
 * token's keys and values are rotated, then quantized, before they are stored) and
 * §End-to-end flow, "The KV cache"; [ROT] §Hardware Execution, 2. End-to-End KV
 * Cache Footprint Reduction.  Reading: one sign vector of length head_dim drawn
 * from `seed`, shared by every head and by K and V.  Either tensor may be NULL
 * (its outputs are then untouched). */
int rqo_kv_rotate_quant(const double *k, const double *v, int64_t tokens, int64_t heads,
                        int64_t head_dim, uint64_t seed, uint32_t flags, uint8_t *kq,
                        float *ks, uint8_t *vq, float *vs)
{
    if (tokens < 0 || heads < 0 || !is_pow2(head_dim) || head_dim < 2)
        return RQO_ERR_ARG;
    const int64_t rows = tokens * heads;
    int st = RQO_OK;
    if (k)
        st = rqo_fwht_quant(k, rows, head_dim, head_dim, seed, flags, kq, ks, NULL, NULL);
    if (st == RQO_OK && v)
        st = rqo_fwht_quant(v, rows, head_dim, head_dim, seed, flags, vq, vs, NULL, NULL);
    return st;
}

/* ------------------------------------------------------------------------- */
/* Attention read of the rotated INT4 cache.                                  */
/* ------------------------------------------------------------------------- */

/* Decode-time attention over a cache written by rqo_kv_rotate_quant.  [QR]
 * §End-to-end flow, "The KV cache": on a later token attention reads the
 * four-bit rotated cache, and rotation invariance keeps the scores those of the
 * full-precision computation; [QR] §The architecture (the invariance box: a
 * rotation is cancelled by its transpose downstream, or by a Hadamard of its
 * own).
 *
 * For every query row m and head h (q is [M][heads][head_dim], fp64):
 *   q~   = q[m][h] R                       (the cache's rotation, same seed/flags)
 *   k^_t = unpack(kq[t][h]) * ks[t][h]     (dequantized rotated key, fp64)
 *   e_t  = softmax_scale * (q~ . k^_t),   p_t = exp(e_t - max e) / sum exp(e - max e)
 *   o~   = sum_t p_t * v^_t                (v^ as k^)
 *   out  = o~ R^T, or o~ itself when `rotated_out` is set.
 * Since R is orthogonal, q~ . k^_t = q . (k^_t R^T): the scores are those of
 * plain attention on the cache taken back to the original basis.  R^T is the
 * rotation with the other sign side (H is symmetric), i.e. rqo_rotate_row with
 * flags bit 0 flipped.
 * Readings: every query row sees every cached token (no mask); one sign vector
 * for all heads, as the cache write.  out is [M][heads][head_dim], fp64. */
int rqo_attn_decode(const double *q, int64_t M, int64_t heads, int64_t head_dim, const uint8_t *kq,
                    const float *ks, const uint8_t *vq, const float *vs, int64_t tokens, uint64_t seed,
                    uint32_t flags, double softmax_scale, int rotated_out, double *out)
{
    if (M < 0 || heads < 0 || tokens < 1 || !is_pow2(head_dim) || head_dim < 2)
        return RQO_ERR_ARG;
    const int64_t D = head_dim;
    int8_t *s = (int8_t *)malloc((size_t)D);
    double *qr = (double *)malloc((size_t)D * sizeof(double));
    double *o = (double *)malloc((size_t)D * sizeof(double));
    double *e = (double *)malloc((size_t)tokens * sizeof(double));
    int8_t *c = (int8_t *)malloc((size_t)D);
    if (!s || !qr || !o || !e || !c) {
        free(s);
        free(qr);
        free(o);
        free(e);
        free(c);
        return RQO_ERR_NOMEM;
    }
    rqo_signs(seed, D, s);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t h = 0; h < heads; ++h) {
            rqo_rotate_row(q + (m * heads + h) * D, D, s, flags, qr);
            double emax = -INFINITY;
            for (int64_t t = 0; t < tokens; ++t) {
                rqo_unpack_row(kq + (t * heads + h) * (D / 2), D, c);
                const double sk = (double)ks[t * heads + h];
                double dot = 0.0;
                for (int64_t j = 0; j < D; ++j)
                    dot += qr[j] * ((double)c[j] * sk);
                e[t] = softmax_scale * dot;
                if (e[t] > emax)
                    emax = e[t];
            }
            double z = 0.0;
            for (int64_t t = 0; t < tokens; ++t) {
                e[t] = exp(e[t] - emax);
                z += e[t];
            }
            for (int64_t j = 0; j < D; ++j)
                o[j] = 0.0;
            for (int64_t t = 0; t < tokens; ++t) {
                rqo_unpack_row(vq + (t * heads + h) * (D / 2), D, c);
                const double pv = (e[t] / z) * (double)vs[t * heads + h];
                for (int64_t j = 0; j < D; ++j)
                    o[j] += pv * (double)c[j];
            }
            double *dst = out + (m * heads + h) * D;
            if (rotated_out)
                memcpy(dst, o, (size_t)D * sizeof(double));
            else
                rqo_rotate_row(o, D, s, flags ^ RQO_SIGNS_FIRST, dst);
        }
    }
    free(s);
    free(qr);
    free(o);
    free(e);
    free(c);
    return RQO_OK;
}

/* ------------------------------------------------------------------------- */
/* W4A8 and per-group weight scales.                                          */
/* ------------------------------------------------------------------------- */

/* Per-row symmetric INT8 for activations: [SQ] §The architecture (after the
 * rotations, weights go to INT4 and activations to INT8, with per-channel or
 * per-group scales), §End-to-end flow (the rotated activation becomes INT8).
 * Reading: scale = max|y| / 127, q = clamp(round_half_even(y / scale), -128, 127)
 * (-128 never occurs with this scale); an all-zero row gets scale 0, codes 0.
 * `ratio` (nullable) receives y / scale. */
void rqo_quant_row8(const double *y, int64_t n, int8_t *q, double *scale, double *ratio)
{
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i)
        if (fabs(y[i]) > amax)
            amax = fabs(y[i]);
    *scale = amax / 127.0;
    for (int64_t i = 0; i < n; ++i) {
        const double r = amax > 0.0 ? y[i] / *scale : 0.0;
        double c = nearbyint(r);
        if (c < -128.0)
            c = -128.0;
        if (c > 127.0)
            c = 127.0;
        q[i] = (int8_t)c;
        if (ratio)
            ratio[i] = r;
    }
}

/* For each row of x: y = x R, then per-row INT8 codes (rows x n bytes) and fp32
 * scales.  Optional fp64 ratios y / scale (rows x n). */
int rqo_fwht_quant8(const double *x, int64_t rows, int64_t n, int64_t ld_x, uint64_t seed, uint32_t flags,
                    int8_t *q, float *scales, double *ratio_out)
{
    if (rot_block(n) == 0 || rows < 0 || ld_x < n)
        return RQO_ERR_ARG;
    int8_t *s = (int8_t *)malloc((size_t)n);
    double *y = (double *)malloc((size_t)n * sizeof(double));
    if (!s || !y) {
        free(s);
        free(y);
        return RQO_ERR_NOMEM;
    }
    rqo_signs(seed, n, s);
    for (int64_t r = 0; r < rows; ++r) {
        double sc = 0.0;
        rqo_rotate_row(x + r * ld_x, n, s, flags, y);
        rqo_quant_row8(y, n, q + r * n, &sc, ratio_out ? ratio_out + r * n : NULL);
        scales[r] = (float)sc;
    }
    free(s);
    free(y);
    return RQO_OK;
}

/* Per-group INT4 weights ([SQ] §The architecture, "per-group scales"): each row
 * of W^T is rotated (the fold), then every group of `group` consecutive elements
 * is quantized on its own with the INT4 rule of rqo_quant_row (scale =
 * max|y_g| / 7).  q: rows x n/2 packed; scales: rows x n/group fp32; ratio
 * (nullable): rows x n. */
int rqo_fwht_quant_groups(const double *x, int64_t rows, int64_t n, int64_t ld_x, uint64_t seed, uint32_t flags,
                          int64_t group, uint8_t *q, float *scales, double *ratio_out)
{
    if (rot_block(n) == 0 || rows < 0 || ld_x < n || group < 2 || (group & 1) || n % group)
        return RQO_ERR_ARG;
    int8_t *s = (int8_t *)malloc((size_t)n);
    double *y = (double *)malloc((size_t)n * sizeof(double));
    int8_t *codes = (int8_t *)malloc((size_t)n);
    if (!s || !y || !codes) {
        free(s);
        free(y);
        free(codes);
        return RQO_ERR_NOMEM;
    }
    rqo_signs(seed, n, s);
    const int64_t ng = n / group;
    for (int64_t r = 0; r < rows; ++r) {
        rqo_rotate_row(x + r * ld_x, n, s, flags, y);
        for (int64_t g = 0; g < ng; ++g) {
            double sc = 0.0;
            rqo_quant_row(y + g * group, group, codes + g * group, &sc,
                          ratio_out ? ratio_out + r * n + g * group : NULL);
            scales[r * ng + g] = (float)sc;
        }
        rqo_pack_row(codes, n, q + r * (n / 2));
    }
    free(s);
    free(y);
    free(codes);
    return RQO_OK;
}

/* W4A8 linear layer: INT8 activations (M x K bytes, per-row scales sa) times
 * packed INT4 weights (N x K/2, one output channel per row) with per-group
 * scales sw (N x K/group; group == K is per-channel):
 *   acc_g[m][c] = sum_{k in group g} qa[m][k] qw[c][k]   (exact integers)
 *   y[m][c]     = sa[m] * sum_g sw[c][g] * acc_g[m][c]    (fp64)
 * [SQ] §End-to-end flow (the INT8 rotated activation is multiplied with the INT4
 * rotated weights), §The architecture.
 * acc (nullable, per-channel only): the whole-K integer sums. */
int rqo_w4a8_gemm(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M, int64_t N,
                  int64_t K, int64_t group, int64_t *acc, double *y)
{
    if (M < 0 || N < 0 || K <= 0 || (K & 1) || group <= 0 || K % group || (acc && group != K))
        return RQO_ERR_ARG;
    int8_t *wrow = (int8_t *)malloc((size_t)K);
    if (!wrow)
        return RQO_ERR_NOMEM;
    const int64_t ng = K / group;
    for (int64_t c = 0; c < N; ++c) {
        rqo_unpack_row(wq + c * (K / 2), K, wrow);
        for (int64_t m = 0; m < M; ++m) {
            double yy = 0.0;
            int64_t total = 0;
            for (int64_t g = 0; g < ng; ++g) {
                int64_t a = 0;
                for (int64_t k = g * group; k < (g + 1) * group; ++k)
                    a += (int64_t)aq[m * K + k] * (int64_t)wrow[k];
                total += a;
                yy += (double)sw[c * ng + g] * (double)a;
            }
            if (acc)
                acc[m * N + c] = total;
            if (y)
                y[m * N + c] = (double)sa[m] * yy;
        }
    }
    free(wrow);
    return RQO_OK;
}
