// fwht_kron.cu -- rotation + INT4 quantization for row lengths n = m 2^k that are
// not powers of two (m in {12, 20, 28}, 2^k in [32, 1024]), on sm_103a.
//
// The pages mention sizes that are not powers of two ("The Computational Cost of
// Arbitrary Rotations"; "SpinQuant": padding, or products of Sylvester-compatible
// sizes).  Here R = diag(s) (H_m (x) H_{2^k}) / sqrt(n) (signs first; the other
// flag puts diag(s) after), with element a 2^k + j of a row in segment a at offset
// j, and H_m a Hadamard matrix from Paley's constructions over GF(q):
//   Jacobsthal matrix Q[i][j] = chi(j - i), chi the quadratic character mod q;
//   m = 12, 20 (q = 11, 19): S = [[0, 1^T], [-1, Q]], H = I + S;
//   m = 28 (q = 13):         S = [[0, 1^T], [1, Q]],
//                            H = S (x) [[1, 1], [1, -1]] + I (x) [[1, -1], [-1, -1]].
// Examples: 14336 = 28 x 512 and 28672 = 28 x 1024 (FFN widths), 3072 = 12 x 256.
//
// Design (one CTA per row at a time, persistent over rows, 8 warps, as many CTAs
// per SM as fit):
//  * the CTA's signs (n SplitMix64 outputs) go into a shared table once, as
//    words with bit 15 / 31 for elements 2j / 2j + 1, so one XOR flips a pair of
//    16-bit inputs;
//  * step 1: warp w takes segments w, w + 8, ...: a lane loads 2^k / 32
//    consecutive elements, flips signs (signs first), runs the butterflies of
//    its element bits in registers and of the lane bits by shuffles, and writes
//    fp32 to the shared row buffer;
//  * step 2: a thread owns column pairs (j, j + 1): it reads the m values of
//    each column from the m segments and forms the m outputs sum_a H[a][a'] x_a
//    with f32x2 adds and subtracts (H_m is built at compile time; for m = 28 the
//    Paley II structure halves the additions), flips signs (signs after), and
//    tracks the row's absmax;
//  * a block reduction gives the scale; the same threads quantize (one f32x2 FMA
//    against a 1.5 * 2^23 bias per pair, round half to even, as the power-of-two
//    kernels) and store one byte per column pair and segment;
//  * code modes as in the power-of-two kernels: INT8 codes per row (two bytes
//    per column pair and segment), or INT4 with one scale per group of 128
//    consecutive elements (n is a multiple of 128: a warp per group reads the
//    finished row buffer, and the quantizer takes its group's multiplier).
// Bound: issue (per element ~20 instructions for the shuffled stages and m/2
// FMAs for H_m), not HBM.
#include "rq.h"
#include "rq_internal.h"
#include "rot_device.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

namespace rq {
namespace {

constexpr int kKWarps = 8;
constexpr int kKThreads = 32 * kKWarps;

struct KronParams {
    const void *x;
    int64_t ld, rows;
    uint8_t *q;
    float *scales;
    float *y;
    uint64_t seed;
    uint32_t flags;
    float inv_sqrt_n;
};

// ---- Paley Hadamard blocks, built at compile time ----
struct Block {
    signed char h[28][28];
};

constexpr int qchar_ce(int x, int q) {
    x %= q;
    if (x < 0) x += q;
    if (x == 0) return 0;
    for (int y = 1; y < q; ++y)
        if ((y * y) % q == x) return 1;
    return -1;
}

constexpr Block make_block(int m) {
    Block b{};
    const int q = m == 12 ? 11 : (m == 20 ? 19 : 13);
    const bool two = m == 28;
    const int o = q + 1;
    int S[14][14] = {};
    int S20[20][20] = {};
    for (int i = 0; i < o; ++i)
        for (int j = 0; j < o; ++j) {
            int v = 0;
            if (i == 0 && j == 0) v = 0;
            else if (i == 0) v = 1;
            else if (j == 0) v = two ? 1 : -1;
            else v = qchar_ce((j - 1) - (i - 1), q);
            if (two) S[i][j] = v;
            else S20[i][j] = v;
        }
    if (!two) {
        for (int i = 0; i < o; ++i)
            for (int j = 0; j < o; ++j) b.h[i][j] = (signed char)(S20[i][j] + (i == j ? 1 : 0));
    } else {
        const int A[2][2] = {{1, 1}, {1, -1}};
        const int Bm[2][2] = {{1, -1}, {-1, -1}};
        for (int i = 0; i < o; ++i)
            for (int j = 0; j < o; ++j)
                for (int u = 0; u < 2; ++u)
                    for (int v = 0; v < 2; ++v)
                        b.h[2 * i + u][2 * j + v] = (signed char)(S[i][j] * A[u][v] + (i == j ? Bm[u][v] : 0));
    }
    return b;
}

template <int M>
struct BlockOf {
    static constexpr Block value = make_block(M);
};

template <int IN>
__device__ __forceinline__ float ld_elem(const void *base, int64_t i) {
    if constexpr (IN == IN_F32) return static_cast<const float *>(base)[i];
    else if constexpr (IN == IN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    else return __half2float(static_cast<const __half *>(base)[i]);
}

template <int IN, int M, int LOGB>
__global__ void __launch_bounds__(kKThreads, 2) fwht_kron_kernel(const __grid_constant__ KronParams p) {
    constexpr int B = 1 << LOGB, N = M * B, E = B / 32;
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    extern __shared__ __align__(16) unsigned char kraw[];
    float *row = reinterpret_cast<float *>(kraw);                       // N floats
    uint32_t *sgn = reinterpret_cast<uint32_t *>(row + N);               // N / 2 sign words
    float *red = reinterpret_cast<float *>(sgn + N / 2);                 // kKWarps
    float *ginv = red + kKWarps;                                          // N / 128 (per-group codes)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool signs_first = (p.flags & 1u) != 0;
    const bool i8 = (p.flags & (RQ_INT8_CODES | RQ_INT4_BYTES)) != 0, per_group = (p.flags & RQ_GROUP_SCALES) != 0;
    static_assert(N % 128 == 0, "m is a multiple of 4 and 2^k >= 32");
    const uint32_t msel = signs_first ? 0xffffffffu : 0u;

    // sign word j: bit 15 / bit 31 set when element 2j / 2j + 1 takes -1 (top bit of
    // SplitMix64 output i), so that one XOR flips a bf16 / fp16 pair, and the high
    // word's bit 31 / the low word shifted by 16 flip fp32 elements
    for (int jw = threadIdx.x; jw < N / 2; jw += kKThreads) {
        const uint32_t a = (uint32_t)(splitmix64_at(p.seed, 2ull * jw) >> 63);
        const uint32_t b = (uint32_t)(splitmix64_at(p.seed, 2ull * jw + 1) >> 63);
        sgn[jw] = (a << 15) | (b << 31);
    }
    __syncthreads();

    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
        const char *xrow = static_cast<const char *>(p.x) + r * p.ld * ES;
        // ---- step 1: the Sylvester transform of every length-B segment ----
        // A warp's segments are a = warp, warp + 8, ...: the raw 16-byte granules of
        // the next one are loaded before the current one is transformed, so a
        // segment's load latency overlaps the previous segment's work.
        constexpr int NG = E * ES >= 16 ? E * ES / 16 : 1;   // granules per lane and segment
        uint4 nxt[NG];
        auto load_seg = [&](int a) {
            if constexpr (E * ES >= 16) {
#pragma unroll
                for (int c = 0; c < NG; ++c)
                    nxt[c] = *reinterpret_cast<const uint4 *>(xrow + (int64_t)(a * B + lane * E) * ES + 16 * c);
            }
        };
        if (warp < M) load_seg(warp);
        for (int a = warp; a < M; a += kKWarps) {
            const int base = a * B + lane * E;
            uint4 cur[NG];
#pragma unroll
            for (int c = 0; c < NG; ++c) cur[c] = nxt[c];
            if (a + kKWarps < M) load_seg(a + kKWarps);
            float v[E];
            if constexpr (E * ES >= 16) {
#pragma unroll
                for (int c = 0; c < E * ES / 16; ++c) {
                    const uint4 g = cur[c];
                    uint32_t w[4] = {g.x, g.y, g.z, g.w};
                    if constexpr (IN == IN_F32) {
                        // elements base + 4c .. + 3: sign words (base + 4c) / 2 and + 1
                        const uint32_t s0 = sgn[(base + 4 * c) / 2] & msel, s1 = sgn[(base + 4 * c) / 2 + 1] & msel;
                        w[0] ^= s0 << 16;
                        w[1] ^= s0 & 0x80000000u;
                        w[2] ^= s1 << 16;
                        w[3] ^= s1 & 0x80000000u;
#pragma unroll
                        for (int k = 0; k < 4; ++k) v[4 * c + k] = __uint_as_float(w[k]);
                    } else {
                        const uint4 m = *reinterpret_cast<const uint4 *>(sgn + (base + 8 * c) / 2);
                        w[0] ^= m.x & msel;
                        w[1] ^= m.y & msel;
                        w[2] ^= m.z & msel;
                        w[3] ^= m.w & msel;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t lo = w[k] & 0xffffu, hi = w[k] >> 16;
                            if constexpr (IN == IN_BF16) {
                                v[8 * c + 2 * k] = __uint_as_float(lo << 16);
                                v[8 * c + 2 * k + 1] = __uint_as_float(hi << 16);
                            } else {
                                v[8 * c + 2 * k] = __half2float(__ushort_as_half((unsigned short)lo));
                                v[8 * c + 2 * k + 1] = __half2float(__ushort_as_half((unsigned short)hi));
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    v[e] = ld_elem<IN>(xrow, base + e);
                    const uint32_t sw = sgn[(base + e) / 2] & msel;
                    const uint32_t bit = ((base + e) & 1) ? (sw & 0x80000000u) : (sw << 16);
                    v[e] = __uint_as_float(__float_as_uint(v[e]) ^ bit);
                }
            }
#pragma unroll
            for (int st = 1; st < E; st <<= 1)
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if (!(e & st)) {
                        const float x0 = v[e], x1 = v[e + st];
                        v[e] = x0 + x1;
                        v[e + st] = x0 - x1;
                    }
            // lane-bit stages: the lower lane keeps v + o, the upper o - v, i.e.
            // v * sg + o with sg = -1 on the upper lane
#pragma unroll
            for (int lm = 1; lm < 32; lm <<= 1) {
                const float sg = (lane & lm) ? -1.f : 1.f;
#pragma unroll
                for (int e = 0; e < E; ++e) v[e] = fmaf(v[e], sg, __shfl_xor_sync(0xffffffffu, v[e], lm));
            }
#pragma unroll
            for (int e = 0; e < E; ++e) row[base + e] = v[e];
        }
        __syncthreads();

        // ---- step 2: H_M across the segments, per column pair (j, j + 1) ----
        constexpr Block H = BlockOf<M>::value;
        float amax = 0.f;
        for (int j = 2 * threadIdx.x; j < B; j += 2 * kKThreads) {
            pair_t col[M];
#pragma unroll
            for (int a = 0; a < M; ++a) col[a] = *reinterpret_cast<const pair_t *>(row + a * B + j);
            pair_t out[M];
            if constexpr (M == 28) {
                // Paley II: H = S (x) [[1, 1], [1, -1]] + I (x) [[1, -1], [-1, -1]], so with
                // p_i = x_2i + x_2i+1, d_i = x_2i - x_2i+1 (S[i][j] = H[2i][2j] off the
                // diagonal, 0 on it):
                //   (xH)_2j = sum_i S[i][j] p_i + d_j,  (xH)_2j+1 = sum_i S[i][j] d_i - p_j
                pair_t pp[14], dd[14];
#pragma unroll
                for (int i = 0; i < 14; ++i) {
                    pp[i] = add2(col[2 * i], col[2 * i + 1]);
                    dd[i] = sub2(col[2 * i], col[2 * i + 1]);
                }
#pragma unroll
                for (int jj = 0; jj < 14; ++jj) {
                    pair_t e0 = dd[jj], e1 = sub2(0ull, pp[jj]);
#pragma unroll
                    for (int i = 0; i < 14; ++i) {
                        if (i == jj) continue;
                        if (H.h[2 * i][2 * jj] > 0) {
                            e0 = add2(e0, pp[i]);
                            e1 = add2(e1, dd[i]);
                        } else {
                            e0 = sub2(e0, pp[i]);
                            e1 = sub2(e1, dd[i]);
                        }
                    }
                    out[2 * jj] = e0;
                    out[2 * jj + 1] = e1;
                }
            } else {
#pragma unroll
                for (int a2 = 0; a2 < M; ++a2) {
                    pair_t acc = 0ull;
#pragma unroll
                    for (int a = 0; a < M; ++a) acc = H.h[a][a2] > 0 ? add2(acc, col[a]) : sub2(acc, col[a]);
                    out[a2] = acc;
                }
            }
#pragma unroll
            for (int a2 = 0; a2 < M; ++a2) {
                pair_t acc = out[a2];
                if (!signs_first) {
                    const uint32_t sw = sgn[(a2 * B + j) / 2];   // elements j, j + 1 (j even)
                    acc ^= ((pair_t)(sw & 0x80000000u) << 32) | (pair_t)(sw << 16);
                }
                amax = fmaxf(amax, fmaxf(fabsf(lo2(acc)), fabsf(hi2(acc))));
                *reinterpret_cast<pair_t *>(row + a2 * B + j) = acc;
            }
        }
        // row absmax over the CTA
#pragma unroll
        for (int k = 0; k < 5; ++k) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1 << k));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < kKWarps; ++w) amax = fmaxf(amax, red[w]);

        // per-group codes: the max of each 128 consecutive elements of the rotated
        // row (complete in the row buffer after the barrier above), a warp per group
        if (per_group) {
            for (int g = warp; g < N / 128; g += kKWarps) {
                const float4 v4 = reinterpret_cast<const float4 *>(row + g * 128)[lane];
                float gm = fmaxf(fmaxf(fabsf(v4.x), fabsf(v4.y)), fmaxf(fabsf(v4.z), fabsf(v4.w)));
#pragma unroll
                for (int k = 0; k < 5; ++k) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 1 << k));
                if (lane == 0) {
                    ginv[g] = gm > 0.f ? 7.0f / gm : 0.f;
                    p.scales[r * (int64_t)(N / 128) + g] = (gm / 7.0f) * p.inv_sqrt_n;
                }
            }
            __syncthreads();
        }

        // ---- quantize, pack, store (the same column pairs) ----
        // INT4 per row (default), INT8 per row, or INT4 per group of 128
        const float qmax = (p.flags & RQ_INT8_CODES) ? 127.0f : 7.0f;   // INT8, or INT4 (also in bytes)
        const float inv = amax > 0.f ? qmax / amax : 0.f;
        const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
        if (!per_group && threadIdx.x == 0) p.scales[r] = (amax / qmax) * p.inv_sqrt_n;
        uint8_t *qrow = p.q + r * (int64_t)(i8 ? N : N / 2);
        float *yrow = p.y ? p.y + r * (int64_t)N : nullptr;
        // one loop per code mode, so the default path carries no per-pair mode tests
        auto quantize = [&](auto i8_tag, auto grp_tag) {
            constexpr bool I8 = decltype(i8_tag)::value, GRP = decltype(grp_tag)::value;
            for (int j = 2 * threadIdx.x; j < B; j += 2 * kKThreads) {
#pragma unroll
                for (int a2 = 0; a2 < M; ++a2) {
                    const int e = a2 * B + j;                       // e, e + 1: one group (e even)
                    const pair_t v2 = *reinterpret_cast<const pair_t *>(row + e);
                    const float ie = GRP ? ginv[e >> 7] : inv;
                    const pair_t qq = fma2(v2, mk2(ie, ie), bias2);
                    if constexpr (I8) {
                        // the low byte of the biased float is the two's-complement code
                        const uint32_t c0 = (uint32_t)qq & 0xffu, c1 = (uint32_t)(qq >> 32) & 0xffu;
                        *reinterpret_cast<uint16_t *>(qrow + e) = (uint16_t)(c0 | (c1 << 8));
                    } else {
                        const uint32_t c0 = (uint32_t)qq & 0xfu, c1 = (uint32_t)(qq >> 32) & 0xfu;
                        qrow[e / 2] = (uint8_t)(c0 | (c1 << 4));
                    }
                    if (yrow)
                        *reinterpret_cast<pair_t *>(yrow + e) = fma2(v2, mk2(p.inv_sqrt_n, p.inv_sqrt_n), 0ull);
                }
            }
        };
        if (i8) quantize(std::true_type{}, std::false_type{});
        else if (per_group) quantize(std::false_type{}, std::true_type{});
        else quantize(std::false_type{}, std::false_type{});
        __syncthreads();   // the row buffer is rewritten by the next row
    }
}

template <int IN, int M, int LOGB>
cudaError_t launch_kron_t(const KronParams &p, cudaStream_t stream) {
    constexpr int N = M << LOGB;
    auto kern = fwht_kron_kernel<IN, M, LOGB>;
    const size_t smem = (size_t)N * 4 + (size_t)(N / 2) * 4 + kKWarps * 4 + (size_t)(N / 128) * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // as many resident CTAs as registers and shared memory allow: a CTA idles at
    // each of its four per-row barriers, another CTA on the SM fills the gap
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kKThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t slots = (int64_t)sms * per_sm;
    const int64_t grid = p.rows < slots ? p.rows : slots;
    kern<<<(unsigned)grid, kKThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int IN, int M>
cudaError_t launch_kron_m(const KronParams &p, int logb, cudaStream_t stream) {
    switch (logb) {
        case 5: return launch_kron_t<IN, M, 5>(p, stream);
        case 6: return launch_kron_t<IN, M, 6>(p, stream);
        case 7: return launch_kron_t<IN, M, 7>(p, stream);
        case 8: return launch_kron_t<IN, M, 8>(p, stream);
        case 9: return launch_kron_t<IN, M, 9>(p, stream);
        case 10: return launch_kron_t<IN, M, 10>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int IN>
cudaError_t launch_kron_in(const KronParams &p, int m, int logb, cudaStream_t stream) {
    switch (m) {
        case 12: return launch_kron_m<IN, 12>(p, logb, stream);
        case 20: return launch_kron_m<IN, 20>(p, logb, stream);
        case 28: return launch_kron_m<IN, 28>(p, logb, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool kron_block_of(int64_t n, int *m, int *logb) {
    const int ms[3] = {12, 20, 28};
    for (int i = 0; i < 3; ++i) {
        if (n % ms[i] != 0) continue;
        const int64_t b = n / ms[i];
        if (b < 32 || b > 1024 || (b & (b - 1)) != 0) continue;
        int lb = 0;
        while ((int64_t(1) << lb) < b) ++lb;
        *m = ms[i];
        *logb = lb;
        return true;
    }
    return false;
}

cudaError_t launch_fwht_kron(const RotJob &job, int m, int logb, int in_type, uint64_t seed, uint32_t flags,
                             cudaStream_t stream) {
    if (job.rows == 0) return cudaSuccess;
    const double n = (double)(m << logb);
    const KronParams p{job.x, job.ld, job.rows, job.q, job.scales, job.y, seed, flags, (float)(1.0 / sqrt(n))};
    switch (in_type) {
        case IN_F32: return launch_kron_in<IN_F32>(p, m, logb, stream);
        case IN_BF16: return launch_kron_in<IN_BF16>(p, m, logb, stream);
        case IN_F16: return launch_kron_in<IN_F16>(p, m, logb, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rq
