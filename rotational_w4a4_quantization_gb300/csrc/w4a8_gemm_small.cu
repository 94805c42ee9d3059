// w4a8_gemm_small.cu -- W4A8 linear layer for few tokens, with per-channel or
// per-group weight scales (sm_103a).  Products of more than 64 tokens are
// dispatched to the tensor-core kernels of w4a4_gemm_tc.cu where their shapes
// allow (per channel: the A8 variant; per group: the group kernel).
//
// "SpinQuant" page, The architecture: the rotated weights go to INT4 and the
// activations to INT8, with per-channel or per-group scales; End-to-end flow:
// the rotated activation is quantized to INT8 and multiplied against the INT4
// rotated weights.  With groups of 128 along K and codes qa (int8), qw (int4):
//   acc_g[m][c] = sum_{k in group g} qa[m][k] qw[c][k]     (exact integers)
//   y[m][c]     = sa[m] * sum_g sw[c][g] acc_g[m][c]
// and with one scale per channel (group = K) the int32 sum itself is exact.
//
// Design (decode-shaped M, bound in principle by reading W once):
//  * a CTA owns 16 output channels and up to 32 tokens; eight warps split K in
//    128-code steps, each a whole group, and meet in shared memory at the end;
//  * the MMA is mma.sync m16n8k32 s8 x s8 -> s32: a weight nibble masked in place
//    is the int8 16 q (one or two logic ops per word: w & 0xF0, (w << 4) & 0xF0),
//    so the accumulator holds 16 sum qa qw exactly (|16 qa qw| <= 2^14, 2^17
//    per 128-code step), with no offset terms; the activation operand is two byte
//    permutes of 8 consecutive codes (even positions, then odd), the order in
//    which the nibble masks deliver the weight codes;
//  * per-group scales: after each step the lane's int32 partials (exact) are
//    scaled by their column's group scale and added in fp32; per-channel scales:
//    the int32 sums run to the end and are scaled once (or returned raw).
#include "rq_internal.h"

#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kW8Warps = 8;
constexpr int kW8Threads = 32 * kW8Warps;
constexpr int kW8Chan = 16;      // output channels per CTA (two n8 MMA tiles)
constexpr int kW8MBlk = 32;      // tokens per CTA (up to two m16 MMA tiles)

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int MT, bool GROUPED>
__global__ void __launch_bounds__(kW8Threads)
w4a8_small_kernel(const int8_t *__restrict__ aq, const float *__restrict__ sa, const uint8_t *__restrict__ wq,
                  const float *__restrict__ sw, int64_t M, int64_t N, int64_t K, void *__restrict__ y, int y_mode) {
    __shared__ float partf[GROUPED ? kW8Warps : 1][kW8MBlk][kW8Chan + 1];
    __shared__ int parti[GROUPED ? 1 : kW8Warps][kW8MBlk][kW8Chan + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int64_t c0 = (int64_t)blockIdx.x * kW8Chan;
    const int64_t m0 = (int64_t)blockIdx.y * kW8MBlk;
    const int64_t steps = K / 128;                  // 128-code steps = groups
    const int64_t s_begin = steps * warp / kW8Warps, s_end = steps * (warp + 1) / kW8Warps;

    int acc[MT][2][4];
    float fo[MT][2][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[i][j][r] = 0;
                fo[i][j][r] = 0.f;
            }

    // rows clamped: rows past M / N read row 0 and are never stored
    const uint8_t *wrow[2];
    const float *swrow[2][2];                       // group scales of this lane's columns 2 tq, 2 tq + 1
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t c = c0 + j * 8 + g;
        wrow[j] = wq + (c < N ? c : 0) * (K / 2) + tq * 16;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int64_t cc = c0 + j * 8 + 2 * tq + e;
            swrow[j][e] = sw + (cc < N ? cc : 0) * (GROUPED ? steps : 1);
        }
    }
    const int8_t *arow[MT][2];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t m = m0 + i * 16 + h * 8 + g;
            arow[i][h] = aq + (m < M ? m : 0) * K + tq * 32;
        }

    for (int64_t s = s_begin; s < s_end; ++s) {
        // this lane's share of the step: 32 weight codes of two channels (16 bytes
        // each) and 32 activation codes of each of its rows (32 bytes each)
        uint4 wv[2], av[MT][2][2];
#pragma unroll
        for (int j = 0; j < 2; ++j) wv[j] = __ldg(reinterpret_cast<const uint4 *>(wrow[j] + s * 64));
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    av[i][h][k] = __ldg(reinterpret_cast<const uint4 *>(arow[i][h] + s * 128 + 16 * k));
#pragma unroll
        for (int q = 0; q < 4; ++q) {   // four k32 MMA steps per 128 codes
            uint32_t b[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t w = (&wv[j].x)[q];
                b[j][0] = (w << 4) & 0xf0f0f0f0u;    // 16 x the even codes
                b[j][1] = w & 0xf0f0f0f0u;           // 16 x the odd codes
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                // codes 8q .. 8q + 7 of the lane's 32: words 2q, 2q + 1 of its chunk
                const uint32_t x00 = (&av[i][0][q >> 1].x)[2 * (q & 1)], x01 = (&av[i][0][q >> 1].x)[2 * (q & 1) + 1];
                const uint32_t x10 = (&av[i][1][q >> 1].x)[2 * (q & 1)], x11 = (&av[i][1][q >> 1].x)[2 * (q & 1) + 1];
                const uint32_t a[4] = {__byte_perm(x00, x01, 0x6420u), __byte_perm(x10, x11, 0x6420u),
                                       __byte_perm(x00, x01, 0x7531u), __byte_perm(x10, x11, 0x7531u)};
#pragma unroll
                for (int j = 0; j < 2; ++j) mma_s8(acc[i][j], a, b[j]);
            }
        }
        if constexpr (GROUPED) {
            // the step is one group: exact partials (16 x) scaled by the group scale
            float sg[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) sg[j][e] = __ldg(swrow[j][e] + s);
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        fo[i][j][r] += (float)(acc[i][j][r] >> 4) * sg[j][r & 1];
                        acc[i][j][r] = 0;
                    }
        }
    }

    // split-K reduction across the warps
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = i * 16 + g + 8 * (r >> 1), col = j * 8 + tq * 2 + (r & 1);
                if constexpr (GROUPED) partf[warp][row][col] = fo[i][j][r];
                else parti[warp][row][col] = acc[i][j][r] >> 4;   // exact: every product is a multiple of 16
            }
    __syncthreads();
    for (int e = threadIdx.x; e < MT * 16 * kW8Chan; e += kW8Threads) {
        const int mm = e / kW8Chan, cc = e % kW8Chan;
        const int64_t m = m0 + mm, c = c0 + cc;
        if (m >= M || c >= N) continue;
        float v;
        if constexpr (GROUPED) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kW8Warps; ++w) sum += partf[w][mm][cc];
            v = sum * sa[m];
        } else {
            int sum = 0;
#pragma unroll
            for (int w = 0; w < kW8Warps; ++w) sum += parti[w][mm][cc];
            if (y_mode == 2) {
                static_cast<int *>(y)[m * N + c] = sum;
                continue;
            }
            v = ((float)sum * sa[m]) * sw[c];
        }
        if (y_mode == 1) static_cast<float *>(y)[m * N + c] = v;
        else static_cast<__half *>(y)[m * N + c] = __float2half_rn(v);
    }
}

template <bool GROUPED>
cudaError_t launch_w8_g(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M, int64_t N,
                        int64_t K, void *y, int y_mode, cudaStream_t stream) {
    const dim3 grid((unsigned)((N + kW8Chan - 1) / kW8Chan), (unsigned)((M + kW8MBlk - 1) / kW8MBlk));
    if (M > 16) w4a8_small_kernel<2, GROUPED><<<grid, kW8Threads, 0, stream>>>(aq, sa, wq, sw, M, N, K, y, y_mode);
    else w4a8_small_kernel<1, GROUPED><<<grid, kW8Threads, 0, stream>>>(aq, sa, wq, sw, M, N, K, y, y_mode);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_w4a8_gemm(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                             int64_t N, int64_t K, int64_t group, void *y, int y_mode, cudaStream_t stream) {
    if (group == K && w4a8_gemm_tc_supported(M, N, K, y_mode))
        return launch_w4a8_gemm_tc(aq, sa, wq, sw, M, N, K, y, y_mode, stream);
    if (group == K) return launch_w8_g<false>(aq, sa, wq, sw, M, N, K, y, y_mode, stream);
    if (group == 128 && w4a8_group_tc_supported(M, N, K, y_mode))
        return launch_w4a8_group_tc(aq, sa, wq, sw, M, N, K, y, y_mode, stream);
    if (group == 128) return launch_w8_g<true>(aq, sa, wq, sw, M, N, K, y, y_mode, stream);
    return cudaErrorInvalidValue;
}

}  // namespace rq
