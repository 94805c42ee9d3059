// w4a4_gemm_small.cu -- W4A4 GEMM for few tokens (decode-shaped M), sm_103a.
//
// acc[m][c] = sum_k qa[m][k] * qw[c][k] exactly in int32, then
// y = acc * sa[m] * sw[c]: the integer product Q(XR)·Q(R^T W) of "Rotational
// Quantization ..." §The Principle of Computational Invariance / §Learned
// Orthogonal Rotations, with the per-token x per-channel dequant.
//
// With a handful of tokens the layer is bound by reading the packed weights
// from HBM (K*N/2 bytes), so this kernel is built around streaming W once:
//  * a CTA owns 16 output channels and one block of up to 64 tokens; its four
//    warps split K four ways and meet in shared memory at the end (no global
//    workspace);
//  * each thread issues 16-byte loads: for one channel row, four lanes read 64
//    contiguous bytes (128 codes) per step;
//  * nibbles widen to int8 with one shift and one mask per 4 codes: the byte
//    (w << 4) & 0xF0 holds 16*q of the even code and w & 0xF0 holds 16*q of
//    the odd one, so the int8 MMA (mma.sync m16n8k32 s8, exact int32
//    accumulation) produces 256*acc, undone by an exact arithmetic shift;
//  * the order of k inside each 128-code step is the same permutation for A
//    and W (a dot product does not depend on the order of its terms).
#include "rq_internal.h"

#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreadsS = 32 * kWarps;
constexpr int kChan = 16;     // output channels per CTA (two n8 MMA tiles)
constexpr int kMBlk = 64;     // tokens per CTA (four m16 MMA tiles)
constexpr int kUnroll = 4;    // 128-code steps in flight per warp

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t lo16(uint32_t w) { return (w << 4) & 0xf0f0f0f0u; }
__device__ __forceinline__ uint32_t hi16(uint32_t w) { return w & 0xf0f0f0f0u; }

template <int MT>  // number of m16 tiles handled (1..4)
__global__ void __launch_bounds__(kThreadsS)
w4a4_small_kernel(const uint8_t *__restrict__ aq, const float *__restrict__ sa,
                  const uint8_t *__restrict__ wq, const float *__restrict__ sw,
                  int64_t M, int64_t N, int64_t K, void *__restrict__ y, int y_mode) {
    __shared__ int part[kWarps][kMBlk][kChan + 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int64_t c0 = (int64_t)blockIdx.x * kChan;
    const int64_t m0 = (int64_t)blockIdx.y * kMBlk;
    const int64_t kb = K / 2;                       // bytes per row
    const int64_t steps = K / 128;                  // 128-code steps (64 bytes per row)
    const int64_t s_begin = steps * warp / kWarps, s_end = steps * (warp + 1) / kWarps;

    int acc[MT][2][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][j][r] = 0;

    // row pointers (clamped: rows past M / N read row 0 and are never stored)
    const uint8_t *wrow[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t c = c0 + j * 8 + g;
        wrow[j] = wq + (c < N ? c : 0) * kb + tq * 16;
    }
    const uint8_t *arow[MT][2];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t m = m0 + i * 16 + h * 8 + g;
            arow[i][h] = aq + (m < M ? m : 0) * kb + tq * 16;
        }

    for (int64_t s = s_begin; s < s_end; s += kUnroll) {
        uint4 wv[kUnroll][2];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                wv[u][j] = (s + u < s_end) ? __ldg(reinterpret_cast<const uint4 *>(wrow[j] + (s + u) * 64))
                                           : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (s + u >= s_end) break;
            uint4 av[MT][2];
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    av[i][h] = __ldg(reinterpret_cast<const uint4 *>(arow[i][h] + (s + u) * 64));
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // four k32 MMA steps per 128 codes
                uint32_t b[2][2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t w = (&wv[u][j].x)[q];
                    b[j][0] = lo16(w);
                    b[j][1] = hi16(w);
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const uint32_t x0 = (&av[i][0].x)[q], x1 = (&av[i][1].x)[q];
                    const uint32_t a[4] = {lo16(x0), lo16(x1), hi16(x0), hi16(x1)};
#pragma unroll
                    for (int j = 0; j < 2; ++j) mma_s8(acc[i][j], a, b[j]);
                }
            }
        }
    }

    // split-K reduction across the warps through shared memory
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            part[warp][i * 16 + g][j * 8 + tq * 2] = acc[i][j][0];
            part[warp][i * 16 + g][j * 8 + tq * 2 + 1] = acc[i][j][1];
            part[warp][i * 16 + g + 8][j * 8 + tq * 2] = acc[i][j][2];
            part[warp][i * 16 + g + 8][j * 8 + tq * 2 + 1] = acc[i][j][3];
        }
    __syncthreads();
    for (int e = threadIdx.x; e < MT * 16 * kChan; e += kThreadsS) {
        const int mm = e / kChan, cc = e % kChan;
        const int64_t m = m0 + mm, c = c0 + cc;
        if (m >= M || c >= N) continue;
        int s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += part[w][mm][cc];
        const int a = s >> 8;   // exact: every product carried a factor 16*16
        if (y_mode == 2) {
            static_cast<int *>(y)[m * N + c] = a;
        } else {
            const float v = ((float)a * sa[m]) * sw[c];
            if (y_mode == 1) static_cast<float *>(y)[m * N + c] = v;
            else static_cast<__half *>(y)[m * N + c] = __float2half_rn(v);
        }
    }
}

}  // namespace

cudaError_t launch_w4a4_gemm_small(const GemmArgs &g, cudaStream_t stream) {
    const dim3 grid((unsigned)((g.N + kChan - 1) / kChan), (unsigned)((g.M + kMBlk - 1) / kMBlk));
    const int64_t mt = g.M >= kMBlk ? 4 : (g.M + 15) / 16;
    switch (mt) {
        case 1:
            w4a4_small_kernel<1><<<grid, kThreadsS, 0, stream>>>(g.a_q, g.a_scales, g.w_q, g.w_scales, g.M, g.N, g.K, g.y, g.y_mode);
            break;
        case 2:
            w4a4_small_kernel<2><<<grid, kThreadsS, 0, stream>>>(g.a_q, g.a_scales, g.w_q, g.w_scales, g.M, g.N, g.K, g.y, g.y_mode);
            break;
        case 3:
            w4a4_small_kernel<3><<<grid, kThreadsS, 0, stream>>>(g.a_q, g.a_scales, g.w_q, g.w_scales, g.M, g.N, g.K, g.y, g.y_mode);
            break;
        default:
            w4a4_small_kernel<4><<<grid, kThreadsS, 0, stream>>>(g.a_q, g.a_scales, g.w_q, g.w_scales, g.M, g.N, g.K, g.y, g.y_mode);
            break;
    }
    return cudaGetLastError();
}

}  // namespace rq
