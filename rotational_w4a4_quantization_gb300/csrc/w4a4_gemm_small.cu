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
//    eight warps split K and meet in shared memory at the end (no global
//    workspace);
//  * each thread issues 16-byte loads: for one channel row, four lanes read 64
//    contiguous bytes (128 codes) per step.  A warp issues the loads of W and of
//    the activations for a group of steps (all of its steps for K = 4096 and up
//    to 16 tokens) before any MMA, so that the whole weight slice of the CTA is
//    in flight at once: the kernel is bound by reading W, and what limits that
//    is the number of bytes in flight, not the arithmetic;
//  * the MMA is the FP8 one (mma.sync m16n8k32 e4m3, fp32 accumulation): on
//    this part a legacy e4m3 MMA whose operand registers were just written costs
//    ~5.5 cycles per SM (cached operands: ~1.2), the int8 one 16 or more.
//    A code q becomes the E4M3 byte u = q + 8 (the nibble with its top bit
//    flipped; bytes 0x00..0x0F are exactly u * 2^-9), so the accumulator holds
//    sum u_a u_w * 2^-18 exactly, and sum q_a q_w = sum u_a u_w - 8 sum u_a -
//    8 sum u_w + 64 K with the u sums kept per row and per column alongside;
//  * the order of k inside each 128-code step is the same permutation for A
//    and W (a dot product does not depend on the order of its terms).
#include "rq_internal.h"

#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kWarps = 8;
constexpr int kThreadsS = 32 * kWarps;
constexpr int kChan = 16;     // output channels per CTA (two n8 MMA tiles)
constexpr int kMBlk = 64;     // tokens per CTA (four m16 MMA tiles)
// 128-code steps whose loads a warp issues together (registers: 8 per step for W
// plus 8 per m16 tile for the activations)
__host__ __device__ constexpr int unroll_for(int mt) { return mt == 1 ? 4 : (mt == 2 ? 2 : 1); }

__device__ __forceinline__ void mma_e4m3(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// E4M3 bytes u = q + 8 of the even (ulo) and odd (uhi) codes of a packed word
__device__ __forceinline__ uint32_t ulo(uint32_t w) { return (w ^ 0x88888888u) & 0x0f0f0f0fu; }
__device__ __forceinline__ uint32_t uhi(uint32_t w) { return ((w >> 4) ^ 0x08080808u) & 0x0f0f0f0fu; }
// sum of the u of both halves of a word (bytes <= 30, no carries)
__device__ __forceinline__ int usum(uint32_t lo, uint32_t hi, int acc) { return __dp4a((int)(lo + hi), 0x01010101, acc); }

template <int MT>  // number of m16 tiles handled (1..4)
__global__ void __launch_bounds__(kThreadsS)
w4a4_small_kernel(const uint8_t *__restrict__ aq, const float *__restrict__ sa,
                  const uint8_t *__restrict__ wq, const float *__restrict__ sw,
                  int64_t M, int64_t N, int64_t K, void *__restrict__ y, int y_mode) {
    __shared__ int part[kWarps][kMBlk][kChan + 1];
    __shared__ int rsum[kWarps][kMBlk], csum[kWarps][kChan];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int64_t c0 = (int64_t)blockIdx.x * kChan;
    const int64_t m0 = (int64_t)blockIdx.y * kMBlk;
    const int64_t kb = K / 2;                       // bytes per row
    const int64_t steps = K / 128;                  // 128-code steps (64 bytes per row)
    const int64_t s_begin = steps * warp / kWarps, s_end = steps * (warp + 1) / kWarps;

    // acc holds sum u_a u_w * 2^-18 exactly (every partial sum is a multiple of
    // 2^-18 below 2^6); sa_ / sw_ are this thread's sums of u over its k
    float acc[MT][2][4];
    int sa_[MT][2], sw_[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            sa_[i][j] = 0;
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;
        }

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

    constexpr int U = unroll_for(MT);
    for (int64_t s = s_begin; s < s_end; s += U) {
        uint4 wv[U][2], avu[U][MT][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool valid = s + u < s_end;
#pragma unroll
            for (int j = 0; j < 2; ++j)
                wv[u][j] = valid ? __ldg(reinterpret_cast<const uint4 *>(wrow[j] + (s + u) * 64)) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    avu[u][i][h] = valid ? __ldg(reinterpret_cast<const uint4 *>(arow[i][h] + (s + u) * 64))
                                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s + u >= s_end) break;
            const uint4 (&av)[MT][2] = avu[u];
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // four k32 MMA steps per 128 codes
                uint32_t b[2][2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t w = (&wv[u][j].x)[q];
                    b[j][0] = ulo(w);
                    b[j][1] = uhi(w);
                    sw_[j] = usum(b[j][0], b[j][1], sw_[j]);
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    const uint32_t x0 = (&av[i][0].x)[q], x1 = (&av[i][1].x)[q];
                    const uint32_t a[4] = {ulo(x0), ulo(x1), uhi(x0), uhi(x1)};
                    sa_[i][0] = usum(a[0], a[2], sa_[i][0]);
                    sa_[i][1] = usum(a[1], a[3], sa_[i][1]);
#pragma unroll
                    for (int j = 0; j < 2; ++j) mma_e4m3(acc[i][j], a, b[j]);
                }
            }
        }
    }

    // split-K reduction across the warps through shared memory: the partial
    // sums of u_a u_w as exact integers (x 2^18), and each row's / column's sum
    // of u (the four lanes sharing a row or column hold its four 16-byte chunks)
    auto to_int = [](float v) { return __float2int_rn(v * 262144.0f); };
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            part[warp][i * 16 + g][j * 8 + tq * 2] = to_int(acc[i][j][0]);
            part[warp][i * 16 + g][j * 8 + tq * 2 + 1] = to_int(acc[i][j][1]);
            part[warp][i * 16 + g + 8][j * 8 + tq * 2] = to_int(acc[i][j][2]);
            part[warp][i * 16 + g + 8][j * 8 + tq * 2 + 1] = to_int(acc[i][j][3]);
        }
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int v = sa_[i][h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (tq == 0) rsum[warp][i * 16 + h * 8 + g] = v;
        }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        int v = sw_[j];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (tq == 0) csum[warp][j * 8 + g] = v;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < MT * 16 * kChan; e += kThreadsS) {
        const int mm = e / kChan, cc = e % kChan;
        const int64_t m = m0 + mm, c = c0 + cc;
        if (m >= M || c >= N) continue;
        // sum q_a q_w = sum u_a u_w - 8 sum u_a - 8 sum u_w + 64 K
        int s = 0, su = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            s += part[w][mm][cc];
            su += rsum[w][mm] + csum[w][cc];
        }
        const int a = s - 8 * su + 64 * (int)K;
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
