// w4a4_gemm_tc.cu -- W4A4 GEMM on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// acc[m][c] = sum_k qa[m][k] * qw[c][k] (exact), y = acc * sa[m] * sw[c]: the
// product Q(XR)·Q(R^T W) of "Rotational Quantization ..." §The Principle of
// Computational Invariance / §Learned Orthogonal Rotations, run on tensor cores
// as §Hardware Execution and Serving Economics, 1. describes.
//
// The tcgen05 ISA of sm_103a has no integer MMA kind, so the 4-bit codes are
// widened to FP8 (E4M3) and multiplied with kind::f8f6f4:
//  * a code q in [-8, 7] becomes the byte u = q + 8 (its nibble with the top bit
//    flipped).  Bytes 0x00..0x0F of E4M3 are the 8 subnormals and the first
//    normal binade, i.e. exactly u * 2^-9: a linear, exact encoding;
//  * products are (u_a u_w) 2^-18 and every partial sum is a multiple of 2^-18
//    below 2^24 * 2^-18 (K <= 65536), so the fp32 accumulator in tensor memory
//    holds sum u_a u_w exactly;
//  * sum q_a q_w = sum u_a u_w - 8 sum u_a - 8 sum u_w + 64 K: the converter
//    warps add up each row's u while widening, and the epilogue removes the
//    offset, then applies the per-token x per-channel scales.
//
// Pipeline (persistent: one CTA per SM walks 128 x 256 output tiles; K in
// blocks of 128 codes; two TMEM accumulators so tile i's epilogue overlaps
// tile i+1's MMAs):
//   warp 0    TMA producer: packed A (128 x 64 B) and W (256 x 64 B) tiles into a
//             3-stage ring (mbarrier transaction counts);
//   warp 1    allocates 512 TMEM columns; one lane issues 4 MMAs (M128 N256 K32)
//             per K block into the tile's accumulator and commits them to the
//             operand ring's "empty" barriers and, per tile, to "acc full";
//   warps 2-9 widen nibbles to E4M3 into a 3-stage operand ring laid out in the
//             128-byte-swizzled K-major form the MMA descriptors expect, keep
//             per-row code sums, and hand each tile's offset terms and weight
//             scales to the epilogue through shared memory;
//   warps 10-17 epilogue: tcgen05.ld of the fp32 accumulator, offset removal,
//             scales (broadcast from shared memory), 16-byte stores.
// The order of k inside each 8-code group is permuted the same way for A and W
// (even codes, then odd codes), which leaves every dot product unchanged.
// Every mbarrier wait is bounded: on expiry the CTA raises the library's error
// word, stops, releases its tensor memory and returns.
#include "rq_internal.h"

#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>

namespace rq {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;      // tile (K in codes)
#ifndef RQ_TC_OP_STAGES
#define RQ_TC_OP_STAGES 3
#endif
constexpr int PK_STAGES = 3, OP_STAGES = RQ_TC_OP_STAGES;
constexpr int kConvWarps = 8;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreadsTC = 32 * (2 + kConvWarps + kEpiWarps);
constexpr int PK_A = BM * BK / 2, PK_W = BN * BK / 2;   // packed bytes per stage
constexpr int OP_A = BM * BK, OP_W = BN * BK;           // e4m3 bytes per stage
constexpr uint32_t kTmemCols = 512;                 // two 128x256 fp32 accumulators
constexpr long long kWaitLimitCycles = 4000000000ll;    // ~2 s at 2 GHz

struct Smem {
    alignas(1024) uint8_t opA[OP_STAGES][OP_A];
    alignas(1024) uint8_t opW[OP_STAGES][OP_W];
    alignas(128) uint8_t pkA[PK_STAGES][PK_A];
    alignas(128) uint8_t pkW[PK_STAGES][PK_W];
    int rowterm[2][BM];      // -8 * sum_k u_a, per tile parity
    int colterm[2][BN];      // 64 K - 8 * sum_k u_w
    float wscale[2][BN];     // weight scales of the tile's columns
    alignas(8) uint64_t pk_full[PK_STAGES];
    uint64_t pk_empty[PK_STAGES];
    uint64_t op_full[OP_STAGES];
    uint64_t op_empty[OP_STAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t sum_full[2], sum_empty[2];
    uint32_t tmem_base;
    volatile int abort_flag;
};

struct TcParams {
    const float *sa, *sw;
    void *y;
    int64_t M, N, K;
    int *err;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false (and raises the abort flag and the error word) if
// the phase does not complete in time or another role has aborted.
__device__ __forceinline__ bool mbar_wait(Smem &s, uint64_t *b, uint32_t parity, int *err) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(b, parity)) return true;
        if (s.abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            s.abort_flag = 1;
            atomicExch(err, 1);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);            // start address
    d |= (uint64_t)1 << 16;                             // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                   // stride byte offset
    d |= (uint64_t)1 << 46;                             // descriptor version
    d |= (uint64_t)2 << 61;                             // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, both K-major.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Widen one packed word (8 codes) to 8 E4M3 bytes u = q + 8: even codes in `lo`,
// odd codes in `hi`; returns the byte-lane sums for the row total.
__device__ __forceinline__ uint32_t widen(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x88888888u;
    lo = x & 0x0f0f0f0fu;
    hi = (x >> 4) & 0x0f0f0f0fu;
    return lo + hi;   // four bytes, each <= 30
}

template <int YMODE>
__global__ void __launch_bounds__(kThreadsTC, 1)
w4a4_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ TcParams prm) {
    extern __shared__ uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = (int)(prm.K / BK);
    const int64_t n_tiles_n = (prm.N + BN - 1) / BN;
    const int64_t n_tiles = n_tiles_n * ((prm.M + BM - 1) / BM);

    if (threadIdx.x == 0) {
        for (int i = 0; i < PK_STAGES; ++i) {
            mbar_init(&s.pk_full[i], 1);
            mbar_init(&s.pk_empty[i], kConvThreads);
        }
        for (int i = 0; i < OP_STAGES; ++i) {
            mbar_init(&s.op_full[i], kConvThreads);
            mbar_init(&s.op_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], kEpiThreads);
            mbar_init(&s.sum_full[i], kConvThreads);
            mbar_init(&s.sum_empty[i], kEpiThreads);
        }
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int64_t g = 0;                                   // global K-block counter
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const int m0 = (int)(tile / n_tiles_n) * BM, n0 = (int)(tile % n_tiles_n) * BN;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int st = (int)(g % PK_STAGES);
                    if (!mbar_wait(s, &s.pk_empty[st], (uint32_t)((g / PK_STAGES) & 1) ^ 1, prm.err)) { ok = false; break; }
                    mbar_expect_tx(&s.pk_full[st], PK_A + PK_W);
                    tma_load_2d(s.pkA[st], &tmA, &s.pk_full[st], kb * (BK / 2), m0);
                    tma_load_2d(s.pkW[st], &tmW, &s.pk_full[st], kb * (BK / 2), n0);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int64_t g = 0;
            int it = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
                const int buf = it & 1;
                // the epilogue must have drained this accumulator (two tiles ago)
                if (!mbar_wait(s, &s.acc_empty[buf], (uint32_t)((it >> 1) & 1) ^ 1, prm.err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int st = (int)(g % OP_STAGES);
                    if (!mbar_wait(s, &s.op_full[st], (uint32_t)((g / OP_STAGES) & 1), prm.err)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = smem_u32(s.opA[st]), w0 = smem_u32(s.opW[st]);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_f8(d, sw128_desc(a0 + 32 * k), sw128_desc(w0 + 32 * k), (kb | k) != 0);
                    mma_commit(&s.op_empty[st]);
                }
                if (ok) mma_commit(&s.acc_full[buf]);
            }
        }
    } else if (warp < 2 + kConvWarps) {
        // ---------------- converters ----------------
        const int t = threadIdx.x - 64;          // 0..255
        const int ch = t & 3;                    // 16-byte chunk of the 64-byte packed row
        const int rq = t >> 2;                   // 0..63
        int64_t g = 0;
        int it = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
            const int n0 = (int)(tile % n_tiles_n) * BN;
            uint32_t sumA[2] = {0, 0}, sumW[4] = {0, 0, 0, 0};
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                const int ps = (int)(g % PK_STAGES);
                if (!mbar_wait(s, &s.pk_full[ps], (uint32_t)((g / PK_STAGES) & 1), prm.err)) { ok = false; break; }
                uint4 a[2], w[4];
#pragma unroll
                for (int j = 0; j < 2; ++j) a[j] = reinterpret_cast<const uint4 *>(s.pkA[ps])[t + 256 * j];
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = reinterpret_cast<const uint4 *>(s.pkW[ps])[t + 256 * j];
                // The next TMA refill of this stage writes through the async proxy:
                // order this thread's generic reads of the stage before it, or the
                // refill can overtake them.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&s.pk_empty[ps]);

                const int os = (int)(g % OP_STAGES);
                if (!mbar_wait(s, &s.op_empty[os], (uint32_t)((g / OP_STAGES) & 1) ^ 1, prm.err)) { ok = false; break; }
                // row r, chunk ch -> 32 e4m3 bytes = granules 2ch, 2ch+1 of the 128-byte row
                auto emit = [&](uint8_t *base, int r, const uint4 &v, uint32_t &sum) {
                    uint32_t lo[4], hi[4], acc = 0;
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc += widen(wv[i], lo[i], hi[i]);
                    sum = __dp4a(acc, 0x01010101u, sum);
                    uint8_t *row = base + r * 128;
                    const int g0 = (2 * ch) ^ (r & 7), g1 = (2 * ch + 1) ^ (r & 7);
                    *reinterpret_cast<uint4 *>(row + 16 * g0) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
                    *reinterpret_cast<uint4 *>(row + 16 * g1) = make_uint4(lo[2], hi[2], lo[3], hi[3]);
                };
#pragma unroll
                for (int j = 0; j < 2; ++j) emit(s.opA[os], rq + 64 * j, a[j], sumA[j]);
#pragma unroll
                for (int j = 0; j < 4; ++j) emit(s.opW[os], rq + 64 * j, w[j], sumW[j]);
                // every writer makes its own stores visible to the tensor core's
                // (async-proxy) reads, then arrives itself
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(&s.op_full[os]);
            }
            if (!ok) break;
            // row sums: the four lanes sharing a row hold its four chunks
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                sumA[j] += __shfl_xor_sync(0xffffffffu, sumA[j], 1);
                sumA[j] += __shfl_xor_sync(0xffffffffu, sumA[j], 2);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sumW[j] += __shfl_xor_sync(0xffffffffu, sumW[j], 1);
                sumW[j] += __shfl_xor_sync(0xffffffffu, sumW[j], 2);
            }
            // hand this tile's offset terms and weight scales to the epilogue
            const int buf = it & 1;
            if (!mbar_wait(s, &s.sum_empty[buf], (uint32_t)((it >> 1) & 1) ^ 1, prm.err)) { ok = false; break; }
            if (ch == 0) {
                for (int j = 0; j < 2; ++j) s.rowterm[buf][rq + 64 * j] = -8 * (int)sumA[j];
                for (int j = 0; j < 4; ++j) s.colterm[buf][rq + 64 * j] = 64 * (int)prm.K - 8 * (int)sumW[j];
            }
            if (YMODE != 2) s.wscale[buf][t] = (n0 + t < prm.N) ? prm.sw[n0 + t] : 0.f;
            mbar_arrive(&s.sum_full[buf]);
        }
    } else {
        // ---------------- epilogue: TMEM -> offset removal -> scales -> global ----------------
        const int e = threadIdx.x - 64 - kConvThreads;   // 0..255
        const int q = warp & 3;                          // TMEM lane quarter this warp may read
        const int colhalf = e >> 7;                      // columns 0-127 or 128-255
        int it = 0;
        for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t par = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait(s, &s.acc_full[buf], par, prm.err)) break;
            if (!mbar_wait(s, &s.sum_full[buf], par, prm.err)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int64_t m0 = (tile / n_tiles_n) * BM, n0 = (tile % n_tiles_n) * BN;
            const int mr = 32 * q + lane;
            const int64_t m = m0 + mr;
            const int rowt = s.rowterm[buf][mr];
            const float sa = (YMODE != 2 && m < prm.M) ? prm.sa[m] : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                const int col0 = colhalf * 128 + 32 * c;
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * BN + col0), r);
                if (m < prm.M) {
                    int acc[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int u = __float2int_rn(__uint_as_float(r[j]) * 262144.0f);   // exact: x 2^18
                        acc[j] = u + rowt + s.colterm[buf][col0 + j];
                    }
                    const int64_t nb = n0 + col0;
                    if (YMODE == 2) {
                        int *yr = static_cast<int *>(prm.y) + m * prm.N + nb;
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            if (nb + j + 3 < prm.N)
                                *reinterpret_cast<int4 *>(yr + j) = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                    } else if (YMODE == 1) {
                        float *yr = static_cast<float *>(prm.y) + m * prm.N + nb;
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            if (nb + j + 3 >= prm.N) continue;
                            float4 o;
                            o.x = ((float)acc[j] * sa) * s.wscale[buf][col0 + j];
                            o.y = ((float)acc[j + 1] * sa) * s.wscale[buf][col0 + j + 1];
                            o.z = ((float)acc[j + 2] * sa) * s.wscale[buf][col0 + j + 2];
                            o.w = ((float)acc[j + 3] * sa) * s.wscale[buf][col0 + j + 3];
                            *reinterpret_cast<float4 *>(yr + j) = o;
                        }
                    } else {
                        __half *yr = static_cast<__half *>(prm.y) + m * prm.N + nb;
#pragma unroll
                        for (int j = 0; j < 32; j += 8) {
                            if (nb + j + 7 >= prm.N) continue;
                            __align__(16) __half h[8];
#pragma unroll
                            for (int e2 = 0; e2 < 8; ++e2)
                                h[e2] = __float2half_rn(((float)acc[j + e2] * sa) * s.wscale[buf][col0 + j + e2]);
                            *reinterpret_cast<uint4 *>(yr + j) = *reinterpret_cast<const uint4 *>(h);
                        }
                    }
                }
            }
            // this accumulator and these offset terms may be reused
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&s.acc_empty[buf]);
            mbar_arrive(&s.sum_empty[buf]);
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {BK / 2, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int YMODE>
cudaError_t launch_mode(const CUtensorMap &ta, const CUtensorMap &tw, const TcParams &p, cudaStream_t stream) {
    auto kern = w4a4_tc_kernel<YMODE>;
    const size_t smem = sizeof(Smem) + 1024;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = ((p.N + BN - 1) / BN) * ((p.M + BM - 1) / BM);
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);   // persistent: one CTA per SM
    kern<<<grid, kThreadsTC, smem, stream>>>(ta, tw, p);
    return cudaGetLastError();
}

}  // namespace

bool w4a4_gemm_tc_supported(const GemmArgs &g) { return g.M > 64 && g.K % BK == 0 && g.K <= 65536; }

cudaError_t launch_w4a4_gemm_tc(const GemmArgs &g, cudaStream_t stream) {
    CUtensorMap ta, tw;
    if (!make_map(&ta, g.a_q, g.M, g.K / 2, BM) || !make_map(&tw, g.w_q, g.N, g.K / 2, BN))
        return cudaErrorInvalidValue;
    TcParams p{g.a_scales, g.w_scales, g.y, g.M, g.N, g.K, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    switch (g.y_mode) {
        case 0: return launch_mode<0>(ta, tw, p, stream);
        case 1: return launch_mode<1>(ta, tw, p, stream);
        default: return launch_mode<2>(ta, tw, p, stream);
    }
}

}  // namespace rq
