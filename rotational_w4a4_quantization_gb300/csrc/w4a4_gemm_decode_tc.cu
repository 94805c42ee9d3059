// w4a4_gemm_decode_tc.cu -- W4A4 product for decode batches on the 5th-generation
// tensor cores (tcgen05), sm_103a.
//
// acc[m][c] = sum_k qa[m][k] qw[c][k] exactly, y = acc sa[m] sw[c]: the product
// Q(XR)·Q(R^T W) of "Rotational Quantization ..." §The Principle of
// Computational Invariance / §Learned Orthogonal Rotations, on tensor cores as
// §Hardware Execution and Serving Economics, 1. describes, for a handful of
// tokens (M <= 64, N a multiple of 128, K a multiple of 128 up to 8192).
//
// With few tokens the layer is bound by reading the packed weights (K N / 2
// bytes) from HBM, so the kernel is built around streaming them once:
//  * the roles of the operands are swapped: a CTA's 128 output channels are the
//    MMA's M side (the TMEM lanes) and the tokens its N side (16, 32, 48 or
//    64), so one M128 N16 K32 MMA consumes 32 codes of 128 channels;
//  * the weights sit in tensor memory, the MMA's A operand: TMA brings the
//    CTA's packed slice (128 channels x KS codes, KS <= 1024) into shared memory
//    as K blocks of 128 codes, all requested at the start, each completing on
//    its own single-use mbarrier.  As a block lands, the threads of each TMEM
//    lane quarter widen their channel's 64 packed bytes and store them to
//    tensor memory (tcgen05.st, one column range per warp): no shared-memory
//    round trip for the widened weights, whose bytes would otherwise dominate
//    the shared-memory traffic;
//  * codes widen exactly: a weight code q becomes the E4M3 byte u = q + 8 (its
//    nibble with the top bit flipped; bytes 0x00..0x0F of E4M3 are exactly
//    u 2^-9), an activation code keeps its sign (sign bit plus |q| <= 8 as
//    |q| 2^-9).  Products are q_a u_w 2^-18 and every partial sum of a slice is
//    a multiple of 2^-18 below 2^0 (|q_a u_w| <= 120, KS <= 1024), exact in the
//    fp32 accumulator; sum q_a q_w = sum q_a u_w - 8 sum q_a, with the
//    activation code sums formed while widening them;
//  * K is split over the S CTAs of a thread-block cluster (S = 1, 2, 4 or 8,
//    chosen so that the grid fills the SMs once where it can).  Each CTA turns
//    its accumulators into exact integer partials in shared memory; after a
//    cluster barrier, CTA r adds the S partials of channels
//    [128 r / S, 128 (r + 1) / S) through distributed shared memory (integer
//    sums: the order does not matter) and applies the scales.  No global
//    workspace;
//  * within each group of 8 codes the order of k is permuted the same way for
//    the weights and the activations (even codes, then odd), which leaves every
//    dot product unchanged.
// Every mbarrier wait is bounded: on expiry the CTA raises the library's error
// word, skips the rest of its work and its stores, still meets both cluster
// barriers, waits (bounded) for copies still in flight and frees its tensor
// memory.
#include "rq_internal.h"
#include "rot_device.cuh"

#include <cuda_fp16.h>

#include <utility>

namespace rq {
namespace {

constexpr int DBK = 128;                 // codes per K block
constexpr int DCH = 128;                 // output channels per CTA (MMA M, TMEM lanes)
constexpr int DTHREADS = 256;            // eight warps: two per TMEM lane quarter
constexpr int DMAXB = 8;                 // K blocks per CTA: KS <= 1024 codes
constexpr int DMAXS = 8;                 // CTAs per cluster
constexpr uint32_t DTMEM_COLS = 512;     // weights: 32 columns per K block (<= 256); accumulators after
constexpr uint32_t DACC_COL = 256;
constexpr int DNACC = 4;                 // independent accumulators: K step j goes to accumulator j % 4
constexpr long long kDecodeWaitLimit = 4000000000ll;   // ~2 s at 2 GHz
constexpr size_t kOneCtaPerSmBytes = 116 * 1024;        // dynamic shared memory that keeps one CTA per SM

// Rotation buffer of the fused kernel: up to 16384 fp32 values (the CTA's rows
// of one n, padded to a power of two), stored XOR-swizzled (see rot_phys).
constexpr int kRotBufWords = 16384;

template <int MT, bool FUSED>   // token tiles of 16 (the MMA's N is 16 MT); fused rotation or codes from HBM
struct DSmem {
    alignas(1024) uint8_t pkw[DMAXB][DCH * DBK / 2];   // packed weight blocks (TMA), 8 KB each
    alignas(1024) uint8_t opb[DMAXB][16 * MT * DBK];   // activation operand: E4M3, 128-byte-swizzled K-major
    // exact partial products that the cluster's CTAs push here for this CTA's
    // share of the channels: [source CTA][token][channel - 128 rank / S]
    alignas(16) int recv[16 * MT * DCH];
    int aborts[DMAXS];                                  // abort flags the cluster's CTAs push here
    float wsc[DCH];                                     // weight scales of the channels this CTA stores
    float tsc[16 * MT];                                 // token scales (decode product: loaded at the start)
    int qsum[16 * MT];                                  // sum of each token's activation codes over the slice
    // fused only: the slice's packed activation codes and every token's scale, as
    // the CTAs of the cluster that rotate the tokens write them; the rotation
    // buffer, sign bits and row maxima
    alignas(16) uint8_t apk[FUSED ? 16 * MT : 1][FUSED ? DMAXB * DBK / 2 : 16];
    float asc[FUSED ? 16 * MT : 1];
    uint32_t sgn[FUSED ? 256 : 1];
    uint32_t rowmax[FUSED ? 16 : 1];
    alignas(16) float xs[FUSED ? kRotBufWords : 4];
    alignas(8) uint64_t wfull[DMAXB];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort_flag;
};

struct DParams {
    const uint8_t *aq;
    const float *sa, *sw;
    void *y;
    int64_t M, N, K;
    int y_mode;
    int *err;
};

__device__ __forceinline__ uint32_t d_smem(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void d_mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(d_smem(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void d_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(d_smem(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool d_try_wait(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(d_smem(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on phase `parity`; false (and the error word raised) on expiry.
__device__ __forceinline__ bool d_wait(uint64_t *b, uint32_t parity, int *err) {
    if (d_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!d_try_wait(b, parity)) {
        if (clock64() - t0 > kDecodeWaitLimit) {
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void d_tma_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(d_smem(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(d_smem(bar))
        : "memory");
}

// Shared-memory operand descriptor: K-major, 128-byte swizzle, 8-row groups 1024
// bytes apart.
__device__ __forceinline__ uint64_t d_sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f8f6f4, A = B = E4M3, D = F32, both K-major, M = 128, N = 16 MT.
template <int MT>
constexpr uint32_t d_idesc() {
    return (1u << 4) | ((uint32_t)((16 * MT) >> 3) << 17) | ((uint32_t)(DCH >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, K = 32 (A: 128 lanes x 8 columns of 4 codes).
template <int MT>
__device__ __forceinline__ void d_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(d_idesc<MT>()), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void d_tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// 16 columns of the warp's 32 lanes; completes at the next d_tmem_wait_ld.
__device__ __forceinline__ void d_tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void d_tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Split cluster barrier at the start: every CTA of the cluster has started (its
// shared memory exists) before any CTA writes into another's.
__device__ __forceinline__ void d_cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void d_cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ void d_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Offset form of one packed word (8 codes): u = q + 8 of the even codes in `lo`,
// of the odd codes in `hi`, one per byte lane.
__device__ __forceinline__ void d_widen_u(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t x = w ^ 0x88888888u;
    lo = x & 0x0f0f0f0fu;
    hi = (x >> 4) & 0x0f0f0f0fu;
}

// Byte lanes holding 4-bit two's-complement codes (0..15) -> E4M3 bytes of the
// same signed value times 2^-9: |q| <= 8 in bits 0..3, the sign in bit 7.
__device__ __forceinline__ uint32_t d_e4m3_signed(uint32_t x) {
    const uint32_t neg = (x >> 3) & 0x01010101u;
    return (x ^ (neg * 0x8fu)) + neg;
}

// ---------------------------------------------------------------------------
// Phases shared by the decode product and the fused rotation + product
// ---------------------------------------------------------------------------

// At entry, warp 0: lane 0 initializes the barriers, then lane b requests K
// block b of the weight slice (the layer is bound by this stream, so it starts
// before anything else).  A block is one box of 64 bytes x 128 channels with the
// 64-byte swizzle: chunk j of channel r lands at 16-byte position
// j ^ ((r >> 1) & 3) of the channel's 64 bytes, so the lanes reading chunk j of
// 32 consecutive channels hit distinct bank groups.
template <class S_>
__device__ __forceinline__ void d_start_weights(S_ &s, const CUtensorMap *tm, int lane, int b0, int nb, int64_t c0) {
    if (lane == 0) {
        for (int b = 0; b < DMAXB; ++b) d_mbar_init(&s.wfull[b], 1);
        d_mbar_init(&s.mma_done, 1);
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (lane < nb) {
        d_expect_tx(&s.wfull[lane], DCH * DBK / 2);
        d_tma_2d(s.pkw[lane], tm, &s.wfull[lane], (b0 + lane) * (DBK / 2), (int)c0);
    }
    __syncwarp();
}

// Tensor memory (512 columns), zeroed token sums; every thread then sees the
// barriers warp 0 initialized.
template <class S_>
__device__ __forceinline__ uint32_t d_setup(S_ &s, int tid, int warp, int mp) {
    if (tid < mp) s.qsum[tid] = 0;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(d_smem(&s.tmem_base)),
                     "r"(DTMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    d_cluster_arrive_relaxed();   // matched by d_cluster_wait before the first remote store
    return s.tmem_base;
}

// Activation codes of the slice -> signed E4M3 operand (tokens >= M stay zero
// codes) and each token's code sum.  d_load_acts issues every load of the
// thread (load(m, off) returns the 16 packed bytes at byte offset off of token
// m's slice: 32 codes = operand granules 2 ch, 2 ch + 1), d_store_acts widens
// and stores them once they have landed.
template <int MT>
struct ActChunks {
    static constexpr int MAXC = 16 * MT * DMAXB * 4 / DTHREADS;   // chunks per thread at most (1 .. 8)
    uint4 v[MAXC];
};

template <int MT, class Load>
__device__ __forceinline__ void d_load_acts(ActChunks<MT> &a, int tid, int nb, int M, Load load) {
    constexpr int MP = 16 * MT;
    const int per_row = nb * 4;
#pragma unroll
    for (int i = 0; i < ActChunks<MT>::MAXC; ++i) {
        const int e = tid + DTHREADS * i;
        const int m = e / per_row, rem = e - m * per_row;
        a.v[i] = (e < MP * per_row && m < M) ? load(m, (rem >> 2) * (DBK / 2) + 16 * (rem & 3))
                                              : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <int MT, class S_>
__device__ __forceinline__ void d_store_acts(S_ &s, const ActChunks<MT> &a, int tid, int nb, int M) {
    constexpr int MP = 16 * MT;
    const int per_row = nb * 4;
#pragma unroll
    for (int i = 0; i < ActChunks<MT>::MAXC; ++i) {
        const int e = tid + DTHREADS * i;
        if (e >= MP * per_row) break;
        const int m = e / per_row, rem = e - m * per_row, b = rem >> 2, ch = rem & 3;
        const uint4 v = a.v[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8], usum = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[2 * k] = d_e4m3_signed(wv[k] & 0x0f0f0f0fu);
            o[2 * k + 1] = d_e4m3_signed((wv[k] >> 4) & 0x0f0f0f0fu);
            uint32_t ul, uh;
            d_widen_u(wv[k], ul, uh);
            usum = __dp4a(ul + uh, 0x01010101u, usum);   // byte lanes <= 30
        }
        uint8_t *rowp = s.opb[b] + m * DBK;
        const int sw = m & 7;
        *reinterpret_cast<uint4 *>(rowp + 16 * ((2 * ch) ^ sw)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4 *>(rowp + 16 * ((2 * ch + 1) ^ sw)) = make_uint4(o[4], o[5], o[6], o[7]);
        if (m < M) atomicAdd(&s.qsum[m], (int)usum - 8 * 32);   // sum of q = sum of u - 8 per code
    }
    // the operand stores are read by the tensor core (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Weights: warp w widens the K blocks b = w / 4, w / 4 + 2, ... of the 32
// channels of TMEM lane quarter w % 4 (one channel per thread) as they land.
template <class S_>
__device__ __forceinline__ void d_widen_weights(S_ &s, uint32_t tmem, int nb, int warp, int lane, int *err) {
    const unsigned full = 0xffffffffu;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;                            // channel within the tile = TMEM lane
    const uint32_t tlane = tmem + ((uint32_t)(32 * q4) << 16);
    for (int b = warp >> 2; b < nb; b += 2) {
        const bool ok = __all_sync(full, d_wait(&s.wfull[b], 0, err));
        if (!ok) {
            if (lane == 0) s.abort_flag = 1;
            break;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // chunk j (codes 32 j .. 32 j + 31) of this thread's channel (64-byte swizzle)
            const uint4 v = *reinterpret_cast<const uint4 *>(s.pkw[b] + r * (DBK / 2) + 16 * (j ^ ((r >> 1) & 3)));
            uint32_t o[8];
            d_widen_u(v.x, o[0], o[1]);
            d_widen_u(v.y, o[2], o[3]);
            d_widen_u(v.z, o[4], o[5]);
            d_widen_u(v.w, o[6], o[7]);
            // the columns of K step j of block b (the address is the same for the
            // whole warp: tcgen05.st takes one address per warp)
            d_tmem_st8(tlane + (uint32_t)(32 * b + 8 * j), o);
        }
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void d_st_cluster(const void *local, uint32_t rank, int v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(d_smem(local)), "r"(rank));
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// The weight scale of one channel this CTA stores (thread tid < 128 / S), and a
// token scale (tid < M): loaded at entry into registers, stored into shared
// memory after the widening, so that their latency overlaps everything before.
struct ScalePrefetch {
    float w, t;
};
__device__ __forceinline__ ScalePrefetch d_load_scales(int tid, uint32_t rank, int nsplit, int64_t c0, const float *sw,
                                                       const float *sa, int M, int y_mode) {
    const int cw = DCH / nsplit;
    ScalePrefetch p{0.f, 0.f};
    if (y_mode != 2) {
        if (tid < cw) p.w = __ldg(sw + c0 + (int)rank * cw + tid);
        if (sa && tid < M) p.t = __ldg(sa + tid);
    }
    return p;
}
template <class S_>
__device__ __forceinline__ void d_store_scales(S_ &s, const ScalePrefetch &p, int tid, uint32_t rank, int nsplit,
                                               int M, bool tokens) {
    const int cw = DCH / nsplit;
    if (tid < cw) s.wsc[(int)rank * cw + tid] = p.w;
    if (tokens && tid < M) s.tsc[tid] = p.t;
}

// After every thread's operands are in place: one thread issues the slice's
// MMAs; the four lane-quarter warps turn the accumulators into exact integer
// partials acc 2^18 - 8 sum q_a and push each into the shared memory of the CTA
// that reduces its channel (remote stores complete without a round trip); then
// every CTA's abort flag goes to every CTA.  Returns this CTA's abort state.
template <int MT, bool WAIT_STARTED, class S_>
__device__ __forceinline__ bool d_product(S_ &s, uint32_t tmem, int nb, int tid, int warp, int lane, int M,
                                          uint32_t rank, int nsplit, int *err) {
    const unsigned full = 0xffffffffu;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if constexpr (WAIT_STARTED) d_cluster_wait();   // every CTA of the cluster has started
    const bool aborted = s.abort_flag != 0;
    if (tid == 0 && !aborted) {
        // K step 4 b + k accumulates into accumulator k: four independent chains
        for (int b = 0; b < nb; ++b) {
            const uint32_t bb = d_smem(s.opb[b]);
#pragma unroll
            for (int k = 0; k < DBK / 32; ++k)
                d_mma_ts<MT>(tmem + DACC_COL + (uint32_t)(16 * MT * k), tmem + (uint32_t)(32 * b + 8 * k),
                             d_sw128_desc(bb + 32 * k), b != 0);
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         d_smem(&s.mma_done))
                     : "memory");
    }
    bool ok = !aborted;
    if (warp < 4) {
        if (ok) ok = __all_sync(full, d_wait(&s.mma_done, 0, err));
        if (ok) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int r = 32 * warp + lane;
            const int cw = DCH / nsplit;
            const uint32_t owner = (uint32_t)(r / cw);
            int *dst = s.recv + (int)rank * (16 * MT) * cw + (r - (int)owner * cw);   // + m cw
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                int acc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = 0;
                uint32_t v[DNACC][16];   // the four accumulators' columns of token tile t, one wait
#pragma unroll
                for (int a = 0; a < DNACC; ++a)
                    d_tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + DACC_COL + (uint32_t)(16 * MT * a + 16 * t), v[a]);
                d_tmem_wait_ld();
#pragma unroll
                for (int a = 0; a < DNACC; ++a)   // each accumulator holds an exact multiple of 2^-18
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] += __float2int_rn(__uint_as_float(v[a][j]) * 262144.0f);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = 16 * t + j;
                    if (m < M) d_st_cluster(dst + m * cw, owner, acc[j] - 8 * s.qsum[m]);
                }
            }
        } else if (lane == 0) {
            s.abort_flag = 1;
        }
    }
    __syncthreads();   // this CTA's abort flag is final
    if (tid < nsplit) d_st_cluster(&s.aborts[rank], (uint32_t)tid, s.abort_flag);
    return aborted;
}

// After a cluster barrier: CTA `rank` adds the partials that the slices pushed
// for channels [128 rank / S, 128 (rank + 1) / S) and stores y (a token's scale
// from sa(m), the channel's from s.wsc, loaded at the start).
template <int MT, class S_, class Scale>
__device__ __forceinline__ void d_reduce_store(S_ &s, int tid, uint32_t rank, int nsplit, int M, int64_t N, int64_t c0,
                                               void *y, int y_mode, Scale sa) {
    const int cw = DCH / nsplit;
    bool any_abort = false;
    for (int j = 0; j < nsplit; ++j) any_abort |= s.aborts[j] != 0;
    if (any_abort) return;
    for (int e = tid; e < M * cw; e += DTHREADS) {
        const int m = e / cw, cc = e - m * cw, c = (int)rank * cw + cc;
        int tot = 0;
        for (int j = 0; j < nsplit; ++j) tot += s.recv[(j * (16 * MT) + m) * cw + cc];
        const int64_t col = c0 + c;
        const int64_t o = (int64_t)m * N + col;
        if (y_mode == 2) {
            static_cast<int *>(y)[o] = tot;
        } else {
            const float v = ((float)tot * sa(m)) * s.wsc[c];
            if (y_mode == 1) static_cast<float *>(y)[o] = v;
            else static_cast<__half *>(y)[o] = __float2half_rn(v);
        }
    }
}

// The end of both kernels (every remote store into this CTA came before the
// cluster barrier it has passed): no bulk copy into shared memory outlives the
// CTA; tensor memory is freed.
template <class S_>
__device__ __forceinline__ void d_teardown(S_ &s, uint32_t tmem, bool aborted, int tid, int warp, int nb, int *err) {
    if (aborted && tid == 0)
        for (int b = 0; b < nb; ++b) d_wait(&s.wfull[b], 0, err);
    __syncwarp();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(DTMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Decode product: activation codes read from HBM
// ---------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(DTHREADS, 1)
w4a4_decode_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ DParams prm) {
    using S_ = DSmem<MT, false>;
    extern __shared__ uint8_t smem_raw[];
    S_ &s = *reinterpret_cast<S_ *>(smem_raw + ((1024u - (d_smem(smem_raw) & 1023u)) & 1023u));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsplit = (int)gridDim.x;                 // CTAs of the cluster = K slices
    const uint32_t rank = blockIdx.x;                  // cluster dims (nsplit, 1, 1)
    const int64_t c0 = (int64_t)blockIdx.y * DCH;      // first output channel of the tile
    const int kblocks = (int)(prm.K / DBK);
    const int b0 = (int)(((int64_t)rank * kblocks) / nsplit);
    const int nb = (int)(((int64_t)(rank + 1) * kblocks) / nsplit) - b0;   // 1 .. DMAXB
    const int M = (int)prm.M;

    if (warp == 0) d_start_weights(s, &tmW, lane, b0, nb, c0);
    const uint8_t *abase = prm.aq + (int64_t)b0 * (DBK / 2);
    const int64_t lda = prm.K / 2;
    ActChunks<MT> acts;
    d_load_acts<MT>(acts, tid, nb, M, [&](int m, int off) {
        return __ldg(reinterpret_cast<const uint4 *>(abase + (int64_t)m * lda + off));
    });
    const ScalePrefetch sc = d_load_scales(tid, rank, nsplit, c0, prm.sw, prm.sa, M, prm.y_mode);
    const uint32_t tmem = d_setup(s, tid, warp, 16 * MT);
    d_widen_weights(s, tmem, nb, warp, lane, prm.err);   // each block as it lands
    d_store_acts<MT>(s, acts, tid, nb, M);
    d_store_scales(s, sc, tid, rank, nsplit, M, true);
    const bool aborted = d_product<MT, true>(s, tmem, nb, tid, warp, lane, M, rank, nsplit, prm.err);
    d_cluster_sync();   // every CTA's partials (and abort flag) are in place
    d_reduce_store<MT>(s, tid, rank, nsplit, M, prm.N, c0, prm.y, prm.y_mode, [&](int m) { return s.tsc[m]; });
    d_teardown(s, tmem, aborted, tid, warp, nb, prm.err);
}

// ---------------------------------------------------------------------------
// Fused decode: rotation + INT4 quantization + product in one launch
//
// The rows of x (M <= 16 tokens, n = K = 1024 .. 8192) are rotated by the
// CTAs of each cluster: CTA r takes tokens r, r + S, r + 2 S, ...  The rotated
// rows never reach HBM: each CTA quantizes its tokens and writes the packed
// codes of slice d into CTA d's shared memory (and every token's scale into
// every CTA), then the product runs as above.
//
// Rotation: the randomized Hadamard of "Rotational Quantization ..."
// §Incoherence Processing via Randomized Hadamard Transforms, as butterflies
// (§Weight Absorption and Online Fast Walsh-Hadamard Transforms, 2.).  The
// result of a Sylvester butterfly network in fp32 is fixed by the order in which
// its bit stages run, not by which thread computes what; here the stages run in
// the order the rotation kernel of rq_fwht_quant uses for the same n, so the
// codes and scales are those of rq_fwht_quant bit for bit.  The CTA's rows
// (padded with zero rows to T = 8192 or 16384 values) sit in shared memory as
// fp32 (XOR-swizzled so that every warp access is bank-conflict free); each pass
// loads E = T / 256 values per thread
// that differ in the pass's bits, runs those stages in registers (fp32 pairs)
// and stores them back.  Pass 0 reads x from HBM (runs of 8 consecutive
// elements: every stage order begins with bits 0, 1, 2).  The output phase
// gives each thread 32 consecutive values of a row: row absmax (warp maxima,
// shared-memory atomics), codes rne(y 7 / max|y|) by the same fused multiply-add
// against 1.5 2^23 as the rotation kernel, packing, and the stores.
// ---------------------------------------------------------------------------

// Stage order (element bits) of rq_fwht_quant's rotation kernel for n = 2^L.
__host__ __device__ constexpr int stage_bit(int L, int k) {
    constexpr int o10[10] = {0, 1, 2, 5, 6, 7, 8, 3, 4, 9};
    constexpr int o11[11] = {0, 1, 2, 5, 6, 7, 8, 3, 4, 9, 10};
    constexpr int o12[12] = {0, 1, 2, 6, 7, 8, 9, 10, 11, 3, 4, 5};
    constexpr int o13[13] = {0, 1, 2, 6, 7, 8, 9, 10, 11, 12, 3, 4, 5};
    return L == 10 ? o10[k] : (L == 11 ? o11[k] : (L == 12 ? o12[k] : o13[k]));
}

// Passes over the stage order: E2 bits per pass at most (E = 2^E2 values per
// thread), the first pass at least 3 bits (its runs of 8 are 16-byte loads), the
// last one full.
template <int L, int E2>
struct RotPasses {
    static constexpr int LT = 8 + E2;                  // index bits of the CTA's T values (8 thread bits)
    static constexpr int REM = L - E2;
    static constexpr int NP = REM <= E2 ? 2 : 3;
    static constexpr int size(int p) {
        return NP == 2 ? (p == 0 ? REM : E2)
                       : (p == 2 ? E2
                                 : (REM - E2 >= 3 ? (p == 0 ? REM - E2 : E2) : (p == 0 ? (REM + 1) / 2 : REM / 2)));
    }
    static constexpr int first(int p) { return p == 0 ? 0 : (p == 1 ? size(0) : size(0) + size(1)); }
    static constexpr int pbit(int p, int i) { return stage_bit(L, first(p) + i); }
    static constexpr bool in_pass(int p, int pos) {
        for (int i = 0; i < size(p); ++i)
            if (pbit(p, i) == pos) return true;
        return false;
    }
    // k-th lowest index bit not transformed by pass p: thread bits take k < 8,
    // the thread's value groups the rest
    static constexpr int comp(int p, int k) {
        int c = -1;
        for (int pos = 0; pos < LT; ++pos)
            if (!in_pass(p, pos) && ++c == k) return pos;
        return -1;
    }
    static constexpr int joff(int p, int j) {
        int g = 0;
        for (int i = 0; i < size(p); ++i)
            if ((j >> i) & 1) g |= 1 << pbit(p, i);
        return g;
    }
    static constexpr int goff(int p, int grp);   // below: needs the thread bit placement
    static_assert(L >= 10 && L <= 13 && (E2 == 5 || E2 == 6), "rotation sizes");
};

// Buffer position of value index g: g ^ f(g >> 5), f linear over GF(2) with
// column rot_swz_col(i) for index bit 5 + i.  A bijection inside each 32-word
// segment, and the bank of g is (g ^ f(g >> 5)) & 31.  The columns were chosen
// so that in every pass of every size above the five index bits that the lanes
// of a warp vary (rot_lane_pos) give five independent bank vectors: every
// 4-byte access of a warp touches 32 distinct banks.  Linear, so the position
// of a thread base | offset (disjoint bits) is the XOR of their positions.
__host__ __device__ constexpr int rot_swz_col(int i) {   // {25, 15, 16, 21, 13, 26, 7, 4, 16}
    return i == 0 ? 25 : (i == 1 ? 15 : (i == 2 ? 16 : (i == 3 ? 21 : (i == 4 ? 13 : (i == 5 ? 26 : (i == 6 ? 7 : (i == 7 ? 4 : 16)))))));
}
__host__ __device__ constexpr int rot_swz(int hi) {
    int f = 0;
    for (int i = 0; i < 9; ++i)
        if ((hi >> i) & 1) f ^= rot_swz_col(i);
    return f;
}
__host__ __device__ constexpr int rot_phys(int g) { return g ^ rot_swz(g >> 5); }
__host__ __device__ constexpr int rot_bank_vec(int pos) { return pos < 5 ? (1 << pos) : rot_swz_col(pos - 5); }

// Index bit of thread bit k (k < 5: the lanes, on the first index bits not in
// the pass whose bank vectors are independent; then the warp bits), and of the
// thread's value-group bit k.
template <int L, int E2>
__host__ __device__ constexpr int rot_tpos(int p, int k) {
    using RP = RotPasses<L, E2>;
    int basis[5] = {0, 0, 0, 0, 0};
    int lanes[5] = {-1, -1, -1, -1, -1};
    int nl = 0;
    for (int c = 0; c < RP::LT - RP::size(p) && nl < 5; ++c) {
        const int pos = RP::comp(p, c);
        int v = rot_bank_vec(pos);
        for (int b = 4; b >= 0; --b) {
            if (!((v >> b) & 1)) continue;
            if (!basis[b]) {
                basis[b] = v;
                lanes[nl++] = pos;
                break;
            }
            v ^= basis[b];
        }
    }
    if (k < 5) return lanes[k];
    int r = -1;   // the (k - 5)-th index bit outside the pass that is not a lane bit
    for (int c = 0; c < RP::LT - RP::size(p); ++c) {
        const int pos = RP::comp(p, c);
        bool lane = false;
        for (int i = 0; i < 5; ++i) lane = lane || lanes[i] == pos;
        if (!lane && ++r == k - 5) return pos;
    }
    return -1;
}

template <int L, int E2>
constexpr int RotPasses<L, E2>::goff(int p, int grp) {
    int g = 0;
    for (int k = 0; k < E2 - size(p); ++k)
        if ((grp >> k) & 1) g |= 1 << rot_tpos<L, E2>(p, 8 + k);
    return g;
}

// Compile-time constants of pass P: index bit of thread bit K, and the (raw,
// swizzled) offset of the thread's value A.
template <int L, int E2, int P, int K>
struct RotTPos {
    static constexpr int value = rot_tpos<L, E2>(P, K);
};
template <int L, int E2, int P, int A>
struct RotOff {
    static constexpr int e = RotPasses<L, E2>::size(P);
    static constexpr int raw = RotPasses<L, E2>::goff(P, A >> e) | RotPasses<L, E2>::joff(P, A & ((1 << e) - 1));
    static constexpr int phys = rot_phys(raw);
};

template <int L, int E2, int P, int... K>
__device__ __forceinline__ int rot_thread_base_impl(int t, std::integer_sequence<int, K...>) {
    return (0 | ... | (((t >> K) & 1) << RotTPos<L, E2, P, K>::value));
}
template <int L, int E2, int P>
__device__ __forceinline__ int rot_thread_base(int t) {
    return rot_thread_base_impl<L, E2, P>(t, std::make_integer_sequence<int, 8>{});
}

// Stages of pass P on the thread's values (array bit i = the pass's i-th stage).
template <int L, int E2, int P>
__device__ __forceinline__ void rot_stages(pair_t (&v)[(1 << E2) / 2]) {
    constexpr int e = RotPasses<L, E2>::size(P);
#pragma unroll
    for (int i = 0; i < (1 << E2) / 2; ++i) v[i] = bfly_in(v[i]);
#pragma unroll
    for (int rb = 1; rb < e; ++rb) butterfly_pairs<(1 << E2) / 2>(v, rb);
}

template <int L, int E2, int P, int... A>
__device__ __forceinline__ void rot_store_impl(float *xs, const pair_t (&v)[(1 << E2) / 2], int tphys,
                                               std::integer_sequence<int, A...>) {
    ((xs[tphys ^ RotOff<L, E2, P, A>::phys] = (A & 1) ? hi2(v[A >> 1]) : lo2(v[A >> 1])), ...);
}
template <int L, int E2, int P>
__device__ __forceinline__ void rot_store(float *xs, const pair_t (&v)[(1 << E2) / 2], int tphys) {
    rot_store_impl<L, E2, P>(xs, v, tphys, std::make_integer_sequence<int, (1 << E2)>{});
}

template <int L, int E2, int P, int... A2>
__device__ __forceinline__ void rot_load_impl(const float *xs, pair_t (&v)[(1 << E2) / 2], int tphys,
                                              std::integer_sequence<int, A2...>) {
    ((v[A2] = mk2(xs[tphys ^ RotOff<L, E2, P, 2 * A2>::phys], xs[tphys ^ RotOff<L, E2, P, 2 * A2 + 1>::phys])), ...);
}
template <int L, int E2, int P>
__device__ __forceinline__ void rot_load(const float *xs, pair_t (&v)[(1 << E2) / 2], int tphys) {
    rot_load_impl<L, E2, P>(xs, v, tphys, std::make_integer_sequence<int, (1 << E2) / 2>{});
}

template <int L, int E2, int P, int... R>
__device__ __forceinline__ void rot_run_offsets(int (&o)[sizeof...(R)], std::integer_sequence<int, R...>) {
    ((o[R] = RotOff<L, E2, P, 8 * R>::raw), ...);
}

struct FParams {
    const void *x;
    int64_t ldx;
    int in_type;            // IN_BF16 or IN_F16
    uint64_t seed;
    uint32_t flags;
    const float *sw;
    void *y;
    int64_t M, N, K;
    int y_mode;
    uint8_t *aq_out;        // optional [M][K/2]
    float *as_out;          // optional [M]
    int *err;
};

template <int L, int E2>
__global__ void __launch_bounds__(DTHREADS, 1)
fused_decode_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ FParams prm) {
    using S_ = DSmem<1, true>;
    using RP = RotPasses<L, E2>;
    constexpr int n = 1 << L;
    constexpr int E = 1 << E2;                          // values per thread and pass
    constexpr int T = 256 * E;                          // values in the CTA's rotation buffer
    constexpr int RPAD = T / n;                         // rows in the buffer (zero rows pad)
    extern __shared__ uint8_t smem_raw[];
    S_ &s = *reinterpret_cast<S_ *>(smem_raw + ((1024u - (d_smem(smem_raw) & 1023u)) & 1023u));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned full = 0xffffffffu;
    const int nsplit = (int)gridDim.x;
    const uint32_t rank = blockIdx.x;
    const int64_t c0 = (int64_t)blockIdx.y * DCH;
    const int kblocks = n / DBK;
    const int b0 = (int)(((int64_t)rank * kblocks) / nsplit);
    const int nb = (int)(((int64_t)(rank + 1) * kblocks) / nsplit) - b0;
    const int M = (int)prm.M;
    const bool signs_first = (prm.flags & 1u) != 0;

    if (warp == 0) d_start_weights(s, &tmW, lane, b0, nb, c0);
    const ScalePrefetch sc = d_load_scales(tid, rank, nsplit, c0, prm.sw, nullptr, M, prm.y_mode);
    const uint32_t tmem = d_setup(s, tid, warp, 16);

    // sign bits: word j holds elements 32 j .. 32 j + 31 (one SplitMix64 output each)
    for (int base = 0; base < n; base += DTHREADS) {
        const uint32_t bit = (uint32_t)(splitmix64_at(prm.seed, (uint64_t)(base + tid)) >> 63);
        const uint32_t word = __ballot_sync(full, bit != 0);
        if (lane == 0) s.sgn[(base + 32 * warp) >> 5] = word;
    }
    if (tid < 16) s.rowmax[tid] = 0u;
    __syncthreads();

    // pass 0: x from HBM (tokens rank + S i; rows past M or past the CTA's share are zero)
    pair_t v[E / 2];
    {
        constexpr int P = 0, e = RP::size(0);
        const int tb = rot_thread_base<L, E2, P>(tid);
        int run_off[E / 8];   // raw index offset of each run of 8 values (compile-time constants)
        rot_run_offsets<L, E2, P>(run_off, std::make_integer_sequence<int, E / 8>{});
#pragma unroll
        for (int a8 = 0; a8 < E; a8 += 8) {
            const int g = tb | run_off[a8 >> 3];
            const int elem = g & (n - 1), row = g >> L;
            const int64_t m = (int64_t)rank + (int64_t)nsplit * row;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (m < M)
                raw = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(prm.x) + m * prm.ldx + elem));
            const uint32_t sg = signs_first ? (s.sgn[elem >> 5] >> (elem & 24)) & 0xffu : 0u;
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float f0, f1;
                if (prm.in_type == IN_BF16) {
                    f0 = __uint_as_float(w[k] << 16);
                    f1 = __uint_as_float(w[k] & 0xffff0000u);
                } else {
                    const __half2 h = *reinterpret_cast<const __half2 *>(&w[k]);
                    const float2 f = __half22float2(h);
                    f0 = f.x;
                    f1 = f.y;
                }
                f0 = __uint_as_float(__float_as_uint(f0) ^ (((sg >> (2 * k)) & 1u) << 31));
                f1 = __uint_as_float(__float_as_uint(f1) ^ (((sg >> (2 * k + 1)) & 1u) << 31));
                v[(a8 >> 1) + k] = mk2(f0, f1);
            }
        }
        rot_stages<L, E2, P>(v);
        rot_store<L, E2, P>(s.xs, v, rot_phys(tb));
    }
    __syncthreads();
    {
        constexpr int P = 1;
        const int tb = rot_phys(rot_thread_base<L, E2, P>(tid));
        rot_load<L, E2, P>(s.xs, v, tb);
        rot_stages<L, E2, P>(v);
        __syncthreads();   // every thread's loads of this pass are done before the stores
        rot_store<L, E2, P>(s.xs, v, tb);
    }
    __syncthreads();
    if constexpr (RP::NP == 3) {
        constexpr int P = 2;
        const int tb = rot_phys(rot_thread_base<L, E2, P>(tid));
        rot_load<L, E2, P>(s.xs, v, tb);
        rot_stages<L, E2, P>(v);
        __syncthreads();
        rot_store<L, E2, P>(s.xs, v, tb);
        __syncthreads();
    }

    d_cluster_wait();   // every CTA of the cluster has started: remote stores below

    // output phase: thread-chunk c = 32 consecutive values of a row (c = tid + 256 i)
    constexpr int CPT = T / 32 / DTHREADS;              // chunks per thread: 1 or 2
    float yv[CPT][32];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + DTHREADS * i;
        const int row = (32 * c) >> L, cq = c & (n / 32 - 1);
        const uint32_t sg = signs_first ? 0u : s.sgn[cq];
        const int fc = rot_swz(c);                        // value k of chunk c sits at 32 c + (k ^ fc)
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float val = s.xs[32 * c + (k ^ fc)];
            val = __uint_as_float(__float_as_uint(val) ^ (((sg >> k) & 1u) << 31));
            yv[i][k] = val;
            mx = fmaxf(mx, fabsf(val));
        }
        // the 32 chunks of a warp lie in one row (a row holds n / 32 >= 32 chunks)
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(full, mx, o));
        if (lane == 0) atomicMax(&s.rowmax[row], __float_as_uint(mx));
    }
    __syncthreads();
    const float inv_sqrt_n = (L & 1) ? (0.70710678118654752440f / (float)(1 << (L / 2))) : (1.0f / (float)(1 << (L / 2)));
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + DTHREADS * i;
        const int row = (32 * c) >> L, cq = c & (n / 32 - 1);
        const int64_t m = (int64_t)rank + (int64_t)nsplit * row;
        if (m >= M) continue;
        const float amax = __uint_as_float(s.rowmax[row]);
        const float inv = amax > 0.f ? 7.0f / amax : 0.f;
        uint32_t words[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t code[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) code[k] = __float_as_uint(__fmaf_rn(yv[i][8 * q + k], inv, 12582912.0f));
            words[q] = pack8(code);
        }
        const uint4 packed = make_uint4(words[0], words[1], words[2], words[3]);
        // owner of K block cq / 4 and the offset inside its slice
        const int blk = cq >> 2;
        int d = 0;
        while (d + 1 < nsplit && (int)(((int64_t)(d + 1) * kblocks) / nsplit) <= blk) ++d;
        const int off = (blk - (int)(((int64_t)d * kblocks) / nsplit)) * (DBK / 2) + 16 * (cq & 3);
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(d_smem(&s.apk[m][off])), "r"((uint32_t)d));
        asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(packed.x), "r"(packed.y),
                     "r"(packed.z), "r"(packed.w)
                     : "memory");
        if (prm.aq_out) *reinterpret_cast<uint4 *>(prm.aq_out + m * (int64_t)(n / 2) + 16 * cq) = packed;
        if (cq == 0) {
            const float scale = (amax / 7.0f) * inv_sqrt_n;
            for (int j = 0; j < nsplit; ++j) {
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(d_smem(&s.asc[m])), "r"((uint32_t)j));
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(scale) : "memory");
            }
            if (prm.as_out) prm.as_out[m] = scale;
        }
    }
    d_cluster_sync();   // every token's codes of this CTA's slice, and every scale, are in place

    {
        ActChunks<1> acts;
        d_load_acts<1>(acts, tid, nb, M, [&](int m, int off) { return *reinterpret_cast<const uint4 *>(&s.apk[m][off]); });
        d_store_acts<1>(s, acts, tid, nb, M);
    }
    d_store_scales(s, sc, tid, rank, nsplit, M, false);
    d_widen_weights(s, tmem, nb, warp, lane, prm.err);
    const bool aborted = d_product<1, false>(s, tmem, nb, tid, warp, lane, M, rank, nsplit, prm.err);
    d_cluster_sync();
    d_reduce_store<1>(s, tid, rank, nsplit, M, prm.N, c0, prm.y, prm.y_mode, [&](int m) { return s.asc[m]; });
    d_teardown(s, tmem, aborted, tid, warp, nb, prm.err);
    (void)RPAD;
}

// K slices per channel tile: a power of two with at most DMAXB blocks per CTA,
// raised while the grid still fits one wave of one CTA per SM.  0: K too large.
int pick_split(int64_t kblocks, int64_t tiles, int sms) {
    int s = 1;
    while ((int64_t)s * DMAXB < kblocks) s <<= 1;
    if (s > DMAXS) return 0;
    while (s < DMAXS && 2 * s <= kblocks && tiles * 2 * s <= sms) s <<= 1;
    return s;
}

// At most one CTA per SM: each allocates all 512 TMEM columns, and a second CTA
// blocked in tcgen05.alloc while its cluster peers wait at a cluster barrier
// could stall two clusters on each other.  Two CTAs of this size do not fit in
// an SM's 228 KB.
template <class S_>
constexpr size_t launch_smem() {
    return sizeof(S_) + 1024 > kOneCtaPerSmBytes ? sizeof(S_) + 1024 : kOneCtaPerSmBytes;
}

template <class Kern, class Params>
cudaError_t launch_cluster(Kern kern, size_t smem, int nsplit, int64_t tiles, const CUtensorMap &tw, const Params &p,
                           cudaStream_t stream) {
    // set on every launch: the attribute is per device, and a process may use several
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit, (unsigned)tiles);
    cfg.blockDim = dim3(DTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tw, p);
}

template <int MT>
cudaError_t launch_decode_mt(const GemmArgs &g, int nsplit, cudaStream_t stream) {
    CUtensorMap tw;
    if (!make_tma_map_u8(&tw, g.w_q, g.N, g.K / 2, DBK / 2, DCH, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
    const DParams p{g.a_q, g.a_scales, g.w_scales, g.y, g.M, g.N, g.K, g.y_mode, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    return launch_cluster(w4a4_decode_tc_kernel<MT>, launch_smem<DSmem<MT, false>>(), nsplit, g.N / DCH, tw, p, stream);
}

template <int L>
cudaError_t launch_fused_l(const FParams &p, const CUtensorMap &tw, int nsplit, cudaStream_t stream) {
    // the CTA's rows (tokens rank + S i, at most 16 / S of them) padded to a power
    // of two, and to at least 8192 values: E = 32 or 64 values per thread
    int rows = (int)((16 + nsplit - 1) / nsplit);
    rows = rows > (int)((p.M + nsplit - 1) / nsplit) ? (int)((p.M + nsplit - 1) / nsplit) : rows;
    int rpad = 1;
    while (rpad < rows) rpad <<= 1;
    const bool e64 = (int64_t)rpad << L > 8192;
    const int64_t tiles = p.N / DCH;
    if (e64) return launch_cluster(fused_decode_tc_kernel<L, 6>, launch_smem<DSmem<1, true>>(), nsplit, tiles, tw, p, stream);
    return launch_cluster(fused_decode_tc_kernel<L, 5>, launch_smem<DSmem<1, true>>(), nsplit, tiles, tw, p, stream);
}

}  // namespace

bool w4a4_gemm_decode_tc_supported(const GemmArgs &g) {
    return g.M >= 1 && g.M <= 64 && g.N % DCH == 0 && g.N / DCH <= 65535 && g.K % DBK == 0 &&
           g.K <= (int64_t)DBK * DMAXB * DMAXS;
}

cudaError_t launch_w4a4_gemm_decode_tc(const GemmArgs &g, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const int nsplit = pick_split(g.K / DBK, g.N / DCH, sms);
    if (nsplit == 0) return cudaErrorInvalidValue;
    switch ((g.M + 15) / 16) {
        case 1: return launch_decode_mt<1>(g, nsplit, stream);
        case 2: return launch_decode_mt<2>(g, nsplit, stream);
        case 3: return launch_decode_mt<3>(g, nsplit, stream);
        default: return launch_decode_mt<4>(g, nsplit, stream);
    }
}

bool fused_decode_supported(int64_t M, int64_t K, int64_t N) {
    return M >= 1 && M <= 16 && (K == 1024 || K == 2048 || K == 4096 || K == 8192) && N % DCH == 0 &&
           N / DCH <= 65535;
}

cudaError_t launch_fused_decode(const void *x, int in_type, int64_t M, int64_t ldx, uint64_t seed, uint32_t flags,
                                const uint8_t *wq, const float *sw, int64_t N, int64_t K, void *y, int y_mode,
                                uint8_t *aq, float *as, cudaStream_t stream) {
    if (!fused_decode_supported(M, K, N) || (in_type != IN_BF16 && in_type != IN_F16)) return cudaErrorInvalidValue;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const int nsplit = pick_split(K / DBK, N / DCH, sms);
    if (nsplit == 0) return cudaErrorInvalidValue;
    CUtensorMap tw;
    if (!make_tma_map_u8(&tw, wq, N, K / 2, DBK / 2, DCH, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
    const FParams p{x, ldx, in_type, seed, flags, sw, y, M, N, K, y_mode, aq, as, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    switch (K) {
        case 1024: return launch_fused_l<10>(p, tw, nsplit, stream);
        case 2048: return launch_fused_l<11>(p, tw, nsplit, stream);
        case 4096: return launch_fused_l<12>(p, tw, nsplit, stream);
        default: return launch_fused_l<13>(p, tw, nsplit, stream);
    }
}

}  // namespace rq
