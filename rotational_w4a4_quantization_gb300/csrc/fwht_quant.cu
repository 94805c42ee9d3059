// fwht_quant.cu -- randomized fast Walsh-Hadamard transform fused with per-row
// symmetric INT4 quantization and nibble packing (sm_103a).
//
// Computes, for every row x of length n = 2^L (the activation of one token, one
// (token, head) vector of K or V, or one output channel of W^T for the offline
// fold):
//   y = x diag(s) H_n    (RQ_SIGNS_FIRST)   or   y = x H_n diag(s)   (flags 0)
//   scale = max|y| / 7,  q = round_half_even(y / scale),  packed two per byte.
// H_n is the Sylvester Hadamard of the H_2k recursion in "Rotational
// Quantization ..." §Incoherence Processing via Randomized Hadamard Transforms;
// the transform is the butterfly form of §Weight Absorption and Online Fast
// Walsh-Hadamard Transforms, 2. (n log2 n additions/subtractions and a single
// 1/sqrt(n) scale, which here folds into the stored scale: the codes depend only
// on y/max|y|).
//
// Design (HBM-bound; every input byte is read once and every output byte
// written once):
//  * An element index i = 8*c + e splits into the position e inside an
//    8-element "chunk" (one 16-byte bf16/fp16 vector) and the chunk index c
//    (C = L-3 bits).  Each thread owns 16 chunks (128 elements) of one row in
//    registers; P = 2^(C-4) threads share a row (1 for n <= 128, 32 for n = 4096,
//    64 for n = 8192).
//  * Loads never stall the butterflies: every warp copies its NEXT group of rows
//    into a private shared-memory buffer with cp.async while it computes the
//    current one.  The buffer is laid out lane-major per 16-byte granule, so the
//    phase-1 reads (one 128-bit load per chunk) are bank-conflict free.
//  * Values live as fp32 pairs in 64-bit registers for the whole transform, so
//    every butterfly stage except the one inside a pair runs two lanes at a time
//    with the packed add/sub.f32x2; the in-pair stage is fused with the bf16
//    unpack (mixed-precision add/sub.f32.bf16 on the two halves of a word).
//  * Phase 1: the thread reads its chunks (chunk bits 0,1 on lanes, so four
//    lanes fetch 64 contiguous bytes from HBM), flips signs, and runs the
//    butterflies of every bit it holds (e bits and 4 chunk bits) in registers;
//    one or two further bits for n >= 4096 are exchanged with warp shuffles.
//  * The row goes through shared memory once, as fp32 (XOR-swizzled 16-byte
//    granules: conflict-free for n >= 1024), into the phase-2 layout, where the
//    thread holds the remaining bits plus chunk bits 0 and 1, i.e. four runs
//    of 32 consecutive elements.
//  * Phase 2: remaining butterflies, row absmax (registers, shuffles, and a
//    shared-memory exchange when a row spans two warps), codes by one fused
//    multiply-add against a 1.5*2^23 bias, two values per f32x2 FMA
//    (round-half-even to an integer whose low bits are the two's-complement
//    code), packing with byte permutes, and
//    16-byte stores of 32 codes each, coalesced across the warp.
//  * CTAs are persistent: each computes the sign masks of its n positions once
//    (SplitMix64, one call per element) into shared memory, while its first
//    input copies are in flight, and then walks groups of rows.
//  * n = 4096 and n = 8192 (the activation sizes of the serving paths) have
//    their own variants with 64 values per thread and three butterfly phases
//    joined by two shared-memory transposes, without shuffles (see below); the
//    plans above serve n <= 2048.
#include "rq.h"
#include "rq_internal.h"
#include "rot_device.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rq {
namespace {


// --------------------------------------------------------------------------
// Bit plans.  a(k)/ta(k): chunk bit held by phase-1 slot bit k / row-thread
// bit k.  b(k)/tb(k): the same for phase 2.  shuf(j): the row-thread bits of
// phase 1 whose butterflies run through warp shuffles.
// --------------------------------------------------------------------------
template <int C>
struct Plan {
    // slot bits per thread: the whole row for n <= 64, half a row for n = 128
    // (two threads per row: a lighter register footprint, so more warps hide
    // the butterflies' latencies), 16 chunks beyond that
    static constexpr int S = C <= 3 ? C : (C == 4 ? 3 : 4);
    static constexpr int T = C - S;
    static constexpr int P = 1 << T;
    static constexpr int NSLOT = 1 << S;
    static constexpr int E = 8 * NSLOT;
    static constexpr bool kTwoPhase = C >= 5;

    static constexpr int a(int k) {
        return C <= 4 ? k : (C == 5 ? k + 1 : k + 2);
    }
    static constexpr int ta(int k) {
        // C=4: {3}; C=5: {0}; C=6: {0,1}; C>=7: {0,1,6,7,...}
        return C == 4 ? 3 : (k < 2 ? k : k + 4);
    }
    static constexpr int b(int k) {
        if (C <= 4) return k;
        if (C <= 6) return k;                   // {0,1,2,3}
        return k < 2 ? k : C - 4 + k;           // {0,1,C-2,C-1}
    }
    static constexpr int tb(int k) {
        if (C <= 6) return 4 + k;               // {4} / {4,5}
        return 2 + k;                           // {2,...}
    }
    static constexpr int kNumShuf = C >= 9 ? C - 8 : (C == 4 ? 1 : 0);
    // row-thread bits exchanged by shuffles: bit 0 for n = 128, bits 2 (and 3) for n >= 4096
    static constexpr int shuf(int j) { return C == 4 ? 0 : 2 + j; }

    static constexpr bool chunk_bit_done_in_phase1(int cb) {
        for (int k = 0; k < S; ++k)
            if (a(k) == cb) return true;
        for (int j = 0; j < kNumShuf; ++j)
            if (ta(shuf(j)) == cb) return true;
        return false;
    }
};

struct KParams {
    RotJob job[2];
    int njobs;
    int64_t groups_per_job;
    uint64_t seed;
    uint32_t flags;
    int *err;          // library error word: set when a bounded wait gives up
};

constexpr long long kWaitLimitCycles = 4000000000ll;    // ~2 s at 2 GHz

// Job of row group g (jobs hold groups_per_job groups each; at most two jobs, so
// a comparison replaces the 64-bit division).
__device__ __forceinline__ int job_of(int64_t g, int64_t groups_per_job) { return g >= groups_per_job ? 1 : 0; }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for a bulk copy; on expiry raise the error word and report failure.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, uint32_t parity, int *err,
                                                  long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > limit) {
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}
// Bulk global -> shared copy (TMA engine), completing on an mbarrier.
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Shared-memory granule position of 16-byte half h of chunk c in a row buffer:
// (2c + h) ^ swz(c) ^ (row & 7).  swz is a XOR of chunk bits, so for c = cs | ct
// (slot bits cs known at compile time, thread bits ct at run time, disjoint)
// the position splits into granule_k(cs, h) ^ granule_t(ct, row).
__host__ __device__ constexpr int swz(int c) {
    return (((c >> 2) ^ (c >> 6)) & 1) | (((c >> 3) & 1) << 1) | (((c >> 4) & 1) << 2);
}
__host__ __device__ constexpr int granule_k(int cs, int h) { return (2 * cs + h) ^ swz(cs); }
__device__ __forceinline__ int granule_t(int ct, int row_in_cta) { return (2 * ct) ^ swz(ct) ^ (row_in_cta & 7); }

// chunk index = slot part | thread part
template <int C>
__host__ __device__ constexpr int chunk_s(int s, bool phase2) {
    int c = 0;
    for (int k = 0; k < Plan<C>::S; ++k) c |= ((s >> k) & 1) << (phase2 ? Plan<C>::b(k) : Plan<C>::a(k));
    return c;
}
template <int C>
__device__ __forceinline__ int chunk_t(int t, bool phase2) {
    using PL = Plan<C>;
    int c = 0;
#pragma unroll
    for (int k = 0; k < PL::T; ++k) c |= ((t >> k) & 1) << (phase2 ? PL::tb(k) : PL::ta(k));
    return c;
}
template <int C>
__device__ __forceinline__ int chunk_of(int t, int s, bool phase2) {
    return chunk_s<C>(s, phase2) | chunk_t<C>(t, phase2);
}

// Threads per CTA: 8 warps for the two-phase plans with 16-bit input, so that
// one CTA per SM shares the sign-mask setup (n SplitMix64 calls) among 8 rows;
// 4 warps otherwise (with fp32 input, 8 warps' input rings and row buffers would
// not fit in shared memory).
__host__ __device__ constexpr int threads_for(int log_n, int in_type) {
    return (log_n - 3 >= 5 && in_type != IN_F32) ? 256 : 128;
}

template <int LOGN, int IN>
__global__ void __launch_bounds__(threads_for(LOGN, IN), LOGN == 7 ? 4 : 1)
fwht_quant_kernel(const __grid_constant__ KParams prm) {
    constexpr int C = LOGN - 3;
    using PL = Plan<C>;
    constexpr int n = 1 << LOGN;
    constexpr int NSLOT = PL::NSLOT;
    constexpr int NP = PL::E / 2;                        // fp32 pairs per thread
    constexpr int P = PL::P;
    constexpr int THREADS = threads_for(LOGN, IN);
    constexpr int ROWS = THREADS / P;
    constexpr int G = IN == IN_F32 ? 2 : 1;              // 16-byte granules per chunk
    constexpr int Q = NSLOT * G;                         // granules per thread per group
    constexpr int ES = IN == IN_F32 ? 4 : 2;             // input element bytes

    constexpr int DEPTH = PL::kTwoPhase ? 1 : 2;          // input groups in flight per warp
    constexpr int NW = THREADS / 32;
    constexpr int WREG = 32 * Q * 16;                     // bytes of one warp's input region
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);                       // NW*DEPTH
    uint32_t *sgn = reinterpret_cast<uint32_t *>(smem_raw + 128);                  // n/2 words
    float *red = reinterpret_cast<float *>(smem_raw + 128 + n * 2);               // ROWS*2 floats
    unsigned char *inbuf = smem_raw + 128 + n * 2 + 128 * ((ROWS * 2 * 4 + 127) / 128);
    ulonglong2 *rowbuf = reinterpret_cast<ulonglong2 *>(inbuf + NW * DEPTH * WREG);
    // one row per thread: packed codes of a warp's 32 rows (contiguous in q) are
    // staged here and written by one bulk store; two buffers per warp
    constexpr int OSTG = PL::kTwoPhase ? 0 : (32 / P) * (n / 2);
    unsigned char *ostage = inbuf + NW * DEPTH * WREG + (PL::kTwoPhase ? (size_t)ROWS * n * 4 : 0);

    const bool signs_first = (prm.flags & 1u) != 0;
    const uint32_t msel = signs_first ? 0xffffffffu : 0u;

    if (threadIdx.x < NW * DEPTH) mbar_init(&bars[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();    // barriers initialized before the warps issue their first copies

    const int row_in_cta = threadIdx.x / P;
    const int t = threadIdx.x % P;
    const int lane = threadIdx.x & 31;
    const int gt1 = granule_t(chunk_t<C>(t, false), row_in_cta);   // per-thread swizzle parts
    const int gt2 = granule_t(chunk_t<C>(t, true), row_in_cta);
    const float inv_sqrt_n = (LOGN & 1) ? (0.70710678118654752440f / (float)(1 << (LOGN / 2)))
                                        : (1.0f / (float)(1 << (LOGN / 2)));
    const unsigned full = 0xffffffffu;
    const int warp = threadIdx.x >> 5;
    const int64_t total_groups = prm.groups_per_job * prm.njobs;

    // Single-phase plans: the threads of warp row r read their chunks in slot
    // order s ^ r, so a shared-memory wavefront spreads over the bank groups of
    // the linear input copy.  Running the Sylvester network on input permuted by
    // XOR with a leaves output j in place but multiplied by (-1)^popcount(j & a);
    // all threads of a row share a, so the factor passes through the shuffle
    // stage and is folded into the quantization multiplier below.  Two-phase
    // plans exchange values between rows' threads with different layouts, so
    // they read in natural order (a = 0).
    const int xr = PL::kTwoPhase ? 0 : ((lane / P) & (NSLOT - 1));
    const int cb1 = chunk_t<C>(t, false) | chunk_s<C>(xr, false);   // chunk(s) = cb1 ^ chunk_s(s)
    // byte offset of this thread's chunk base inside the warp's input region
    constexpr int RB = n * ES;                                        // bytes per input row
    constexpr int RPW = P <= 32 ? 32 / P : 1;                         // rows per warp region
    constexpr int REG_BYTES = P <= 32 ? RPW * RB : RB / 2;
    static_assert(REG_BYTES == WREG, "warp input region size");
    const int rw = P <= 32 ? lane / P : 0;                            // row within the warp region
    const uint32_t xin = (uint32_t)(rw * RB) + (uint32_t)((16 * G * cb1) & (P <= 32 ? RB - 1 : RB / 2 - 1));
    // transpose swizzle base including the XOR permutation
    const int gt1x = gt1 ^ granule_k(chunk_s<C>(xr, false), 0);

    // Issue the bulk copies of group g's rows for this warp (lane 0 only).
    auto issue = [&](int64_t g, int slot) {
        const int jb = job_of(g, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row0 = (g - (int64_t)jb * prm.groups_per_job) * ROWS + (P <= 32 ? warp * RPW : warp / 2);
        const char *x = static_cast<const char *>(job.x);
        unsigned char *dst = inbuf + (warp * DEPTH + slot) * WREG;
        uint64_t *bar = &bars[warp * DEPTH + slot];
        if constexpr (P <= 32) {
            int64_t valid = job.rows - row0;
            valid = valid < 0 ? 0 : (valid > RPW ? RPW : valid);
            mbar_expect_tx(bar, (uint32_t)(valid * RB));
            if (job.ld * ES == RB) {
                if (valid > 0) bulk_copy(dst, x + row0 * RB, (uint32_t)(valid * RB), bar);
            } else {
                for (int r = 0; r < valid; ++r) bulk_copy(dst + r * RB, x + (row0 + r) * job.ld * ES, RB, bar);
            }
        } else {
            const bool valid = row0 < job.rows;
            mbar_expect_tx(bar, valid ? (uint32_t)(RB / 2) : 0u);
            if (valid) bulk_copy(dst, x + row0 * job.ld * ES + (warp & 1) * (RB / 2), RB / 2, bar);
        }
    };

    if (lane == 0) {
#pragma unroll
        for (int d = 0; d < DEPTH; ++d) {
            const int64_t g = (int64_t)blockIdx.x + (int64_t)d * gridDim.x;
            if (g < total_groups) issue(g, d);
        }
    }
    // Sign masks (computed while the first copies are in flight): word j covers elements 2j (bit 15) and 2j+1 (bit 31).
    for (int j = threadIdx.x; j < n / 2; j += THREADS) {
        const uint32_t s0 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j) >> 63);
        const uint32_t s1 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j + 1) >> 63);
        sgn[j] = (s0 << 15) | (s1 << 31);
    }
    __syncthreads();


    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    int obuf = 0;
    for (int64_t grp = blockIdx.x; grp < total_groups; grp += gridDim.x) {
        const int jb = job_of(grp, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (grp - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;
        const unsigned char *wbuf = inbuf + (warp * DEPTH + slot) * WREG;

        pair_t v[NP];
        // ---------------- phase 1: input from the bulk copy, signs, butterflies ----------------
        // A copy that never lands raises the error word; the iteration then runs
        // on stale data with its stores disabled, so barriers stay matched.
        if (!mbar_wait_bounded(&bars[warp * DEPTH + slot], phase, prm.err)) aborted = true;
        const bool active = row < job.rows && !aborted;
#pragma unroll
        for (int s = 0; s < NSLOT; ++s) {
            const int c = cb1 ^ chunk_s<C>(s, false);
            const uint4 m = reinterpret_cast<const uint4 *>(sgn)[c];
            uint4 g[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint32_t off = (xin ^ (uint32_t)(16 * G * chunk_s<C>(s, false))) + 16 * h;
                g[h] = *reinterpret_cast<const uint4 *>(wbuf + off);
            }
            convert_chunk<IN>(g, m, msel, &v[4 * s]);   // includes the in-pair stage
        }
        // Hand the buffer back to the copy engine: order these generic reads
        // before the next bulk write (async proxy) into it.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && !aborted) {
            const int64_t g = grp + (int64_t)DEPTH * gridDim.x;
            if (g < total_groups) issue(g, slot);
        }
        if (++slot == DEPTH) {
            slot = 0;
            phase ^= 1u;
        }

#pragma unroll
        for (int rb = 1; rb < 3 + PL::S; ++rb) butterfly_pairs<NP>(v, rb);
#pragma unroll
        for (int j = 0; j < PL::kNumShuf; ++j) {
            const int lm = 1 << PL::shuf(j);
            const float sg = ((t >> PL::shuf(j)) & 1) ? -1.f : 1.f;
            const pair_t sg2 = mk2(sg, sg);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const float p0 = __shfl_xor_sync(full, lo2(v[i]), lm);
                const float p1 = __shfl_xor_sync(full, hi2(v[i]), lm);
                v[i] = fma2(v[i], sg2, mk2(p0, p1));
            }
        }

        // ---------------- transpose through shared memory ----------------
        if constexpr (PL::kTwoPhase) {
            ulonglong2 *buf = rowbuf + (size_t)row_in_cta * (n / 4);
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) {
                const int cs = chunk_s<C>(s, false);
                buf[granule_k(cs, 0) ^ gt1x] = make_ulonglong2(v[4 * s], v[4 * s + 1]);
                buf[granule_k(cs, 1) ^ gt1x] = make_ulonglong2(v[4 * s + 2], v[4 * s + 3]);
            }
            if constexpr (P > 32) {
                asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            } else {
                __syncwarp();
            }
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) {
                const int cs = chunk_s<C>(s, true);
                const ulonglong2 lo = buf[granule_k(cs, 0) ^ gt2];
                const ulonglong2 hi = buf[granule_k(cs, 1) ^ gt2];
                v[4 * s] = lo.x; v[4 * s + 1] = lo.y; v[4 * s + 2] = hi.x; v[4 * s + 3] = hi.y;
            }
            // phase-2 butterflies over the slot bits not done in phase 1
#pragma unroll
            for (int k = 0; k < PL::S; ++k) {
                if (!PL::chunk_bit_done_in_phase1(PL::b(k))) butterfly_pairs<NP>(v, 3 + k);
            }
        }

        // ---------------- row absmax ----------------
        // Two-phase plans end with chunks chunk_of(t, s, phase 2).  From n = 1024
        // on, slot bits 2, 3 are chunk bits C-2, C-1 and row-thread bits 0, 1 chunk
        // bits 2, 3, so a group of 128 elements (16 chunks) is four slots of each
        // of four threads, and a thread's outputs touch four groups (gmax[q], q =
        // slot bits 2, 3).  For n = 256, 512 a thread holds 16 consecutive chunks:
        // one group.
        constexpr bool kGroups4 = PL::kTwoPhase && C >= 7;
        const bool i8 = PL::kTwoPhase && (prm.flags & (RQ_INT8_CODES | RQ_INT4_BYTES)) != 0;
        const bool per_group = PL::kTwoPhase && (prm.flags & RQ_GROUP_SCALES) != 0;
        const bool e4 = PL::kTwoPhase && (prm.flags & RQ_E4M3_CODES) != 0;
        float gmax[kGroups4 ? 4 : 1];
        float amax;
        if constexpr (kGroups4) {
            static_assert(NP == 64, "16 slots of 4 pairs");
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                gmax[q4] = pairs_absmax<16>(*reinterpret_cast<const pair_t(*)[16]>(&v[16 * q4]));
            amax = fmaxf(fmaxf(gmax[0], gmax[1]), fmaxf(gmax[2], gmax[3]));
            if (per_group) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    gmax[q4] = fmaxf(gmax[q4], __shfl_xor_sync(full, gmax[q4], 1));
                    gmax[q4] = fmaxf(gmax[q4], __shfl_xor_sync(full, gmax[q4], 2));
                }
            }
        } else {
            amax = pairs_absmax<NP>(v);
            gmax[0] = amax;                                    // n = 256, 512: the thread's group
        }
        if constexpr (P > 1) {
#pragma unroll
            for (int k = 0; k < (PL::T < 5 ? PL::T : 5); ++k)
                amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1 << k));
        }
        if constexpr (P > 32) {
            // two warps per row: exchange through shared memory
            const int w = t >> 5;
            if ((t & 31) == 0) red[row_in_cta * 2 + w] = amax;
            asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            amax = fmaxf(red[row_in_cta * 2], red[row_in_cta * 2 + 1]);
        }

        // ---------------- quantize, pack, store ----------------
        // codes: INT4 per row (default), INT8 per row, or INT4 per group of 128
        // (the last two for two-phase plans only; the host rejects the others)
        const float qmax = (prm.flags & RQ_INT8_CODES) ? 127.0f : 7.0f;   // INT8, or INT4 (also in bytes)
        const float inv = amax > 0.f ? qmax / amax : 0.f;
        float ginv[kGroups4 ? 4 : 1];
#pragma unroll
        for (int q4 = 0; q4 < (kGroups4 ? 4 : 1); ++q4) ginv[q4] = per_group ? (gmax[q4] > 0.f ? 7.0f / gmax[q4] : 0.f) : inv;
        const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
        uint8_t *stg = ostage + (warp * 2 + obuf) * OSTG;
        if constexpr (!PL::kTwoPhase) {
            // the bulk store that last read this staging buffer must be done
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            __syncwarp();
        }
        if (active) {
            if (PL::kTwoPhase && per_group) {
                if constexpr (kGroups4) {
                    if ((t & 3) == 0) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            job.scales[row * (int64_t)(n / 128) + ((t >> 2) | ((q4 & 1) << (C - 6)) | ((q4 >> 1) << (C - 5)))] =
                                (gmax[q4] / 7.0f) * inv_sqrt_n;
                    }
                } else {
                    job.scales[row * (int64_t)(n / 128) + t] = (gmax[0] / 7.0f) * inv_sqrt_n;
                }
            } else if (t == 0) {
                job.scales[e4 ? 2 * row : row] = (amax / qmax) * inv_sqrt_n;   // E4M3: (scale, code sum) per row
            }
            uint8_t *qrow = PL::kTwoPhase ? job.q + row * (int64_t)(n / 2) : stg + (lane / P) * (n / 2);
            // output chunk of slot s: phase-2 map, or natural order for one row per thread
            auto out_chunk = [&](int s) { return PL::kTwoPhase ? chunk_of<C>(t, s, true) : (chunk_t<C>(t, false) | s); };
            // (-1)^popcount(s & xr): the sign left by the permuted read order
            auto out_neg = [&](int s) { return !PL::kTwoPhase && (__popc(s & xr) & 1); };
            // one branch per row for each option (signs after the transform, fp32 output)
            if (!signs_first) {
#pragma unroll
                for (int s = 0; s < NSLOT; ++s) {
                    const uint4 m = reinterpret_cast<const uint4 *>(sgn)[out_chunk(s)];
                    const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        v[4 * s + k] ^= ((pair_t)(mm[k] & 0x80000000u) << 32) | (pair_t)(mm[k] << 16);
                }
            }
            if (job.y) {
                float *yrow = job.y + row * (int64_t)n;
#pragma unroll
                for (int s = 0; s < NSLOT; ++s) {
                    const float ys = out_neg(s) ? -inv_sqrt_n : inv_sqrt_n;
                    const pair_t sc2 = mk2(ys, ys), z2 = 0ull;
                    ulonglong2 *yp = reinterpret_cast<ulonglong2 *>(yrow + 8 * out_chunk(s));
                    yp[0] = make_ulonglong2(fma2(v[4 * s], sc2, z2), fma2(v[4 * s + 1], sc2, z2));
                    yp[1] = make_ulonglong2(fma2(v[4 * s + 2], sc2, z2), fma2(v[4 * s + 3], sc2, z2));
                }
            }
            if (PL::kTwoPhase && i8) {
                // one byte per code (the low byte of the biased float is the
                // two's-complement code): chunks c0 .. c0 + 3 are 32 bytes
                const pair_t inv2 = mk2(inv, inv);
#pragma unroll
                for (int s4 = 0; s4 < NSLOT; s4 += 4) {
                    uint32_t words[8];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int s = s4 + cc;
                        uint32_t code[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const pair_t qq = fma2(v[4 * s + k], inv2, bias2);
                            code[2 * k] = (uint32_t)qq;
                            code[2 * k + 1] = (uint32_t)(qq >> 32);
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            words[2 * cc + h] = __byte_perm(__byte_perm(code[4 * h], code[4 * h + 1], 0x0040u),
                                                            __byte_perm(code[4 * h + 2], code[4 * h + 3], 0x0040u), 0x5410u);
                    }
                    uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)n + 8 * out_chunk(s4));
                    qp[0] = make_uint4(words[0], words[1], words[2], words[3]);
                    qp[1] = make_uint4(words[4], words[5], words[6], words[7]);
                }
            } else {
            int csum = 0;   // E4M3: this thread's part of the row's code sum
#pragma unroll
            for (int s4 = 0; s4 < NSLOT; s4 += 4) {
                uint32_t words[4];
                const int c0 = out_chunk(s4);
                // the row's multiplier, or (groups) that of the group of slots s4 .. s4 + 3
                const float ginv_s = ginv[kGroups4 ? (s4 >> 2) : 0];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int s = s4 + cc;
                    const float sinv = out_neg(s) ? -ginv_s : ginv_s;
                    const pair_t inv2 = mk2(sinv, sinv);
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * s + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
                    if (e4) {
                        // one signed E4M3 byte per code, in the product's operand
                        // order (even codes, then odd codes, of each chunk)
                        *reinterpret_cast<uint2 *>(job.q + row * (int64_t)n + 8 * (c0 + cc)) =
                            make_uint2(e4m3_word_sum(code[0], code[2], code[4], code[6], csum),
                                       e4m3_word_sum(code[1], code[3], code[5], code[7], csum));
                    } else {
                        words[cc] = pack8(code);
                    }
                }
                // chunks c0..c0+3 are consecutive (slot bits 0,1 = chunk bits 0,1)
                if (!e4) *reinterpret_cast<uint4 *>(qrow + 4 * c0) = make_uint4(words[0], words[1], words[2], words[3]);
            }
            if constexpr (PL::kTwoPhase && P <= 32) {
                if (e4) {
                    // the row's P threads are consecutive lanes, all active or all not
                    const unsigned rmask = (full >> (32 - P)) << (lane & ~(P - 1));
#pragma unroll
                    for (int k = 0; k < PL::T; ++k) csum += __shfl_xor_sync(rmask, csum, 1 << k);
                    if (t == 0) job.scales[2 * row + 1] = (float)csum;
                }
            }
            }
        }
        if constexpr (!PL::kTwoPhase) {
            // one bulk store of this warp's valid rows
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                const int64_t wrow0 = row;                      // lane 0 holds the warp's first row
                int64_t valid = job.rows - wrow0;
                valid = valid < 0 ? 0 : (valid > 32 / P ? 32 / P : valid);
                if (valid > 0 && !aborted) {
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                                     job.q + wrow0 * (int64_t)(n / 2)),
                                 "r"(smem_addr(stg)), "r"((uint32_t)(valid * (n / 2)))
                                 : "memory");
                }
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            obuf ^= 1;
        }
        if constexpr (P > 32) {
            // the two warps of a row leave together: share the abort decision
            if (aborted && (t & 31) == 0) red[row_in_cta * 2] = __int_as_float(-1);
            asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            const bool any = __float_as_int(red[row_in_cta * 2]) == -1;
            asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            if (any) { aborted = true; break; }
        } else {
            if constexpr (PL::kTwoPhase) __syncwarp();
            if (__any_sync(full, aborted)) { aborted = true; break; }
        }
    }
    if constexpr (!PL::kTwoPhase) {
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    if (aborted) {
        // wait (bounded) for this warp's copies still in flight before leaving
        for (int d = 0; d < DEPTH; ++d) {
            const uint32_t par = d >= slot ? phase : (phase ^ 1u);
            mbar_wait_bounded(&bars[warp * DEPTH + d], par, prm.err);
        }
    }
}

// --------------------------------------------------------------------------
// n = 4096: three butterfly phases with two transposes, 64 values per thread.
//
// The general plan above keeps 128 values per thread, which needs the whole
// register file (8 warps per SM) and leaves the kernel latency-bound.  For the
// activation size of the serving path this variant halves the per-thread state
// (two warps per row, 16 warps per SM) and replaces the shuffle stage by a
// second shared-memory transpose.  Chunk c = 8 elements, 9 chunk bits; a thread
// t (0..63; bit 5 = which warp of the row) holds 8 chunks (slot s = 3 bits):
//   phase 1: slots = chunk bits 3,4,5; t0,t1,t2 -> bits 0,1,2; t3,t4 -> 6,7; t5 -> 8
//            (8 lanes read 128 contiguous input bytes; element bits and slot
//            bits: 6 butterfly stages in registers)
//   phase 2: slots = chunk bits 6,7,8; t0..t5 -> bits 0..5 (3 stages)
//   phase 3: slots = chunk bits 0,1,2; t0..t5 -> bits 3..8 (3 stages): a thread
//            ends with 64 consecutive elements, i.e. 32 bytes of codes.
// Row buffer: fp32, 16-byte granule g = 2c + h (h = half chunk) XOR a swizzle of
// chunk bits that makes every quarter-warp access touch 8 different bank groups
// on both sides of each transpose:
//   transpose 1: granule bit 0 ^= c2
//   transpose 2: granule bits 0,1,2 ^= (c2 ^ c5, c3, c4)
// --------------------------------------------------------------------------
constexpr int K4_LOGN = 12, K4_N = 4096;

// Threads per CTA (two warps per row): at most 8 rows (4 for fp32 input, whose
// buffers are twice as large); small batches use 2-row CTAs so that they spread
// over more SMs (16 decode rows: 8 CTAs instead of 2).  Batches that need
// several rounds of 8-row CTAs take 7-row CTAs when that lowers the rows an SM
// handles in all (rounds x rows per CTA): 2048 rows on 152 SMs are 2 rounds
// either way, 14 rows per SM instead of 16 (15.7 -> 14.9 us, CUDA event means).
__host__ __device__ constexpr int k4_max_threads(int in_type) { return in_type == IN_F32 ? 256 : 512; }
inline int k4_pick_threads(int64_t rows, int in_type, int sms) {
    if (in_type != IN_F32 && rows > 8ll * sms) {
        const int64_t r8 = (rows + 8ll * sms - 1) / (8ll * sms) * 8, r7 = (rows + 7ll * sms - 1) / (7ll * sms) * 7;
        return r7 < r8 ? 448 : 512;
    }
    for (int t = k4_max_threads(in_type); t > 128; t /= 2)
        if ((rows + t / 64 - 1) / (t / 64) >= sms) return t;
    return 128;
}

template <int IN, int THREADS>
size_t k4_smem_bytes() {
    constexpr int NW = THREADS / 32, ROWS = THREADS / 64;
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    // barriers | sign words | absmax exchange | per-warp input halves | fp32 row buffers
    return 128 + (size_t)K4_N * 2 + 128 + (size_t)NW * (K4_N * ES / 2) + (size_t)ROWS * K4_N * 4;
}

template <int IN, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
fwht_quant_k4_kernel(const __grid_constant__ KParams prm) {
    constexpr int n = K4_N;
    constexpr int NW = THREADS / 32, ROWS = THREADS / 64;
    constexpr int G = IN == IN_F32 ? 2 : 1;              // 16-byte granules per input chunk
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    constexpr int HB = n * ES / 2;                        // input bytes of half a row (one warp)
    constexpr int NP = 32;                                // fp32 pairs per thread
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);                  // NW
    uint32_t *sgn = reinterpret_cast<uint32_t *>(smem_raw + 128);             // n/2 words
    float *red = reinterpret_cast<float *>(smem_raw + 128 + n * 2);          // ROWS*2
    unsigned char *inbuf = smem_raw + 128 + n * 2 + 128;                      // NW halves
    ulonglong2 *rowbuf = reinterpret_cast<ulonglong2 *>(inbuf + NW * HB);    // ROWS rows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_in_cta = warp >> 1;
    const int t = threadIdx.x & 63;
    const int half = t >> 5;
    const bool signs_first = (prm.flags & 1u) != 0;
    const uint32_t msel = signs_first ? 0xffffffffu : 0u;
    const unsigned full = 0xffffffffu;
    const int64_t total_groups = prm.groups_per_job * prm.njobs;
    unsigned char *wbuf = inbuf + warp * HB;
    ulonglong2 *buf = rowbuf + (size_t)row_in_cta * (n / 4);
    const uint32_t rbar = 1 + row_in_cta;                  // named barrier of the row's two warps
    // thread bases of every access (slot s adds a compile-time offset)
    const K4Addr ad = k4_addr(t);
    const uint4 *sg1 = reinterpret_cast<const uint4 *>(sgn) + ad.c1;         // mask of chunk1(t, s): sg1[8 s]
    const uint4 *sg3 = reinterpret_cast<const uint4 *>(sgn) + 8 * t;         // mask of chunk3(t, s): sg3[s]
    const unsigned char *xb = wbuf + 16 * G * (ad.c1 & 255);                 // input of chunk1(t, s): + 128 G s
    ulonglong2 *const bw1[2] = {buf + ad.w1, buf + (ad.w1 ^ 1)};             // transpose 1 write: [16 s]
    const ulonglong2 *const br1[2] = {buf + ad.r1, buf + (ad.r1 ^ 1)};       // transpose 1 read: [128 s]
    ulonglong2 *const bw2[2] = {buf + ad.w2, buf + (ad.w2 ^ 1)};             // transpose 2 write: [128 s]
    const ulonglong2 *const br2 = buf + 16 * t;                              // transpose 2 read: [k3 ^ m3]

    if (threadIdx.x < NW) mbar_init(&bars[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();    // barriers initialized before the warps issue their first copies

    // This warp's half of row (group g, row_in_cta): chunks with bit 8 = half.
    auto issue = [&](int64_t g) {
        const int jb = job_of(g, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (g - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;
        const bool valid = row < job.rows;
        mbar_expect_tx(&bars[warp], valid ? (uint32_t)HB : 0u);
        if (valid)
            bulk_copy(wbuf, static_cast<const char *>(job.x) + (row * job.ld) * ES + half * HB, HB, &bars[warp]);
    };
    if (lane == 0 && (int64_t)blockIdx.x < total_groups) issue(blockIdx.x);
    // Sign masks (computed while the first copies are in flight): word j covers
    // elements 2j (bit 15) and 2j+1 (bit 31).
    for (int j = threadIdx.x; j < n / 2; j += THREADS) {
        const uint32_t s0 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j) >> 63);
        const uint32_t s1 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j + 1) >> 63);
        sgn[j] = (s0 << 15) | (s1 << 31);
    }
    __syncthreads();

    const float inv_sqrt_n = 1.0f / 64.0f;
    uint32_t phase = 0;
    bool aborted = false;
    for (int64_t grp = blockIdx.x; grp < total_groups; grp += gridDim.x) {
        const int jb = job_of(grp, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (grp - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;

        pair_t v[NP];
        // ---------------- phase 1: input, signs, 6 stages ----------------
        // A copy that never lands raises the error word; the iteration then runs
        // on stale data with its stores disabled, so barriers stay matched.
        if (!mbar_wait_bounded(&bars[warp], phase, prm.err)) aborted = true;
        phase ^= 1u;
        const bool active = row < job.rows && !aborted;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint4 m = sg1[8 * s];
            uint4 g[G];
#pragma unroll
            for (int h = 0; h < G; ++h) g[h] = *reinterpret_cast<const uint4 *>(xb + 128 * G * s + 16 * h);
            convert_chunk<IN>(g, m, msel, &v[4 * s]);   // includes the in-pair stage
        }
        // hand the input half back to the copy engine (generic reads before the
        // next bulk write) and fetch this warp's half of its next row
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && !aborted && grp + gridDim.x < total_groups) issue(grp + gridDim.x);
#pragma unroll
        for (int rb = 1; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- transpose 1, phase 2 ----------------
        // the row's other warp may still be reading the previous row's phase 3
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            bw1[0][16 * s] = make_ulonglong2(v[4 * s], v[4 * s + 1]);
            bw1[1][16 * s] = make_ulonglong2(v[4 * s + 2], v[4 * s + 3]);
        }
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const ulonglong2 lo = br1[0][128 * s], hi = br1[1][128 * s];
            v[4 * s] = lo.x; v[4 * s + 1] = lo.y; v[4 * s + 2] = hi.x; v[4 * s + 3] = hi.y;
        }
#pragma unroll
        for (int rb = 3; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- transpose 2, phase 3 ----------------
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            bw2[0][128 * s] = make_ulonglong2(v[4 * s], v[4 * s + 1]);
            bw2[1][128 * s] = make_ulonglong2(v[4 * s + 2], v[4 * s + 3]);
        }
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const ulonglong2 lo = br2[k4_k3(s, 0) ^ ad.m3], hi = br2[k4_k3(s, 1) ^ ad.m3];
            v[4 * s] = lo.x; v[4 * s + 1] = lo.y; v[4 * s + 2] = hi.x; v[4 * s + 3] = hi.y;
        }
#pragma unroll
        for (int rb = 3; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- row absmax (two warps) ----------------
        float amax = pairs_absmax<NP>(v);
        // a group of 128 elements (per-group scales) is the 64 of threads t and t ^ 1
        const float amax_grp = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
#pragma unroll
        for (int k = 0; k < 5; ++k) amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1 << k));
        if (lane == 0) red[row_in_cta * 2 + half] = aborted ? __int_as_float(-1) : amax;
        // E4M3: the row's code sum is added up in global memory by its warps
        if ((prm.flags & RQ_E4M3_CODES) && active && t == 0) job.scales[2 * row + 1] = 0.f;
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
        const float r0 = red[row_in_cta * 2], r1 = red[row_in_cta * 2 + 1];
        // the two warps of a row leave together: share the abort decision
        const bool any_abort = __float_as_int(r0) == -1 || __float_as_int(r1) == -1;
        amax = fmaxf(r0, r1);
        if (any_abort) { aborted = true; break; }

        // ---------------- quantize, pack, store: 64 consecutive elements ----------------
        if (active) {
            // codes: INT4 per row (default), INT8 per row, or INT4 per group of 128
            const bool i8 = (prm.flags & (RQ_INT8_CODES | RQ_INT4_BYTES)) != 0, grp = (prm.flags & RQ_GROUP_SCALES) != 0;
            const bool e4 = (prm.flags & RQ_E4M3_CODES) != 0;
            const float am = grp ? amax_grp : amax;
            const float qmax = (prm.flags & RQ_INT8_CODES) ? 127.0f : 7.0f;   // INT8, or INT4 (also in bytes)
            const float inv = am > 0.f ? qmax / am : 0.f;
            const pair_t inv2 = mk2(inv, inv);
            const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
            if (grp) {
                if ((t & 1) == 0) job.scales[row * (int64_t)(n / 128) + (t >> 1)] = (am / 7.0f) * inv_sqrt_n;
            } else if (t == 0) {
                job.scales[e4 ? 2 * row : row] = (am / qmax) * inv_sqrt_n;   // E4M3: (scale, code sum) per row
            }
            // the thread's 64 consecutive elements are chunks 8t + s; one branch per
            // row for each option (signs after the transform, fp32 output)
            if (!signs_first) {
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint4 m = sg3[s];
                    const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        v[4 * s + k] ^= ((pair_t)(mm[k] & 0x80000000u) << 32) | (pair_t)(mm[k] << 16);
                }
            }
            if (job.y) {
                const pair_t sc2 = mk2(inv_sqrt_n, inv_sqrt_n), z2 = 0ull;
                ulonglong2 *yp = reinterpret_cast<ulonglong2 *>(job.y + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    yp[2 * s] = make_ulonglong2(fma2(v[4 * s], sc2, z2), fma2(v[4 * s + 1], sc2, z2));
                    yp[2 * s + 1] = make_ulonglong2(fma2(v[4 * s + 2], sc2, z2), fma2(v[4 * s + 3], sc2, z2));
                }
            }
            if (i8) {
                // one byte per code (the low byte of the biased float is the
                // two's-complement code): 64 bytes, four 16-byte stores
                uint32_t words[16];
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * s + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        words[2 * s + h] = __byte_perm(__byte_perm(code[4 * h], code[4 * h + 1], 0x0040u),
                                                       __byte_perm(code[4 * h + 2], code[4 * h + 3], 0x0040u), 0x5410u);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    qp[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
            } else if (e4) {
                // one signed E4M3 byte per code, in the product's operand order
                // (even codes, then odd codes, of each chunk): 64 bytes
                uint32_t words[16];
                int csum = 0;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * s + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
                    words[2 * s] = e4m3_word_sum(code[0], code[2], code[4], code[6], csum);
                    words[2 * s + 1] = e4m3_word_sum(code[1], code[3], code[5], code[7], csum);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    qp[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
                // the warp's part of the code sum (the slot was zeroed before the barrier)
                csum = __reduce_add_sync(full, csum);
                if (lane == 0) atomicAdd(&job.scales[2 * row + 1], (float)csum);
            } else {
                uint32_t words[8];
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * s + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
                    words[s] = pack8(code);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)(n / 2) + 32 * t);
                qp[0] = make_uint4(words[0], words[1], words[2], words[3]);
                qp[1] = make_uint4(words[4], words[5], words[6], words[7]);
            }
        }
    }
    if (aborted) {
        // wait (bounded) for this warp's copy still in flight before leaving
        mbar_wait_bounded(&bars[warp], phase, prm.err);
    }
}

template <int IN, int THREADS>
cudaError_t launch_k4_t(const KParams &p, cudaStream_t stream) {
    auto kern = fwht_quant_k4_kernel<IN, THREADS>;
    const size_t smem = k4_smem_bytes<IN, THREADS>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t total = p.groups_per_job * p.njobs;
    int64_t grid = sms;                                   // one CTA per SM
    if (grid > total) grid = total;
    kern<<<(unsigned)grid, THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int IN>
cudaError_t launch_k4(const KParams &p, int threads, cudaStream_t stream) {
    switch (threads) {
        case 128: return launch_k4_t<IN, 128>(p, stream);
        case 256: return launch_k4_t<IN, 256>(p, stream);
        case 448:
            if constexpr (k4_max_threads(IN) >= 512) return launch_k4_t<IN, 448>(p, stream);
            return cudaErrorInvalidValue;
        default:
            if constexpr (k4_max_threads(IN) >= 512) return launch_k4_t<IN, 512>(p, stream);
            return cudaErrorInvalidValue;
    }
}

// --------------------------------------------------------------------------
// n = 8192: three butterfly phases with two transposes, 64 values per thread,
// four warps per row.  Element i = 8c + e (chunk c, 10 bits) = 4q + e' (quad q,
// 11 bits); thread t = 0..127 of a row is lane + 32 wr:
//   phase 1: chunk slots s = chunk bits 3,4,5 (8 chunks); lane bits 0..2 ->
//            chunk bits 0..2, lane bits 3,4 -> 6,7, wr -> 8,9, so each warp
//            copies and reads a contiguous quarter row (eight lanes read 128
//            contiguous bytes); stages on element bits 0,1,2 and 6,7,8;
//   phase 2: quad slots = quad bits 7..10 (16 quads); lane -> quad bits 0..4,
//            wr -> 5,6; stages on element bits 9..12;
//   phase 3: quad slots = quad bits 0..3; t -> quad bits 4..10; stages on
//            element bits 3,4,5, and the thread ends with 64 consecutive
//            elements (its 64 codes are 32 or 64 contiguous bytes).
// Stage order 0,1,2,6,7,8,9,10,11,12,3,4,5 (the fused decode kernel runs the
// same order for K = 8192, so its codes are these bit for bit).
// Row buffer: fp32 quads in 16-byte granules.  The first transpose keeps quad q
// at q ^ q3 (quad bit 3 into bit 0), the second at q ^ (q4, q5, q6) (bits 0..2):
// every 8-lane phase of both sides of both transposes then touches 8 distinct
// bank groups, and every access but the last transpose's reads is a thread base
// plus a compile-time offset (checked exhaustively on the host for all t, s).
// --------------------------------------------------------------------------
// One fp32 pair from shared memory.  The transposes read their granules as two of
// these (volatile, so they are issued where written): measured 41.2 -> 40.0 us (ncu)
// against 128-bit loads into pairs for 4096 x 8192 rows.
__device__ __forceinline__ pair_t lds64v(const void *p) {
    pair_t r;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(r) : "r"(smem_addr(p)));
    return r;
}
constexpr int K8_LOGN = 13, K8_N = 8192;

__host__ __device__ constexpr int k8_max_rows(int in_type) { return in_type == IN_F32 ? 2 : 4; }
// Rows per CTA: the most that fit, or fewer for small batches so that they
// spread over more SMs (16 decode rows: 16 CTAs instead of 4).
inline int k8_pick_rows(int64_t rows, int in_type, int sms) {
    for (int r = k8_max_rows(in_type); r > 1; r /= 2)
        if ((rows + r - 1) / r >= sms) return r;
    return 1;
}

template <int IN, int ROWS>
size_t k8_smem_bytes() {
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    // barriers | sign words | absmax exchange | per-warp input quarters | fp32 row buffers
    return 128 + (size_t)K8_N * 2 + 128 + (size_t)(4 * ROWS) * (K8_N * ES / 4) + (size_t)ROWS * K8_N * 4;
}

template <int IN, int ROWS>
__global__ void __launch_bounds__(128 * ROWS, 1)
fwht_quant_k8_kernel(const __grid_constant__ KParams prm) {
    constexpr int n = K8_N;
    constexpr int THREADS = 128 * ROWS, NW = THREADS / 32;
    constexpr int G = IN == IN_F32 ? 2 : 1;              // 16-byte granules per input chunk
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    constexpr int QB = n * ES / 4;                        // input bytes of a quarter row (one warp)
    constexpr int NP = 32;                                // fp32 pairs per thread
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);                  // NW
    uint32_t *sgn = reinterpret_cast<uint32_t *>(smem_raw + 128);             // n/2 words
    float *red = reinterpret_cast<float *>(smem_raw + 128 + n * 2);          // ROWS*4
    unsigned char *inbuf = smem_raw + 128 + n * 2 + 128;                      // NW quarters
    ulonglong2 *rowbuf = reinterpret_cast<ulonglong2 *>(inbuf + NW * QB);    // ROWS rows

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_in_cta = warp >> 2;
    const int t = threadIdx.x & 127;
    const int wr = t >> 5;
    const bool signs_first = (prm.flags & 1u) != 0;
    const uint32_t msel = signs_first ? 0xffffffffu : 0u;
    const unsigned full = 0xffffffffu;
    const int64_t total_groups = prm.groups_per_job * prm.njobs;
    unsigned char *wbuf = inbuf + warp * QB;
    ulonglong2 *buf = rowbuf + (size_t)row_in_cta * (n / 4);
    const uint32_t rbar = 1 + row_in_cta;                  // named barrier of the row's four warps
    // thread bases of every access (slot s adds a compile-time offset)
    const int c1 = (lane & 7) | ((lane >> 3) << 6) | (wr << 8);                 // phase-1 chunk of slot s: c1 + 8 s
    const uint4 *sg1 = reinterpret_cast<const uint4 *>(sgn) + c1;               // its sign words: sg1[8 s]
    const uint4 *sg3 = reinterpret_cast<const uint4 *>(sgn) + 8 * t;            // output chunk 8 t + c: sg3[c]
    const unsigned char *xb = wbuf + 16 * G * (c1 & 255);                       // its input: + 128 G s
    const int w1 = (2 * c1) ^ ((c1 >> 2) & 1);
    ulonglong2 *const bw1[2] = {buf + w1, buf + (w1 ^ 1)};                      // quad 2 chunk + h: bw1[h][16 s]
    const int q2 = lane | (wr << 5);                                            // phase-2 quad of slot s: q2 + 128 s
    const ulonglong2 *const br1 = buf + (q2 ^ ((q2 >> 3) & 1));                 // [128 s]
    ulonglong2 *const bw2 = buf + (q2 ^ ((q2 >> 4) & 7));                       // [128 s]
    const ulonglong2 *const br2 = buf + 16 * t;                                 // quad 16 t + s: [s ^ m3]
    const int m3 = t & 7;

    if (threadIdx.x < NW) mbar_init(&bars[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();    // barriers initialized before the warps issue their first copies

    // This warp's quarter of row (group g, row_in_cta): chunks with bits 8,9 = wr.
    auto issue = [&](int64_t g) {
        const int jb = job_of(g, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (g - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;
        const bool valid = row < job.rows;
        mbar_expect_tx(&bars[warp], valid ? (uint32_t)QB : 0u);
        if (valid)
            bulk_copy(wbuf, static_cast<const char *>(job.x) + (row * job.ld) * ES + wr * QB, QB, &bars[warp]);
    };
    if (lane == 0 && (int64_t)blockIdx.x < total_groups) issue(blockIdx.x);
    // Sign masks (computed while the first copies are in flight): word j covers
    // elements 2j (bit 15) and 2j+1 (bit 31).
    for (int j = threadIdx.x; j < n / 2; j += THREADS) {
        const uint32_t s0 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j) >> 63);
        const uint32_t s1 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j + 1) >> 63);
        sgn[j] = (s0 << 15) | (s1 << 31);
    }
    __syncthreads();

    const float inv_sqrt_n = 0.70710678118654752440f / 64.0f;
    uint32_t phase = 0;
    bool aborted = false;
    for (int64_t grp = blockIdx.x; grp < total_groups; grp += gridDim.x) {
        const int jb = job_of(grp, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (grp - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;

        pair_t v[NP];
        // ---------------- phase 1: input, signs, 6 stages ----------------
        // A copy that never lands raises the error word; the iteration then runs
        // on stale data with its stores disabled, so barriers stay matched.
        if (!mbar_wait_bounded(&bars[warp], phase, prm.err)) aborted = true;
        phase ^= 1u;
        const bool active = row < job.rows && !aborted;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint4 m = sg1[8 * s];
            uint4 g[G];
#pragma unroll
            for (int h = 0; h < G; ++h) g[h] = *reinterpret_cast<const uint4 *>(xb + 128 * G * s + 16 * h);
            convert_chunk<IN>(g, m, msel, &v[4 * s]);   // includes the in-pair stage
        }
        // hand the quarter back to the copy engine (generic reads before the
        // next bulk write) and fetch this warp's quarter of its next row
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0 && !aborted && grp + gridDim.x < total_groups) issue(grp + gridDim.x);
#pragma unroll
        for (int rb = 1; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- transpose 1, phase 2 ----------------
        // (the previous row's last reads of the buffer came before its absmax barrier)
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            bw1[0][16 * s] = make_ulonglong2(v[4 * s], v[4 * s + 1]);
            bw1[1][16 * s] = make_ulonglong2(v[4 * s + 2], v[4 * s + 3]);
        }
        asm volatile("bar.sync %0, 128;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            v[2 * s] = lds64v(br1 + 128 * s);
            v[2 * s + 1] = lds64v(reinterpret_cast<const pair_t *>(br1 + 128 * s) + 1);
        }
#pragma unroll
        for (int rb = 2; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- transpose 2, phase 3 ----------------
        asm volatile("bar.sync %0, 128;" ::"r"(rbar) : "memory");   // every thread has read transpose 1
#pragma unroll
        for (int s = 0; s < 16; ++s) bw2[128 * s] = make_ulonglong2(v[2 * s], v[2 * s + 1]);
        asm volatile("bar.sync %0, 128;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            v[2 * s] = lds64v(br2 + (s ^ m3));
            v[2 * s + 1] = lds64v(reinterpret_cast<const pair_t *>(br2 + (s ^ m3)) + 1);
        }
#pragma unroll
        for (int rb = 3; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);

        // ---------------- row absmax (four warps) ----------------
        float amax = pairs_absmax<NP>(v);
        // a group of 128 elements (per-group scales) is the 64 of threads t and t ^ 1
        const float amax_grp = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
#pragma unroll
        for (int k = 0; k < 5; ++k) amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1 << k));
        if (lane == 0) red[row_in_cta * 4 + wr] = aborted ? __int_as_float(-1) : amax;
        // E4M3: the row's code sum is added up in global memory by its warps
        if ((prm.flags & RQ_E4M3_CODES) && active && t == 0) job.scales[2 * row + 1] = 0.f;
        asm volatile("bar.sync %0, 128;" ::"r"(rbar) : "memory");
        const float4 r4 = reinterpret_cast<const float4 *>(red)[row_in_cta];
        // the four warps of a row leave together: share the abort decision
        const bool any_abort = __float_as_int(r4.x) == -1 || __float_as_int(r4.y) == -1 ||
                               __float_as_int(r4.z) == -1 || __float_as_int(r4.w) == -1;
        amax = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
        if (any_abort) { aborted = true; break; }

        // ---------------- quantize, pack, store: 64 consecutive elements ----------------
        if (active) {
            // codes: INT4 per row (default), INT8 per row, or INT4 per group of 128
            const bool i8 = (prm.flags & (RQ_INT8_CODES | RQ_INT4_BYTES)) != 0, grp = (prm.flags & RQ_GROUP_SCALES) != 0;
            const bool e4 = (prm.flags & RQ_E4M3_CODES) != 0;
            const float am = grp ? amax_grp : amax;
            const float qmax = (prm.flags & RQ_INT8_CODES) ? 127.0f : 7.0f;   // INT8, or INT4 (also in bytes)
            const float inv = am > 0.f ? qmax / am : 0.f;
            const pair_t inv2 = mk2(inv, inv);
            const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
            if (grp) {
                if ((t & 1) == 0) job.scales[row * (int64_t)(n / 128) + (t >> 1)] = (am / 7.0f) * inv_sqrt_n;
            } else if (t == 0) {
                job.scales[e4 ? 2 * row : row] = (am / qmax) * inv_sqrt_n;   // E4M3: (scale, code sum) per row
            }
            // the thread's 64 consecutive elements are chunks 8t + c (pairs 4c .. 4c+3);
            // one branch per row for each option (signs after the transform, fp32 output)
            if (!signs_first) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 m = sg3[c];
                    const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        v[4 * c + k] ^= ((pair_t)(mm[k] & 0x80000000u) << 32) | (pair_t)(mm[k] << 16);
                }
            }
            if (job.y) {
                const pair_t sc2 = mk2(inv_sqrt_n, inv_sqrt_n), z2 = 0ull;
                ulonglong2 *yp = reinterpret_cast<ulonglong2 *>(job.y + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int c = 0; c < 16; ++c) yp[c] = make_ulonglong2(fma2(v[2 * c], sc2, z2), fma2(v[2 * c + 1], sc2, z2));
            }
            if (i8) {
                // one byte per code (the low byte of the biased float is the
                // two's-complement code): 64 bytes, four 16-byte stores
                uint32_t words[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * c + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        words[2 * c + h] = __byte_perm(__byte_perm(code[4 * h], code[4 * h + 1], 0x0040u),
                                                       __byte_perm(code[4 * h + 2], code[4 * h + 3], 0x0040u), 0x5410u);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    qp[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
            } else if (e4) {
                // one signed E4M3 byte per code, in the product's operand order
                // (even codes, then odd codes, of each chunk): 64 bytes
                uint32_t words[16];
                int csum = 0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * c + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
                    words[2 * c] = e4m3_word_sum(code[0], code[2], code[4], code[6], csum);
                    words[2 * c + 1] = e4m3_word_sum(code[1], code[3], code[5], code[7], csum);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)n + 64 * t);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    qp[c] = make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
                // the warp's part of the code sum (the slot was zeroed before the barrier)
                csum = __reduce_add_sync(full, csum);
                if (lane == 0) atomicAdd(&job.scales[2 * row + 1], (float)csum);
            } else {
                uint32_t words[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t code[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const pair_t qq = fma2(v[4 * c + k], inv2, bias2);
                        code[2 * k] = (uint32_t)qq;
                        code[2 * k + 1] = (uint32_t)(qq >> 32);
                    }
                    words[c] = pack8(code);
                }
                uint4 *qp = reinterpret_cast<uint4 *>(job.q + row * (int64_t)(n / 2) + 32 * t);
                qp[0] = make_uint4(words[0], words[1], words[2], words[3]);
                qp[1] = make_uint4(words[4], words[5], words[6], words[7]);
            }
        }
    }
    if (aborted) {
        // wait (bounded) for this warp's copy still in flight before leaving
        mbar_wait_bounded(&bars[warp], phase, prm.err);
    }
}

template <int IN, int ROWS>
cudaError_t launch_k8_t(const KParams &p, cudaStream_t stream) {
    auto kern = fwht_quant_k8_kernel<IN, ROWS>;
    const size_t smem = k8_smem_bytes<IN, ROWS>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128 * ROWS, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t total = p.groups_per_job * p.njobs;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > total) grid = total;
    kern<<<(unsigned)grid, 128 * ROWS, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int IN>
cudaError_t launch_k8(const KParams &p, int rows, cudaStream_t stream) {
    switch (rows) {
        case 1: return launch_k8_t<IN, 1>(p, stream);
        case 2: return launch_k8_t<IN, 2>(p, stream);
        default:
            if constexpr (k8_max_rows(IN) >= 4) return launch_k8_t<IN, 4>(p, stream);
            return cudaErrorInvalidValue;
    }
}

// --------------------------------------------------------------------------
// n = 128 (one head of K or V, head_dim 128): a warp pair per 32 rows.
//
// Lane l of the pair's warp h holds half h of row l (64 values as fp32 pairs):
// chunk slots s = element bits 3..5, read in the order s ^ (l & 7) so that the
// eight lanes of a shared-memory phase read eight different 16-byte columns of
// their rows (a Sylvester network on XOR-permuted input leaves output j in
// place times (-1)^popcount(j & a), folded into the quantization multiplier).
// Six stages run in registers; the seventh (element bit 6, across the halves)
// goes through shared memory: warp 0 keeps output chunks 0..3 and warp 1 chunks
// 4..7, each hands the other half of its values to its partner lane (16 pairs,
// 64-bit stores, conflict-free) and forms y = A +- B for the chunks it keeps, i.e.
// two runs of 32 consecutive outputs: 16 bytes of codes each.  Warp 1 runs its
// last register stage (slot bit 2) with sum and difference swapped (the same
// fused multiply-adds with the sign of b flipped), so in both warps registers
// 0..15 hold the kept chunks and 16..31 the ones handed over: the two warps run
// the same instructions, and warp 1's A - B comes out as B - A, a sign folded
// into its multiplier like the read-order signs.  One named barrier per
// pair orders the exchange (and frees the input slot for the next copy), a second
// one the row-maximum exchange.  Compared with two lanes per row and a shuffle
// stage this saves the shuffles' 1.5 instructions per element and most of the
// per-group control, at 16 warps per SM (8 one-pair CTAs).
// --------------------------------------------------------------------------
// One warp pair per CTA; the launch bound of 9 CTAs per SM caps registers at 112
// (96 used, no spills), and shared memory admits 8 (16 warps).  Against two pairs
// per CTA at 128 registers: 37.6 -> 36.9 us median (K, V 8192 x 32 x 128).
constexpr int KV_PAIRS = 1;    // warp pairs per CTA
constexpr int KV_DEPTH = 2;    // input groups in flight per pair

template <int IN>
constexpr int kv_pair_bytes() {
    // input ring (32 rows per group) | exchange [2][16][32] pairs | row maxima [2][32]
    return KV_DEPTH * 32 * 128 * (IN == IN_F32 ? 4 : 2) + 2 * 16 * 32 * 8 + 2 * 32 * 4;
}
template <int IN>
size_t kv_smem_bytes() {
    return 256 + (size_t)KV_PAIRS * kv_pair_bytes<IN>() + 128 + 256;   // alignment | pairs | barriers | sign words
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
    return r;
}

template <int IN>
__global__ void __launch_bounds__(64 * KV_PAIRS, 9)
fwht_quant_kv128_kernel(const __grid_constant__ KParams prm) {
    constexpr int n = 128, G = IN == IN_F32 ? 2 : 1, ES = IN == IN_F32 ? 4 : 2, RB = n * ES;
    constexpr int NP = 32;                                 // fp32 pairs per thread
    constexpr int PB = kv_pair_bytes<IN>();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 256-byte aligned base: the XOR addressing below needs the chunk-offset bits
    // (4..6, or 5..7 for fp32 rows) of the input rows and the sign table free.
    // Each pair's block is a multiple of 256 bytes.
    static_assert(PB % 256 == 0, "pair blocks keep 256-byte alignment");
    unsigned char *base = smem_raw + ((256u - (smem_addr(smem_raw) & 255u)) & 255u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + KV_PAIRS * PB);      // KV_PAIRS * KV_DEPTH
    uint32_t *sgn = reinterpret_cast<uint32_t *>(base + KV_PAIRS * PB + 128); // 64 words

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp >> 1, h = warp & 1;
    const int a = lane & 7;
    unsigned char *pbase = base + pair * PB;
    unsigned char *ring = pbase;
    pair_t *xch = reinterpret_cast<pair_t *>(pbase + KV_DEPTH * 32 * RB);
    float *amx = reinterpret_cast<float *>(pbase + KV_DEPTH * 32 * RB + 2 * 16 * 32 * 8);
    const uint32_t pbar = 1 + pair;                        // named barrier of the pair (64 threads)
    const bool signs_first = (prm.flags & 1u) != 0;
    const uint32_t msel = signs_first ? 0xffffffffu : 0u;
    const int64_t total_groups = prm.groups_per_job * prm.njobs;
    const int64_t first = (int64_t)blockIdx.x * KV_PAIRS + pair, step = (int64_t)gridDim.x * KV_PAIRS;
    const float inv_sqrt_n = 0.70710678118654752440f / 8.0f;
    // sign of the value in register chunk c of run r against y: (-1)^popcount(s & a)
    // for the butterfly slot s = 4 h + c, and for warp 1's second run (B - A) -1
    float fsg[2][4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        fsg[0][c] = (__popc(((h << 2) | c) & a) & 1) ? -1.f : 1.f;
        fsg[1][c] = h ? -fsg[0][c] : fsg[0][c];
    }
    const float sig = h ? -1.f : 1.f;                      // warp 1: the last stage swapped

    if (threadIdx.x < KV_PAIRS * KV_DEPTH) mbar_init(&bars[threadIdx.x], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    // The 32 rows of group g into ring slot `slot` (one lane of the pair's warp 0).
    auto issue = [&](int64_t g, int slot) {
        const int jb = job_of(g, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row0 = (g - (int64_t)jb * prm.groups_per_job) * 32;
        int64_t valid = job.rows - row0;
        valid = valid < 0 ? 0 : (valid > 32 ? 32 : valid);
        uint64_t *bar = &bars[pair * KV_DEPTH + slot];
        unsigned char *dst = ring + slot * 32 * RB;
        const char *x = static_cast<const char *>(job.x);
        mbar_expect_tx(bar, (uint32_t)(valid * RB));
        if (job.ld * ES == RB) {
            if (valid > 0) bulk_copy(dst, x + row0 * RB, (uint32_t)(valid * RB), bar);
        } else {
            for (int r = 0; r < valid; ++r) bulk_copy(dst + r * RB, x + (row0 + r) * job.ld * ES, RB, bar);
        }
    };
    if (h == 0 && lane == 0) {
#pragma unroll
        for (int d = 0; d < KV_DEPTH; ++d)
            if (first + d * step < total_groups) issue(first + d * step, d);
    }
    if (threadIdx.x < n / 2) {
        const uint32_t s0 = (uint32_t)(splitmix64_at(prm.seed, 2ull * threadIdx.x) >> 63);
        const uint32_t s1 = (uint32_t)(splitmix64_at(prm.seed, 2ull * threadIdx.x + 1) >> 63);
        sgn[threadIdx.x] = (s0 << 15) | (s1 << 31);
    }
    __syncthreads();

    // shared addresses with the lane's XOR order in bits 4..6 (chunk c ^ s is at base ^ 16 G s)
    const uint32_t sg_in = smem_addr(sgn) + 128u * (uint32_t)h + 16u * (uint32_t)a;   // input-side masks
    const uint32_t ring_lane = smem_addr(ring) + (uint32_t)(lane * RB + h * (RB / 2)) + 16u * G * (uint32_t)a;
    pair_t *give = xch + h * 512 + lane;                   // [k]: stride 32 pairs
    const pair_t *take = xch + (h ^ 1) * 512 + lane;
    const uint4 *sg_out = reinterpret_cast<const uint4 *>(sgn);

    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    for (int64_t grp = first; grp < total_groups; grp += step) {
        const int jb = job_of(grp, prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (grp - (int64_t)jb * prm.groups_per_job) * 32 + lane;
        if (!mbar_wait_bounded(&bars[pair * KV_DEPTH + slot], phase, prm.err)) aborted = true;
        const bool active = row < job.rows && !aborted;

        pair_t v[NP];
        const uint32_t rl = ring_lane + (uint32_t)(slot * 32 * RB);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint4 m = lds128(sg_in ^ (16u * s));
            uint4 g[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) g[hh] = lds128((rl ^ (16u * G * s)) + 16u * hh);
            convert_chunk<IN>(g, m, msel, &v[4 * s]);       // includes the in-pair stage
        }
#pragma unroll
        for (int rb = 1; rb <= 4; ++rb) butterfly_pairs<NP>(v, rb);
        {
            // slot bit 2: (a + sig b, a - sig b), i.e. swapped in warp 1
            const pair_t sp = mk2(sig, sig), sn = mk2(-sig, -sig);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const pair_t x = v[k], y = v[16 + k];
                v[k] = fma2(y, sp, x);
                v[16 + k] = fma2(y, sn, x);
            }
        }
        // hand the partner the chunks it keeps
#pragma unroll
        for (int k = 0; k < 16; ++k) give[32 * k] = v[16 + k];
        // the input slot's generic reads, ordered before its next bulk write
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync %0, 64;" ::"r"(pbar) : "memory");
        if (h == 0 && lane == 0 && !aborted && grp + KV_DEPTH * step < total_groups) issue(grp + KV_DEPTH * step, slot);
        if (++slot == KV_DEPTH) {
            slot = 0;
            phase ^= 1u;
        }
        // y = A +- B for the kept chunks: two runs of 32 outputs in v[0..15], v[16..31]
        // (warp 1: own - received = B - A for the second run)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const pair_t o = take[32 * k];
            const pair_t s_ = add2(v[k], o), d_ = sub2(v[k], o);
            v[k] = s_; v[16 + k] = d_;
        }
        float amax = pairs_absmax<NP>(v);
        amx[h * 32 + lane] = aborted ? __int_as_float(-1) : amax;
        // E4M3: the row's code sum is added up in global memory by its two threads
        if ((prm.flags & RQ_E4M3_CODES) && active && h == 0) job.scales[2 * row + 1] = 0.f;
        asm volatile("bar.sync %0, 64;" ::"r"(pbar) : "memory");
        const float m0 = amx[lane], m1 = amx[32 + lane];
        // the two warps of the pair leave together: share the abort decision
        const bool any_abort = __any_sync(0xffffffffu, __float_as_int(m0) == -1 || __float_as_int(m1) == -1);
        if (any_abort) { aborted = true; break; }
        amax = fmaxf(m0, m1);

        if (active) {
            // codes: INT4 packed (default; with RQ_GROUP_SCALES the one group of 128 is
            // the row), INT8 or INT4 one per byte, or the product's E4M3 operand bytes
            const uint32_t fl = prm.flags;
            const bool bytes = (fl & (RQ_INT8_CODES | RQ_INT4_BYTES)) != 0, e4 = (fl & RQ_E4M3_CODES) != 0;
            const float qmax = (fl & RQ_INT8_CODES) ? 127.0f : 7.0f;
            const float inv = amax > 0.f ? qmax / amax : 0.f;
            if (h == 0) job.scales[e4 ? 2 * row : row] = (amax / qmax) * inv_sqrt_n;   // E4M3: (scale, code sum)
            // output chunk of run r, chunk c: 8 r + 4 h + c
            if (!signs_first) {
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 m = sg_out[8 * r + 4 * h + c];
                        const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            v[16 * r + 4 * c + k] ^= ((pair_t)(mm[k] & 0x80000000u) << 32) | (pair_t)(mm[k] << 16);
                    }
            }
            if (job.y) {
                float *yrow = job.y + row * (int64_t)n;
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float ys = fsg[r][c] * inv_sqrt_n;
                        const pair_t sc2 = mk2(ys, ys), z2 = 0ull;
                        ulonglong2 *yp = reinterpret_cast<ulonglong2 *>(yrow + 8 * (8 * r + 4 * h + c));
                        yp[0] = make_ulonglong2(fma2(v[16 * r + 4 * c], sc2, z2), fma2(v[16 * r + 4 * c + 1], sc2, z2));
                        yp[1] = make_ulonglong2(fma2(v[16 * r + 4 * c + 2], sc2, z2), fma2(v[16 * r + 4 * c + 3], sc2, z2));
                    }
            }
            const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
            if (!bytes && !e4) {
                uint8_t *qrow = job.q + row * (int64_t)(n / 2);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    uint32_t words[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float sv = fsg[r][c] * inv;
                        const pair_t inv2 = mk2(sv, sv);
                        uint32_t code[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const pair_t qq = fma2(v[16 * r + 4 * c + k], inv2, bias2);
                            code[2 * k] = (uint32_t)qq;
                            code[2 * k + 1] = (uint32_t)(qq >> 32);
                        }
                        words[c] = pack8(code);
                    }
                    *reinterpret_cast<uint4 *>(qrow + 32 * r + 16 * h) = make_uint4(words[0], words[1], words[2], words[3]);
                }
            } else {
                // one byte per code: run r is 32 bytes at 64 r + 32 h
                uint8_t *qrow = job.q + row * (int64_t)n;
                int csum = 0;
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    uint32_t words[8];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float sv = fsg[r][c] * inv;
                        const pair_t inv2 = mk2(sv, sv);
                        uint32_t code[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const pair_t qq = fma2(v[16 * r + 4 * c + k], inv2, bias2);
                            code[2 * k] = (uint32_t)qq;
                            code[2 * k + 1] = (uint32_t)(qq >> 32);
                        }
                        if (e4) {
                            // signed E4M3 bytes, even codes then odd codes of the chunk
                            words[2 * c] = e4m3_word_sum(code[0], code[2], code[4], code[6], csum);
                            words[2 * c + 1] = e4m3_word_sum(code[1], code[3], code[5], code[7], csum);
                        } else {
                            // two's-complement bytes in element order
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                words[2 * c + hh] = __byte_perm(__byte_perm(code[4 * hh], code[4 * hh + 1], 0x0040u),
                                                                __byte_perm(code[4 * hh + 2], code[4 * hh + 3], 0x0040u), 0x5410u);
                        }
                    }
                    uint4 *qp = reinterpret_cast<uint4 *>(qrow + 64 * r + 32 * h);
                    qp[0] = make_uint4(words[0], words[1], words[2], words[3]);
                    qp[1] = make_uint4(words[4], words[5], words[6], words[7]);
                }
                // this thread's half of the code sum (the slot was zeroed before the barrier)
                if (e4) atomicAdd(&job.scales[2 * row + 1], (float)csum);
            }
        }
    }
    if (aborted) {
        // wait (bounded) for this pair's copies still in flight before leaving
        for (int d = 0; d < KV_DEPTH; ++d) {
            const uint32_t par = d >= slot ? phase : (phase ^ 1u);
            mbar_wait_bounded(&bars[pair * KV_DEPTH + d], par, prm.err);
        }
    }
}

template <int IN>
cudaError_t launch_kv128(const KParams &p, cudaStream_t stream) {
    auto kern = fwht_quant_kv128_kernel<IN>;
    const size_t smem = kv_smem_bytes<IN>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 64 * KV_PAIRS, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t total = p.groups_per_job * p.njobs;
    int64_t grid = (int64_t)sms * per_sm;
    const int64_t need = (total + KV_PAIRS - 1) / KV_PAIRS;
    if (grid > need) grid = need;
    kern<<<(unsigned)grid, 64 * KV_PAIRS, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int LOGN, int IN>
size_t smem_bytes() {
    using PL = Plan<LOGN - 3>;
    constexpr int n = 1 << LOGN;
    constexpr int G = IN == IN_F32 ? 2 : 1;
    constexpr int DEPTH = PL::kTwoPhase ? 1 : 2;
    constexpr int THREADS = threads_for(LOGN, IN);
    constexpr int ROWS = THREADS / PL::P;
    size_t b = 128 + (size_t)n * 2 + 128 * ((ROWS * 2 * 4 + 127) / 128);
    b += (size_t)(THREADS / 32) * DEPTH * 32 * PL::NSLOT * G * 16;   // bulk-copy input rings
    if (PL::kTwoPhase) b += (size_t)ROWS * n * 4;
    else b += (size_t)(THREADS / 32) * 2 * (32 / PL::P) * (n / 2);  // output staging
    return b;
}

template <int LOGN, int IN>
cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    auto kern = fwht_quant_kernel<LOGN, IN>;
    const size_t smem = smem_bytes<LOGN, IN>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads_for(LOGN, IN), smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t total = p.groups_per_job * p.njobs;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > total) grid = total;
    kern<<<(unsigned)grid, threads_for(LOGN, IN), smem, stream>>>(p);
    return cudaGetLastError();
}

template <int LOGN>
cudaError_t launch_n(const KParams &p, int in_type, cudaStream_t stream) {
    switch (in_type) {
        case IN_F32: return launch_t<LOGN, IN_F32>(p, stream);
        case IN_BF16: return launch_t<LOGN, IN_BF16>(p, stream);
        case IN_F16: return launch_t<LOGN, IN_F16>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Failure-detection self-test: one thread waits, through the rotation kernels'
// bounded wait, on a barrier that nothing arrives on.  After `limit` cycles the
// wait gives up and raises the error word, and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(int *err, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait_bounded(&bar, 0, err, limit);   // phase 0 never completes
    }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(long long limit_cycles, cudaStream_t stream) {
    int *err = error_word_device_ptr();
    if (!err) return cudaErrorUnknown;
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_cycles);
    return cudaGetLastError();
}

cudaError_t launch_fwht_quant(const RotJob *jobs, int njobs, int log_n, int in_type, uint64_t seed,
                              uint32_t flags, cudaStream_t stream) {
    if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;   // job_of() assumes one or two jobs
    KParams p{};
    p.njobs = njobs;
    int64_t max_rows = 0;
    for (int j = 0; j < njobs; ++j) {
        p.job[j] = jobs[j];
        if (jobs[j].rows > max_rows) max_rows = jobs[j].rows;
    }
    p.seed = seed;
    p.flags = flags;
    p.err = error_word_device_ptr();
    if (!p.err) return cudaErrorUnknown;
    const int C = log_n - 3;
    const int S = C <= 3 ? C : (C == 4 ? 3 : 4);      // as in Plan<C>
    int k4_threads = 0, k8_rows = 0;
    if (log_n == K4_LOGN || log_n == K8_LOGN) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorUnknown;
        if (log_n == K4_LOGN) k4_threads = k4_pick_threads(max_rows, in_type, sms);
        else k8_rows = k8_pick_rows(max_rows, in_type, sms);
    }
    const int rows_per_group = log_n == K4_LOGN   ? k4_threads / 64
                               : log_n == K8_LOGN ? k8_rows
                               : log_n == 7       ? 32                  // one warp pair per 32 rows
                                                  : threads_for(log_n, in_type) >> (C - S);
    p.groups_per_job = (max_rows + rows_per_group - 1) / rows_per_group;
    if (p.groups_per_job == 0) return cudaSuccess;
    switch (log_n) {
        case 5: return launch_n<5>(p, in_type, stream);
        case 6: return launch_n<6>(p, in_type, stream);
        case 7:
            switch (in_type) {
                case IN_F32: return launch_kv128<IN_F32>(p, stream);
                case IN_BF16: return launch_kv128<IN_BF16>(p, stream);
                case IN_F16: return launch_kv128<IN_F16>(p, stream);
                default: return cudaErrorInvalidValue;
            }
        case 8: return launch_n<8>(p, in_type, stream);
        case 9: return launch_n<9>(p, in_type, stream);
        case 10: return launch_n<10>(p, in_type, stream);
        case 11: return launch_n<11>(p, in_type, stream);
        case 12:
            switch (in_type) {
                case IN_F32: return launch_k4<IN_F32>(p, k4_threads, stream);
                case IN_BF16: return launch_k4<IN_BF16>(p, k4_threads, stream);
                case IN_F16: return launch_k4<IN_F16>(p, k4_threads, stream);
                default: return cudaErrorInvalidValue;
            }
        case 13:
            switch (in_type) {
                case IN_F32: return launch_k8<IN_F32>(p, k8_rows, stream);
                case IN_BF16: return launch_k8<IN_BF16>(p, k8_rows, stream);
                case IN_F16: return launch_k8<IN_F16>(p, k8_rows, stream);
                default: return cudaErrorInvalidValue;
            }
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rq
