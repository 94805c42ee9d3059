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
//  * Phase 1: the thread loads its chunks with 128-bit loads (chunk bits 0,1 on
//    lanes, so four lanes read 64 contiguous bytes), flips signs, and runs the
//    butterflies of every bit it holds (e bits and 4 chunk bits) in registers,
//    two at a time with the packed f32x2 add/sub; one or two further bits for
//    n >= 4096 are exchanged with warp shuffles.
//  * The row goes through shared memory once, as fp32 (XOR-swizzled 16-byte
//    granules: conflict-free for n >= 1024), into the phase-2 layout, where the
//    thread holds the remaining bits plus chunk bits 0 and 1, i.e. four runs
//    of 32 consecutive elements.
//  * Phase 2: remaining butterflies, row absmax (registers, shuffles, and a
//    shared-memory exchange when a row spans two warps), codes by one fused
//    multiply-add against a 1.5*2^23 bias (round-half-even to an integer whose
//    low bits are the two's-complement code), packing with byte permutes, and
//    16-byte stores of 32 codes each, coalesced across the warp.
//  * CTAs are persistent: each computes the sign masks of its n positions once
//    (SplitMix64, one call per element) into shared memory and then walks
//    groups of rows.
#include "rq_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kThreads = 128;

// --------------------------------------------------------------------------
// Bit plans.  a(k)/ta(k): chunk bit held by phase-1 slot bit k / row-thread
// bit k.  b(k)/tb(k): the same for phase 2.  shuf(j): the row-thread bits of
// phase 1 whose butterflies run through warp shuffles.
// --------------------------------------------------------------------------
template <int C>
struct Plan {
    static constexpr int S = C <= 4 ? C : 4;
    static constexpr int T = C - S;
    static constexpr int P = 1 << T;
    static constexpr int NSLOT = 1 << S;
    static constexpr int E = 8 * NSLOT;
    static constexpr int ROWS = kThreads / P;
    static constexpr bool kTwoPhase = T > 0;

    static constexpr int a(int k) {
        return C <= 4 ? k : (C == 5 ? k + 1 : k + 2);
    }
    static constexpr int ta(int k) {
        // C=5: {0}; C=6: {0,1}; C>=7: {0,1,6,7,...}
        return k < 2 ? k : k + 4;
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
    static constexpr int kNumShuf = C >= 9 ? C - 8 : 0;
    static constexpr int shuf(int j) { return 2 + j; }   // row-thread bits 2 (and 3)

    static constexpr bool chunk_bit_done_in_phase1(int cb) {
        for (int k = 0; k < S; ++k)
            if (a(k) == cb) return true;
        for (int j = 0; j < kNumShuf; ++j)
            if (ta(shuf(j)) == cb) return true;
        return false;
    }
};

__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    // SplitMix64 (Steele, Lea, Flood 2014): output i is the mix of seed + (i+1)*gamma.
    uint64_t z = seed + (i + 1ull) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// (a0,a1),(b0,b1) -> (a0+b0, a1+b1), (a0-b0, a1-b1) with packed fp32x2 ops.
__device__ __forceinline__ void bfly2(float &a0, float &a1, float &b0, float &b1) {
    asm("{\n\t.reg .b64 A, B, S, D;\n\t"
        "mov.b64 A, {%0, %1};\n\t"
        "mov.b64 B, {%2, %3};\n\t"
        "add.rn.f32x2 S, A, B;\n\t"
        "sub.rn.f32x2 D, A, B;\n\t"
        "mov.b64 {%0, %1}, S;\n\t"
        "mov.b64 {%2, %3}, D;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// (v0,v1) <- (v0,v1)*(m,m) + (p0,p1)
__device__ __forceinline__ void fma2_scalar(float &v0, float &v1, float m, float p0, float p1) {
    asm("{\n\t.reg .b64 V, M, Q;\n\t"
        "mov.b64 V, {%0, %1};\n\t"
        "mov.b64 M, {%2, %2};\n\t"
        "mov.b64 Q, {%3, %4};\n\t"
        "fma.rn.f32x2 V, V, M, Q;\n\t"
        "mov.b64 {%0, %1}, V;\n\t}"
        : "+f"(v0), "+f"(v1)
        : "f"(m), "f"(p0), "f"(p1));
}

// Butterflies over register-index bit `rb` of v[E] (E elements, 8 per chunk slot).
template <int E>
__device__ __forceinline__ void butterfly_reg_bit(float (&v)[E], int rb) {
    if (rb == 0) {
#pragma unroll
        for (int r = 0; r < E; r += 2) {
            const float a = v[r], b = v[r + 1];
            v[r] = a + b;
            v[r + 1] = a - b;
        }
    } else {
        const int st = 1 << rb;
#pragma unroll
        for (int r = 0; r < E; r += 2) {
            if (!(r & st)) bfly2(v[r], v[r + 1], v[r + st], v[r + st + 1]);
        }
    }
}

// Unpack one 16-byte chunk (8 elements) of bf16/f16 with sign masks m (bit 15 /
// bit 31 of each word flip element 2k / 2k+1), or 2x16 bytes of fp32.
template <int IN>
__device__ __forceinline__ void load_chunk(const void *row, int c, uint4 m, bool use_sign,
                                           float *out) {
    if constexpr (IN == IN_F32) {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const float *>(row) + 8 * c);
        uint4 lo = __ldg(p), hi = __ldg(p + 1);
        uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t e0 = w[2 * k], e1 = w[2 * k + 1];
            if (use_sign) {
                e0 ^= mm[k] << 16;
                e1 ^= mm[k] & 0x80000000u;
            }
            out[2 * k] = __uint_as_float(e0);
            out[2 * k + 1] = __uint_as_float(e1);
        }
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + 8 * c);
        uint4 raw = __ldg(p);
        uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t x = use_sign ? (w[k] ^ mm[k]) : w[k];
            if constexpr (IN == IN_BF16) {
                out[2 * k] = __uint_as_float(x << 16);
                out[2 * k + 1] = __uint_as_float(x & 0xffff0000u);
            } else {
                __half2 h = *reinterpret_cast<const __half2 *>(&x);
                float2 f = __half22float2(h);
                out[2 * k] = f.x;
                out[2 * k + 1] = f.y;
            }
        }
    }
}

// 8 codes (int8 in the low byte of each word) -> one word of 8 nibbles,
// element 2k in the low nibble of byte k.
__device__ __forceinline__ uint32_t pack8(const uint32_t *c) {
    const uint32_t e02 = __byte_perm(c[0], c[2], 0x0040);
    const uint32_t e46 = __byte_perm(c[4], c[6], 0x0040);
    const uint32_t o13 = __byte_perm(c[1], c[3], 0x0040);
    const uint32_t o57 = __byte_perm(c[5], c[7], 0x0040);
    const uint32_t ev = __byte_perm(e02, e46, 0x5410);
    const uint32_t od = __byte_perm(o13, o57, 0x5410);
    return (ev & 0x0f0f0f0fu) | ((od << 4) & 0xf0f0f0f0u);
}

struct KParams {
    RotJob job[2];
    int njobs;
    int64_t groups_per_job;
    uint64_t seed;
    uint32_t flags;
};

// Shared-memory granule position of 16-byte half h of chunk c in a row buffer.
__device__ __forceinline__ int granule(int c, int h, int row_in_cta) {
    const int sw = (((c >> 2) ^ (c >> 6)) & 1) | (((c >> 3) & 1) << 1) | (((c >> 4) & 1) << 2);
    return ((2 * c + h) ^ sw ^ (row_in_cta & 7));
}

template <int LOGN, int IN>
__global__ void __launch_bounds__(kThreads)
fwht_quant_kernel(const __grid_constant__ KParams prm) {
    constexpr int C = LOGN - 3;
    using PL = Plan<C>;
    constexpr int n = 1 << LOGN;
    constexpr int E = PL::E;
    constexpr int NSLOT = PL::NSLOT;
    constexpr int P = PL::P;
    constexpr int ROWS = PL::ROWS;

    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint32_t *sgn = reinterpret_cast<uint32_t *>(smem_raw);          // n/2 words
    float *red = reinterpret_cast<float *>(smem_raw + n * 2);        // ROWS*2 floats
    float4 *rowbuf = reinterpret_cast<float4 *>(smem_raw + n * 2 + 16 * ((ROWS * 2 * 4 + 15) / 16));

    const bool signs_first = (prm.flags & 1u) != 0;

    // Sign masks: word j covers elements 2j (bit 15) and 2j+1 (bit 31).
    for (int j = threadIdx.x; j < n / 2; j += kThreads) {
        const uint32_t s0 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j) >> 63);
        const uint32_t s1 = (uint32_t)(splitmix64_at(prm.seed, 2ull * j + 1) >> 63);
        sgn[j] = (s0 << 15) | (s1 << 31);
    }
    __syncthreads();

    const int row_in_cta = threadIdx.x / P;
    const int t = threadIdx.x % P;
    const float inv_sqrt_n = (LOGN & 1) ? (0.70710678118654752440f / (float)(1 << (LOGN / 2)))
                                        : (1.0f / (float)(1 << (LOGN / 2)));
    const float shuf_sign0 = ((t >> (PL::kNumShuf > 0 ? PL::shuf(0) : 0)) & 1) ? -1.f : 1.f;
    const float shuf_sign1 = ((t >> (PL::kNumShuf > 1 ? PL::shuf(1) : 0)) & 1) ? -1.f : 1.f;
    const unsigned full = 0xffffffffu;

    const int64_t total_groups = prm.groups_per_job * prm.njobs;
    for (int64_t grp = blockIdx.x; grp < total_groups; grp += gridDim.x) {
        const int jb = (int)(grp / prm.groups_per_job);
        const RotJob &job = prm.job[jb];
        const int64_t row = (grp - (int64_t)jb * prm.groups_per_job) * ROWS + row_in_cta;
        const bool active = row < job.rows;
        const int64_t rrow = active ? row : 0;

        float v[E];
        // ---------------- phase 1: load, signs, butterflies ----------------
        {
            const void *xrow = (IN == IN_F32)
                ? (const void *)(static_cast<const float *>(job.x) + rrow * job.ld)
                : (const void *)(static_cast<const uint16_t *>(job.x) + rrow * job.ld);
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) {
                int c = 0;
#pragma unroll
                for (int k = 0; k < PL::S; ++k) c |= ((s >> k) & 1) << PL::a(k);
#pragma unroll
                for (int k = 0; k < PL::T; ++k) c |= ((t >> k) & 1) << PL::ta(k);
                const uint4 m = reinterpret_cast<const uint4 *>(sgn)[c];
                if (active) {
                    load_chunk<IN>(xrow, c, m, signs_first, &v[8 * s]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[8 * s + e] = 0.f;
                }
            }
#pragma unroll
            for (int rb = 0; rb < 3 + PL::S; ++rb) butterfly_reg_bit<E>(v, rb);
#pragma unroll
            for (int j = 0; j < PL::kNumShuf; ++j) {
                const int lm = 1 << PL::shuf(j);
                const float sg = j == 0 ? shuf_sign0 : shuf_sign1;
#pragma unroll
                for (int r = 0; r < E; r += 2) {
                    const float p0 = __shfl_xor_sync(full, v[r], lm);
                    const float p1 = __shfl_xor_sync(full, v[r + 1], lm);
                    fma2_scalar(v[r], v[r + 1], sg, p0, p1);
                }
            }
        }

        // ---------------- transpose through shared memory ----------------
        if constexpr (PL::kTwoPhase) {
            float4 *buf = rowbuf + (size_t)row_in_cta * (n / 4);
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) {
                int c = 0;
#pragma unroll
                for (int k = 0; k < PL::S; ++k) c |= ((s >> k) & 1) << PL::a(k);
#pragma unroll
                for (int k = 0; k < PL::T; ++k) c |= ((t >> k) & 1) << PL::ta(k);
                buf[granule(c, 0, row_in_cta)] = make_float4(v[8 * s], v[8 * s + 1], v[8 * s + 2], v[8 * s + 3]);
                buf[granule(c, 1, row_in_cta)] = make_float4(v[8 * s + 4], v[8 * s + 5], v[8 * s + 6], v[8 * s + 7]);
            }
            if constexpr (P > 32) {
                asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            } else {
                __syncwarp();
            }
#pragma unroll
            for (int s = 0; s < NSLOT; ++s) {
                int c = 0;
#pragma unroll
                for (int k = 0; k < PL::S; ++k) c |= ((s >> k) & 1) << PL::b(k);
#pragma unroll
                for (int k = 0; k < PL::T; ++k) c |= ((t >> k) & 1) << PL::tb(k);
                const float4 lo = buf[granule(c, 0, row_in_cta)];
                const float4 hi = buf[granule(c, 1, row_in_cta)];
                v[8 * s] = lo.x; v[8 * s + 1] = lo.y; v[8 * s + 2] = lo.z; v[8 * s + 3] = lo.w;
                v[8 * s + 4] = hi.x; v[8 * s + 5] = hi.y; v[8 * s + 6] = hi.z; v[8 * s + 7] = hi.w;
            }
            // phase-2 butterflies over the slot bits not done in phase 1
#pragma unroll
            for (int k = 0; k < PL::S; ++k) {
                if (!PL::chunk_bit_done_in_phase1(PL::b(k))) butterfly_reg_bit<E>(v, 3 + k);
            }
        }

        // ---------------- row absmax ----------------
        float amax = 0.f;
#pragma unroll
        for (int r = 0; r < E; ++r) amax = fmaxf(amax, fabsf(v[r]));
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
        const float inv = amax > 0.f ? 7.0f / amax : 0.f;
        if (active) {
            if (t == 0) job.scales[row] = (amax / 7.0f) * inv_sqrt_n;
            uint8_t *qrow = job.q + row * (int64_t)(n / 2);
            float *yrow = job.y ? job.y + row * (int64_t)n : nullptr;
#pragma unroll
            for (int s4 = 0; s4 < NSLOT; s4 += 4) {
                uint32_t words[4];
                int c0 = 0;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int s = s4 + cc;
                    int c = 0;
#pragma unroll
                    for (int k = 0; k < PL::S; ++k) c |= ((s >> k) & 1) << (PL::kTwoPhase ? PL::b(k) : k);
#pragma unroll
                    for (int k = 0; k < PL::T; ++k) c |= ((t >> k) & 1) << PL::tb(k);
                    if (cc == 0) c0 = c;
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = v[8 * s + e];
                    if (!signs_first) {
                        const uint4 m = reinterpret_cast<const uint4 *>(sgn)[c];
                        const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            f[2 * k] = __uint_as_float(__float_as_uint(f[2 * k]) ^ (mm[k] << 16));
                            f[2 * k + 1] = __uint_as_float(__float_as_uint(f[2 * k + 1]) ^ (mm[k] & 0x80000000u));
                        }
                    }
                    if (yrow) {
                        float4 *yp = reinterpret_cast<float4 *>(yrow + 8 * c);
                        yp[0] = make_float4(f[0] * inv_sqrt_n, f[1] * inv_sqrt_n, f[2] * inv_sqrt_n, f[3] * inv_sqrt_n);
                        yp[1] = make_float4(f[4] * inv_sqrt_n, f[5] * inv_sqrt_n, f[6] * inv_sqrt_n, f[7] * inv_sqrt_n);
                    }
                    uint32_t code[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) code[e] = __float_as_uint(__fmaf_rn(f[e], inv, 12582912.0f));
                    words[cc] = pack8(code);
                }
                // chunks c0..c0+3 are consecutive (slot bits 0,1 = chunk bits 0,1)
                *reinterpret_cast<uint4 *>(qrow + 4 * c0) = make_uint4(words[0], words[1], words[2], words[3]);
            }
        }
        if constexpr (PL::kTwoPhase) {
            if constexpr (P > 32) {
                asm volatile("bar.sync %0, %1;" ::"r"(1 + row_in_cta), "r"(P) : "memory");
            } else {
                __syncwarp();
            }
        }
    }
}

template <int LOGN, int IN>
size_t smem_bytes() {
    using PL = Plan<LOGN - 3>;
    constexpr int n = 1 << LOGN;
    size_t b = (size_t)n * 2 + 16 * ((PL::ROWS * 2 * 4 + 15) / 16);
    if (PL::kTwoPhase) b += (size_t)PL::ROWS * n * 4;
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t total = p.groups_per_job * p.njobs;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > total) grid = total;
    kern<<<(unsigned)grid, kThreads, smem, stream>>>(p);
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

}  // namespace

cudaError_t launch_fwht_quant(const RotJob *jobs, int njobs, int log_n, int in_type, uint64_t seed,
                              uint32_t flags, cudaStream_t stream) {
    KParams p{};
    p.njobs = njobs;
    int64_t max_rows = 0;
    for (int j = 0; j < njobs; ++j) {
        p.job[j] = jobs[j];
        if (jobs[j].rows > max_rows) max_rows = jobs[j].rows;
    }
    p.seed = seed;
    p.flags = flags;
    const int rows_per_group = kThreads >> (log_n - 3 > 4 ? log_n - 7 : 0);
    p.groups_per_job = (max_rows + rows_per_group - 1) / rows_per_group;
    if (p.groups_per_job == 0) return cudaSuccess;
    switch (log_n) {
        case 5: return launch_n<5>(p, in_type, stream);
        case 6: return launch_n<6>(p, in_type, stream);
        case 7: return launch_n<7>(p, in_type, stream);
        case 8: return launch_n<8>(p, in_type, stream);
        case 9: return launch_n<9>(p, in_type, stream);
        case 10: return launch_n<10>(p, in_type, stream);
        case 11: return launch_n<11>(p, in_type, stream);
        case 12: return launch_n<12>(p, in_type, stream);
        case 13: return launch_n<13>(p, in_type, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rq
