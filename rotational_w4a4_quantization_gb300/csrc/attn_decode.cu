// attn_decode.cu -- attention of decode queries over the rotated INT4 KV cache
// (sm_103a).
//
// The cache rq_kv_rotate_quant writes holds, per (token, head), the codes and the
// scale of k R and v R (R the randomized Hadamard of size head_dim).  "The
// Architecture" and "End-to-end flow" (The KV cache) of the QuaRot page: a later
// token's attention reads the four-bit rotated cache, and rotation invariance
// keeps its scores those of the full-precision computation.  For a query row q of
// head h:
//   q~ = q R;  e_t = softmax_scale * (q~ . k^_t);  p = softmax(e);
//   o~ = sum_t p_t v^_t;  out = o~ R^T  (or o~, left for a folded output weight)
// with k^_t, v^_t the dequantized rotated cache rows.  q~ . k^_t = q . (k^_t R^T)
// because R is orthogonal, and R^T is the rotation with the other sign side.
//
// Design (bound by reading the cache: 2 (head_dim/2 + 4) bytes per token and head):
//  * one cluster of 8 CTAs per (query row, head); CTA r takes the r-th eighth of
//    the tokens, so a 8192-token, 32-head cache runs as 256 CTAs, two per SM;
//  * every warp rotates the query (shuffle FWHT, its own copy: no CTA barrier)
//    and folds softmax_scale * log2(e) into it, so the scores come out in base 2;
//  * a token is read by head_dim/32 lanes, each holding 32 dimensions (16 bytes
//    of codes of K and of V), streamed through a per-lane cp.async ring four
//    tokens deep (the first requests go out before the query is rotated);
//  * key codes enter the dot product as the denormals n 2^-149 (n = q + 8, one
//    byte permute each, exact), against the lane's query values pre-scaled by a
//    power of two; the lane's partial is scaled back and 8 sum(q~) removed.  Value
//    codes become fp32 through a byte permute into 0x4B0000nn (2^23 + n) and one
//    f32x2 add of -(2^23 + 8).  Products are f32x2 FMAs;
//  * online softmax per token slot with a lazy reference maximum (moved only
//    when a score passes it by 8 in log2 units), then the slots of a warp, the
//    warps of a CTA and the CTAs of a cluster are merged with the same rule;
//    the 7 other CTAs bulk-copy their partial (reference, sum, accumulator) into
//    rank 0's shared memory, completing on its mbarrier; a relaxed cluster
//    barrier keeps the sources alive until then;
//  * rank 0 normalizes, takes the result back by R^T (warp FWHT) unless the
//    caller keeps the rotated basis, and writes fp32.
#include "rq.h"
#include "rq_internal.h"
#include "rot_device.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kAWarps = 8;
constexpr int kAThreads = 32 * kAWarps;
constexpr int kACluster = 8;
constexpr int kARing = 4;                         // tokens in flight per lane (cp.async ring)
constexpr long long kAWaitLimit = 4000000000ll;   // ~2 s at 2 GHz



struct AParams {
    const void *q;
    int64_t M, H, T;
    const uint8_t *kq, *vq;
    const float *ks, *vs;
    uint64_t seed;
    uint32_t flags;
    float qscale;        // softmax_scale * log2(e) / sqrt(head_dim)
    float inv_sqrt_d;    // 1 / sqrt(head_dim)
    float *out;
    int *err;
};

// A CTA's partial softmax state, as copied to rank 0 (16 + 4 D bytes).
template <int D>
struct APart {
    float m, l, pad[2];
    float acc[D];
};

template <int D>
struct ASmem {
    // per-lane copy ring, one array per field so that consecutive lanes touch
    // consecutive words (each lane reads back only its own slots)
    uint4 rk[kARing][kAThreads], rv[kARing][kAThreads];
    float rks[kARing][kAThreads], rvs[kARing][kAThreads];
    float qr[kAWarps][D];               // rotated, scaled query (one copy per warp)
    float wm[kAWarps], wl[kAWarps];     // per-warp partial states
    float wacc[kAWarps][D];
    alignas(16) APart<D> part[kACluster];   // slot r: CTA r's partial (rank 0 holds all)
    alignas(8) uint64_t pbar;           // rank 0: the other CTAs' partials have landed
};
static_assert(sizeof(APart<32>) % 16 == 0 && sizeof(APart<256>) % 16 == 0, "bulk copies move 16-byte multiples");

__device__ __forceinline__ uint32_t a_smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t a_mapa(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a_smem_u32(p)), "r"(rank));
    return r;
}

template <int IN>
__device__ __forceinline__ float load_elem(const void *base, int64_t i) {
    if constexpr (IN == IN_F32) return static_cast<const float *>(base)[i];
    else if constexpr (IN == IN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    else return __half2float(static_cast<const __half *>(base)[i]);
}

// Warp-wide rotation of a D-vector held as E = D/32 values per lane (element
// lane * E + e): signs (before or after), Sylvester butterflies over the e bits in
// registers and over the lane bits by shuffles, then a scale.
template <int E>
__device__ __forceinline__ void lane_signs(float (&sg)[E], int lane, uint64_t seed) {
#pragma unroll
    for (int e = 0; e < E; ++e)
        sg[e] = (splitmix64_at(seed, (uint64_t)(lane * E + e)) >> 63) ? -1.f : 1.f;
}
template <int E>
__device__ __forceinline__ void warp_rotate(float (&v)[E], const float (&sg)[E], int lane, bool signs_before,
                                            float scale) {
    if (signs_before) {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] *= sg[e];
    }
#pragma unroll
    for (int st = 1; st < E; st <<= 1)
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (!(e & st)) {
                const float a = v[e], b = v[e + st];
                v[e] = a + b;
                v[e + st] = a - b;
            }
#pragma unroll
    for (int lm = 1; lm < 32; lm <<= 1)
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], lm);
            v[e] = (lane & lm) ? o - v[e] : v[e] + o;
        }
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = (signs_before ? v[e] : v[e] * sg[e]) * scale;
}

// 8 codes of a packed word -> four fp32 pairs (codes 2k, 2k+1): byte permutes
// into 2^23 + (q + 8), then one f32x2 add of -(2^23 + 8).
__device__ __forceinline__ void codes_to_pairs(uint32_t w, pair_t (&c)[4]) {
    const uint32_t x = w ^ 0x88888888u;
    const uint32_t lo = x & 0x0f0f0f0fu, hi = (x >> 4) & 0x0f0f0f0fu;
    const uint32_t magic = 0x4b000000u;
    const pair_t bias = mk2(-8388616.0f, -8388616.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t e0 = __byte_perm(lo, magic, 0x7650u + k);
        const uint32_t e1 = __byte_perm(hi, magic, 0x7650u + k);
        c[k] = add2(((pair_t)e1 << 32) | (pair_t)e0, bias);
    }
}

// 2^x by the hardware approximation (relative error below 2^-22; flushes to 0
// far below the running maximum, as the softmax wants).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Asynchronous global -> shared copies of one lane (16 bytes, L2 only; 4 bytes).
__device__ __forceinline__ void cp16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a_smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(a_smem_u32(dst)), "l"(src) : "memory");
}

// 8 codes of a packed word -> four pairs of fp32 whose bits are n = q + 8 (the
// denormals n * 2^-149, exact): one byte permute per value, no arithmetic.
__device__ __forceinline__ void nibbles_to_denormal_pairs(uint32_t w, pair_t (&c)[4]) {
    const uint32_t x = w ^ 0x88888888u;
    const uint32_t lo = x & 0x0f0f0f0fu, hi = (x >> 4) & 0x0f0f0f0fu;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t e0 = __byte_perm(lo, 0u, 0x4440u + k);
        const uint32_t e1 = __byte_perm(hi, 0u, 0x4440u + k);
        c[k] = ((pair_t)e1 << 32) | (pair_t)e0;
    }
}

// Merge partial softmax state (mb, lb) into (m, l); returns the factors for the
// accumulators (an empty state has m = -inf and contributes nothing).
__device__ __forceinline__ void merge_factors(float &m, float &l, float mb, float lb, float &fa, float &fb) {
    const float mn = fmaxf(m, mb);
    fa = (m == -INFINITY) ? 0.f : ex2(m - mn);
    fb = (mb == -INFINITY) ? 0.f : ex2(mb - mn);
    l = l * fa + lb * fb;
    m = mn;
}

__device__ __forceinline__ void a_mbar_wait(uint64_t *b, uint32_t parity, int *err) {
    const uint32_t a = a_smem_u32(b);
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return;
        if (clock64() - t0 > kAWaitLimit) {   // a partial never landed: raise the error word
            atomicExch(err, 1);
            return;
        }
    }
}

template <int IN, int LPT>
__global__ void __cluster_dims__(kACluster, 1, 1) __launch_bounds__(kAThreads, 2)
attn_decode_kernel(const __grid_constant__ AParams p) {
    constexpr int D = 32 * LPT;          // head_dim
    constexpr int E = D / 32;            // query elements per lane in the warp rotation
    constexpr int TPW = 32 / LPT;        // token slots per warp
    constexpr int RB = D / 2;            // code bytes per cache row
    extern __shared__ __align__(128) unsigned char araw[];
    ASmem<D> &s = *reinterpret_cast<ASmem<D> *>(araw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int64_t h = blockIdx.x / kACluster, m = blockIdx.y;
    const bool signs_first = (p.flags & 1u) != 0;

    // ---- rank 0's barrier for the other CTAs' partials; relaxed cluster arrive ----
    if (threadIdx.x == 0) {
        const uint32_t pb = a_smem_u32(&s.pbar);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(pb) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (rank == 0)
            asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(pb),
                         "r"((uint32_t)((kACluster - 1) * sizeof(APart<D>)))
                         : "memory");
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- this lane: dimensions 32 j .. 32 j + 31 of token slot tq ----
    const int j = lane % LPT, tq = lane / LPT;
    // the token slot's lanes: they run the token loop in lockstep (lanes of other
    // slots may leave it one iteration earlier), so shuffles inside it name only them
    const unsigned gmask = (LPT == 32 ? 0xffffffffu : ((1u << LPT) - 1u)) << (tq * LPT);
    const int64_t t_begin = p.T * rank / kACluster, t_end = p.T * (rank + 1) / kACluster;
    constexpr int STRIDE = kAWarps * TPW;

    // The lane's tokens t_i = t0 + i STRIDE stream through a kARing-deep ring of
    // cp.async groups: token i + kARing is requested as soon as token i is read.
    // Groups are committed for every index, empty past the slice end, so that
    // "wait until at most kARing - 1 groups are pending" always means "token i
    // has landed".  The first requests go out before the query is rotated.
    const int64_t t0 = t_begin + warp * TPW + tq;
    const int nt = t0 < t_end ? (int)((t_end - t0 + STRIDE - 1) / STRIDE) : 0;
    auto request = [&](int i) {
        if (i < nt) {
            const int64_t r = (t0 + (int64_t)i * STRIDE) * p.H + h;
            const int sl = i % kARing;
            cp16(&s.rk[sl][threadIdx.x], p.kq + r * RB + 16 * j);
            cp16(&s.rv[sl][threadIdx.x], p.vq + r * RB + 16 * j);
            cp4(&s.rks[sl][threadIdx.x], p.ks + r);
            cp4(&s.rvs[sl][threadIdx.x], p.vs + r);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int i = 0; i < kARing; ++i) request(i);

    // ---- the rotated query, scaled for base-2 scores: every warp rotates its own
    // copy (no CTA barrier; the signs stay in registers for the final R^T) ----
    float sg[E];
    float *qw = s.qr[warp];
    {
        const void *qrow = static_cast<const char *>(p.q) + ((m * p.H + h) * D) * (IN == IN_F32 ? 4 : 2);
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = load_elem<IN>(qrow, lane * E + e);
        lane_signs<E>(sg, lane, p.seed);
        warp_rotate<E>(v, sg, lane, signs_first, p.qscale);
#pragma unroll
        for (int e = 0; e < E; ++e) qw[lane * E + e] = v[e];
    }
    __syncwarp();

    // The keys' codes enter as the denormals n 2^-149 (n = q + 8), so the lane's
    // query values are pre-scaled by 2^kq (its largest below 2^125); a lane's
    // partial score is then dot * 2^(149 - kq) - 8 sum(q~) over its 32 values.
    float qmax = 0.f, qsum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        qmax = fmaxf(qmax, fabsf(qw[32 * j + i]));
        qsum += qw[32 * j + i];
    }
    int qex = 0;
    frexpf(qmax, &qex);                                   // qmax < 2^qex
    const int kq = qmax > 0.f ? 125 - qex : 0;
    const int bk = 149 - kq;                              // back-scale exponent, split in two steps
    const float back1 = qmax > 0.f ? ldexpf(1.f, bk / 2) : 0.f, back2 = ldexpf(1.f, bk - bk / 2);
    const float qcorr = 8.f * qsum;
    pair_t q2[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        q2[i] = mk2(ldexpf(qw[32 * j + 2 * i], kq), ldexpf(qw[32 * j + 2 * i + 1], kq));
    float mrun = -INFINITY, lrun = 0.f;
    pair_t acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0ull;

    auto step = [&](const uint4 &kc, float ksc, const uint4 &vc, float vsc) {
        // score: sum over the lane's 32 dimensions, then over the token's lanes
        pair_t d0 = 0ull, d1 = 0ull;
        const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pair_t c[4];
            nibbles_to_denormal_pairs(kw[i], c);
            d0 = fma2(c[0], q2[4 * i], d0);
            d1 = fma2(c[1], q2[4 * i + 1], d1);
            d0 = fma2(c[2], q2[4 * i + 2], d0);
            d1 = fma2(c[3], q2[4 * i + 3], d1);
        }
        const pair_t dd = add2(d0, d1);
        float sc = ((lo2(dd) + hi2(dd)) * back1) * back2 - qcorr;
#pragma unroll
        for (int o = 1; o < LPT; o <<= 1) sc += __shfl_xor_sync(gmask, sc, o);
        sc *= ksc;
        // online softmax with a lazy maximum: the running reference moves only when
        // a score passes it by more than 8 (weights stay below 2^8), so the rescale
        // is rare; the first token always sets it (mrun = -inf)
        if (sc > mrun + 8.f) {
            const float f = ex2(mrun - sc);     // 0 for the first token
            lrun *= f;
            const pair_t f2 = mk2(f, f), z2 = 0ull;
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = fma2(acc[i], f2, z2);
            mrun = sc;
        }
        const float pw = ex2(sc - mrun);
        lrun += pw;
        const float w = pw * vsc;
        const pair_t w2 = mk2(w, w);
        const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pair_t c[4];
            codes_to_pairs(vw[i], c);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[4 * i + k] = fma2(c[k], w2, acc[4 * i + k]);
        }
    };

    for (int i = 0; i < nt; ++i) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kARing - 1) : "memory");
        const int sl = i % kARing;
        const uint4 kc = s.rk[sl][threadIdx.x], vc = s.rv[sl][threadIdx.x];
        const float ksc = s.rks[sl][threadIdx.x], vsc = s.rvs[sl][threadIdx.x];
        step(kc, ksc, vc, vsc);
        request(i + kARing);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");

    // ---- merge the warp's token slots (lanes with the same j) ----
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) {
        const float mb = __shfl_xor_sync(0xffffffffu, mrun, o);
        const float lb = __shfl_xor_sync(0xffffffffu, lrun, o);
        float fa, fb;
        merge_factors(mrun, lrun, mb, lb, fa, fb);
        const pair_t fa2 = mk2(fa, fa), fb2 = mk2(fb, fb);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float blo = __shfl_xor_sync(0xffffffffu, lo2(acc[i]), o);
            const float bhi = __shfl_xor_sync(0xffffffffu, hi2(acc[i]), o);
            acc[i] = fma2(acc[i], fa2, fma2(mk2(blo, bhi), fb2, 0ull));
        }
    }
    if (lane == 0) {
        s.wm[warp] = mrun;
        s.wl[warp] = lrun;
    }
    if (tq == 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            s.wacc[warp][32 * j + 2 * i] = lo2(acc[i]);
            s.wacc[warp][32 * j + 2 * i + 1] = hi2(acc[i]);
        }
    }
    __syncthreads();

    // ---- merge the warps into this CTA's record (slot `rank`) ----
    APart<D> &mine = s.part[rank];
    if (threadIdx.x < D) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAWarps; ++w) mm = fmaxf(mm, s.wm[w]);
        float ll = 0.f, a = 0.f;
#pragma unroll
        for (int w = 0; w < kAWarps; ++w) {
            const float f = s.wm[w] == -INFINITY ? 0.f : ex2(s.wm[w] - mm);
            ll += s.wl[w] * f;
            a += s.wacc[w][threadIdx.x] * f;
        }
        mine.acc[threadIdx.x] = a;
        if (threadIdx.x == 0) {
            mine.m = mm;
            mine.l = ll;
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    // rank 0's barrier is armed (cluster barrier, first phase)
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (rank != 0) {
        if (threadIdx.x == 0)
            asm volatile(
                "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    a_mapa(&mine, 0)),
                "r"(a_smem_u32(&mine)), "r"((uint32_t)sizeof(APart<D>)), "r"(a_mapa(&s.pbar, 0))
                : "memory");
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
        // keep this record alive until rank 0 has it
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        return;
    }

    // ---- rank 0: merge the cluster's records, normalize, take back by R^T ----
    a_mbar_wait(&s.pbar, 0, p.err);
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    if (warp == 0) {
        float mm = -INFINITY, f[kACluster], ll = 0.f;
#pragma unroll
        for (int r = 0; r < kACluster; ++r) mm = fmaxf(mm, s.part[r].m);
#pragma unroll
        for (int r = 0; r < kACluster; ++r) {
            f[r] = s.part[r].m == -INFINITY ? 0.f : ex2(s.part[r].m - mm);
            ll += s.part[r].l * f[r];
        }
        const float il = 1.f / ll;
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            float a = 0.f;
#pragma unroll
            for (int r = 0; r < kACluster; ++r) a += s.part[r].acc[d] * f[r];
            v[e] = a * il;
        }
        if (!(p.flags & RQ_ATTN_ROTATED_OUT))
            warp_rotate<E>(v, sg, lane, !signs_first, p.inv_sqrt_d);
        float *orow = p.out + (m * p.H + h) * D;
#pragma unroll
        for (int e = 0; e < E; ++e) orow[lane * E + e] = v[e];
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int IN, int LPT>
cudaError_t launch_attn_t(const AParams &p, cudaStream_t stream) {
    auto kern = attn_decode_kernel<IN, LPT>;
    const size_t smem = sizeof(ASmem<32 * LPT>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)(p.H * kACluster), (unsigned)p.M), kAThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int IN>
cudaError_t launch_attn_in(const AParams &p, int64_t head_dim, cudaStream_t stream) {
    switch (head_dim) {
        case 32: return launch_attn_t<IN, 1>(p, stream);
        case 64: return launch_attn_t<IN, 2>(p, stream);
        case 128: return launch_attn_t<IN, 4>(p, stream);
        case 256: return launch_attn_t<IN, 8>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool attn_decode_supported(int64_t head_dim) {
    return head_dim == 32 || head_dim == 64 || head_dim == 128 || head_dim == 256;
}

cudaError_t launch_attn_decode(const void *q, int in_type, int64_t M, int64_t heads, int64_t head_dim,
                               const uint8_t *kq, const float *ks, const uint8_t *vq, const float *vs,
                               int64_t tokens, uint64_t seed, uint32_t flags, float softmax_scale, float *out,
                               cudaStream_t stream) {
    const double isd = 1.0 / sqrt((double)head_dim);
    const AParams p{q, M, heads, tokens, kq, vq, ks, vs, seed, flags,
                    (float)((double)softmax_scale * 1.4426950408889634 * isd), (float)isd, out,
                    error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    switch (in_type) {
        case IN_F32: return launch_attn_in<IN_F32>(p, head_dim, stream);
        case IN_BF16: return launch_attn_in<IN_BF16>(p, head_dim, stream);
        case IN_F16: return launch_attn_in<IN_F16>(p, head_dim, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rq
