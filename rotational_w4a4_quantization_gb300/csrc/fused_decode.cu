// fused_decode.cu -- decode-sized rotation + INT4 quantization + W4A4 GEMM in one
// launch (sm_103a).
//
// y = dequant(Q(x R) . Q(R^T W)) for M <= 16 token rows x of length K = 4096:
// the randomized Hadamard rotation and per-token INT4 quantization of
// "Rotational Quantization ..." §Incoherence Processing via Randomized Hadamard
// Transforms / §Weight Absorption and Online Fast Walsh-Hadamard Transforms, 2.,
// fused with the W4A4 product of §Hardware Execution and Serving Economics, 1.,
// so that the rotated activations never go through HBM.  W is the folded weight
// Q(R^T W) (N x K/2 packed codes, per-channel scales).
//
// Design (a decode layer is bound by reading W, N*K/2 bytes):
//  * clusters of 4 CTAs; a CTA owns 32 output channels (grid = N/32, one wave:
//    with clusters of 8 only 15 clusters fit at once and the launch ran in
//    three waves).  All threads load their activation chunks first; once they
//    are in, one thread issues a single 64 KB bulk copy (TMA) of the CTA's
//    weight rows (issued earlier, the 8 MB weight stream delayed the
//    activations by ~1 us); it lands during the rotation;
//  * each CTA of a cluster rotates and quantizes rows rank + 4 j (j = 0..3; two
//    warps per row, the three-phase 4096-element layout of the rotation kernel,
//    identical arithmetic, so codes and scales equal the unfused kernel's bit
//    for bit) and writes each row as one record (packed codes, scale, sum of
//    u = q + 8) into its own shared memory; one thread then bulk-copies the
//    record into the other 3 CTAs (shared::cta -> shared::cluster), completing
//    bytes on their activation barriers.  Per-store signalling (st.async) and
//    plain remote stores under a release cluster barrier both measured slower.
//    The first cluster also writes codes and scales to global memory when the
//    caller asks for them;
//  * once its barrier has counted the other CTAs' rows, every CTA holds all M
//    rows and runs the product as the decode GEMM does: FP8 mma.sync (m16n8k32
//    e4m3, fp32 accumulation) on the bytes u = q + 8, eight warps splitting K,
//    a shared-memory reduction, and sum q_a q_w = sum u_a u_w - 8 sum u_a -
//    8 sum u_w + 64 K;
//  * the rotation is repeated once per cluster (N/128 times); at 4 rows per CTA
//    that costs less than a second launch.  No global scratch: inter-CTA data
//    moves through distributed shared memory; a relaxed cluster barrier (arrive
//    once a CTA's rows are in, wait before exit) keeps every source alive until
//    its copies have landed.
#include "rq_internal.h"
#include "rot_device.cuh"

#include <cuda_fp16.h>

namespace rq {
namespace {

constexpr int kFN = 4096;                  // K: the rotation length
constexpr int kFWarps = 8;
constexpr int kFThreads = 32 * kFWarps;
constexpr int kFCluster = 4;
constexpr int kFChan = 32;                 // output channels per CTA (four n8 MMA tiles)
constexpr int kFRowsPerCta = 4;            // rows rotated by one CTA (two warps each)
constexpr long long kFWaitLimit = 4000000000ll;   // ~2 s at 2 GHz
constexpr int kFMaxM = 16;                 // token rows (one m16 MMA tile)
constexpr int kFSteps = kFN / 128 / kFWarps;   // 128-code steps per warp (4)
static_assert(kFSteps % 2 == 0, "column sums fold every two steps");
static_assert(kFChan == 32 && kFThreads % kFChan == 0, "epilogue thread e serves channel e % 32 == its lane");

struct FParams {
    const void *x;
    int64_t ldx, M, N;
    uint64_t seed;
    uint32_t flags;
    const uint8_t *wq;
    const float *sw;
    void *y;
    uint8_t *aq;          // optional outputs: activation codes / scales
    float *as;
    int *err;             // library error word (a bounded wait gave up)
};

// One quantized activation row as the cluster exchanges it (one bulk copy): the
// packed codes with their 16-byte granules XOR-ed by (r & 1) << 2 for row r, so
// that the MMA fragment loads of the 8 lanes of a quarter-warp (rows g, g + 1,
// chunks tq) hit 8 bank groups; the row's scale; its sum of u = q + 8.
struct ARow {
    uint4 q[kFN / 32];
    float scale;
    int usum;
    uint32_t pad[2];
};
static_assert(sizeof(ARow) % 16 == 0, "bulk copies move 16-byte multiples");

// Shared memory (dynamic).
struct FSmem {
    uint4 w[kFChan][kFN / 32];             // the CTA's weight rows (64 KB, one bulk copy)
    uint32_t sgn[kFN / 2];                 // sign words (bit 15 / 31: element 2j / 2j+1)
    ulonglong2 rowbuf[kFRowsPerCta][kFN / 4];   // fp32 transposes of this CTA's rows
    ARow arow[kFMaxM];                     // every activation row of the batch
    float red[kFRowsPerCta][2];
    int ured[kFRowsPerCta][2];
    int part[kFWarps][kFMaxM][kFChan + 1];
    int csum[kFWarps][kFChan];
    alignas(8) uint64_t wbar;              // completion of the weight copy
    alignas(8) uint64_t abar;              // arrival of the other CTAs' activation rows
};

__device__ __forceinline__ uint32_t f_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t f_smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t f_mapa(const void *local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(f_smem_u32(local)), "r"(rank));
    return remote;
}
// Bulk copy of `bytes` from this CTA's shared memory to the same offset in CTA `rank`
// of the cluster, completing the byte count on that CTA's barrier at `bar`'s offset.
__device__ __forceinline__ void bulk_to_peer(const void *src, uint32_t bytes, uint32_t rank, const uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     f_mapa(src, rank)),
                 "r"(f_smem_u32(src)), "r"(bytes), "r"(f_mapa(bar, rank))
                 : "memory");
}

__device__ __forceinline__ void f_mma_e4m3(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// E4M3 bytes u = q + 8 of the even / odd codes of a packed word, and their sum
__device__ __forceinline__ uint32_t f_ulo(uint32_t w) { return (w ^ 0x88888888u) & 0x0f0f0f0fu; }
__device__ __forceinline__ uint32_t f_uhi(uint32_t w) { return ((w >> 4) ^ 0x08080808u) & 0x0f0f0f0fu; }
__device__ __forceinline__ int f_usum(uint32_t lo, uint32_t hi, int acc) {
    return __dp4a((int)(lo + hi), 0x01010101, acc);
}

// Bounded parity wait.  CLUSTER: acquire at cluster scope (the phase was completed by
// other CTAs' stores).
template <bool CLUSTER>
__device__ __forceinline__ void f_mbar_wait(uint64_t *b, uint32_t parity, int *err) {
    const uint32_t a = f_smem_u32(b);
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        if (CLUSTER)
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        else
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return;
        if (clock64() - t0 > kFWaitLimit) {   // the copy never landed: raise the error word
            atomicExch(err, 1);
            return;
        }
    }
}

template <int IN, int YMODE>
__global__ void __cluster_dims__(kFCluster, 1, 1) __launch_bounds__(kFThreads, 1)
fused_decode_kernel(const __grid_constant__ FParams prm) {
    constexpr int ES = IN == IN_F32 ? 4 : 2;
    extern __shared__ __align__(128) unsigned char fsmem_raw[];
    FSmem &s = *reinterpret_cast<FSmem *>(fsmem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    const uint32_t rank = f_cluster_rank();
    const int64_t c0 = (int64_t)blockIdx.x * kFChan;
    const int64_t K = kFN, kbytes = kFN / 2;

    // ---- 1. barriers: the weight copy's, and the activation rows' (armed with the
    // bytes of the rows the other CTAs of the cluster will copy in); the cluster
    // barrier's arrive here, its wait before the first copy, orders those copies
    // after every CTA's initialisation ----
    if (threadIdx.x == 0) {
        const uint32_t wb = f_smem_u32(&s.wbar), ab = f_smem_u32(&s.abar);
        const int64_t own = prm.M > rank ? (prm.M - rank + kFCluster - 1) / kFCluster : 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wb) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(ab) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(ab),
                     "r"((uint32_t)((prm.M - own) * (int64_t)sizeof(ARow)))
                     : "memory");
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- 2. this thread's 8 input chunks (row rank + 4 slot, slot = warp / 2),
    // issued before the sign table, whose computation hides their latency ----
    static_assert(IN != IN_F32, "16-bit activations only");
    const int slot = warp >> 1;
    const int64_t row = (int64_t)rank + kFCluster * slot;
    const int t = threadIdx.x & 63, half = t >> 5;
    const bool active = row < prm.M;
    const K4Addr ad = k4_addr(t);                      // thread bases of every access below
    uint4 xg[8];
    {
        const char *xrow = static_cast<const char *>(prm.x) + (active ? row : 0) * prm.ldx * ES + 16 * ad.c1;
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) xg[sl] = __ldg(reinterpret_cast<const uint4 *>(xrow + 128 * sl));
    }
    // the weight scale of this thread's output channel (the epilogue's channel
    // c0 + lane for both of its outputs), fetched now, off the epilogue's path
    const float w_scale = YMODE == 2 ? 0.f : __ldg(prm.sw + c0 + lane);
    for (int j = threadIdx.x; j < kFN / 2; j += kFThreads) {
        const uint32_t a = (uint32_t)(splitmix64_at(prm.seed, 2ull * j) >> 63);
        const uint32_t b = (uint32_t)(splitmix64_at(prm.seed, 2ull * j + 1) >> 63);
        s.sgn[j] = (a << 15) | (b << 31);
    }
    __syncthreads();

    // ---- 3. rotate + quantize row rank + 4 slot ----
    // The same operations in the same order as the 4096-element rotation kernel.
    {
        const uint32_t rbar = 1 + slot;
        const bool signs_first = (prm.flags & 1u) != 0;
        const uint32_t msel = signs_first ? 0xffffffffu : 0u;
        const unsigned full = 0xffffffffu;
        ulonglong2 *buf = s.rowbuf[slot];
        constexpr int NP = 32;
        pair_t v[NP];
        // phase 1: the chunks loaded above, signs, 6 stages
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            const uint4 m = reinterpret_cast<const uint4 *>(s.sgn)[ad.c1 + 8 * sl];
            convert_chunk<IN>(&xg[sl], m, msel, &v[4 * sl]);
        }
        // the activations are in: now the CTA's 32 weight rows (contiguous, 64 KB)
        // in one bulk copy, which would have delayed them in the memory system
        if (threadIdx.x == 0) {
            const uint32_t wb = f_smem_u32(&s.wbar);
            asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(wb),
                         "r"((uint32_t)sizeof(s.w))
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    f_smem_u32(&s.w[0][0])),
                "l"(prm.wq + c0 * kbytes), "r"((uint32_t)sizeof(s.w)), "r"(wb)
                : "memory");
        }
#pragma unroll
        for (int rb = 1; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);
        // transpose 1, phase 2
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            buf[ad.w1 + 16 * sl] = make_ulonglong2(v[4 * sl], v[4 * sl + 1]);
            buf[(ad.w1 ^ 1) + 16 * sl] = make_ulonglong2(v[4 * sl + 2], v[4 * sl + 3]);
        }
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            const ulonglong2 lo = buf[ad.r1 + 128 * sl], hi = buf[(ad.r1 ^ 1) + 128 * sl];
            v[4 * sl] = lo.x; v[4 * sl + 1] = lo.y; v[4 * sl + 2] = hi.x; v[4 * sl + 3] = hi.y;
        }
#pragma unroll
        for (int rb = 3; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);
        // transpose 2, phase 3
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            buf[ad.w2 + 128 * sl] = make_ulonglong2(v[4 * sl], v[4 * sl + 1]);
            buf[(ad.w2 ^ 1) + 128 * sl] = make_ulonglong2(v[4 * sl + 2], v[4 * sl + 3]);
        }
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            const ulonglong2 lo = buf[16 * t + (k4_k3(sl, 0) ^ ad.m3)], hi = buf[16 * t + (k4_k3(sl, 1) ^ ad.m3)];
            v[4 * sl] = lo.x; v[4 * sl + 1] = lo.y; v[4 * sl + 2] = hi.x; v[4 * sl + 3] = hi.y;
        }
#pragma unroll
        for (int rb = 3; rb <= 5; ++rb) butterfly_pairs<NP>(v, rb);
        // row absmax over the two warps
        float amax = pairs_absmax<NP>(v);
#pragma unroll
        for (int k = 0; k < 5; ++k) amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1 << k));
        if (lane == 0) s.red[slot][half] = amax;
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
        amax = fmaxf(s.red[slot][0], s.red[slot][1]);
        // quantize and pack 64 consecutive elements (chunks 8t .. 8t + 7)
        const float inv = amax > 0.f ? 7.0f / amax : 0.f;
        const pair_t inv2 = mk2(inv, inv);
        const pair_t bias2 = mk2(12582912.0f, 12582912.0f);   // 1.5 * 2^23
        if (!signs_first) {                           // signs after the transform: one branch
#pragma unroll
            for (int sl = 0; sl < 8; ++sl) {
                const uint4 m = reinterpret_cast<const uint4 *>(s.sgn)[8 * t + sl];
                const uint32_t mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    v[4 * sl + k] ^= ((pair_t)(mm[k] & 0x80000000u) << 32) | (pair_t)(mm[k] << 16);
            }
        }
        uint32_t words[8];
        int usum = 0;
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
            uint32_t code[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const pair_t qq = fma2(v[4 * sl + k], inv2, bias2);
                code[2 * k] = (uint32_t)qq;
                code[2 * k + 1] = (uint32_t)(qq >> 32);
            }
            words[sl] = pack8(code);
            usum = f_usum(f_ulo(words[sl]), f_uhi(words[sl]), usum);
        }
#pragma unroll
        for (int k = 0; k < 5; ++k) usum += __shfl_xor_sync(full, usum, 1 << k);
        if (lane == 0) s.ured[slot][half] = usum;
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
        usum = s.ured[slot][0] + s.ured[slot][1];
        const float scale = (amax / 7.0f) * (1.0f / 64.0f);
        const uint4 w0 = make_uint4(words[0], words[1], words[2], words[3]);
        const uint4 w1 = make_uint4(words[4], words[5], words[6], words[7]);
        if (active) {
            // the row record in this CTA's shared memory, visible to the async proxy
            const int sw = ((int)row & 1) << 2;
            ARow &ar = s.arow[row];
            ar.q[(2 * t) ^ sw] = w0;
            ar.q[(2 * t + 1) ^ sw] = w1;
            if (t == 0) {
                ar.scale = scale;
                ar.usum = usum;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        asm volatile("bar.sync %0, 64;" ::"r"(rbar) : "memory");
        // every CTA of the cluster has armed its activation barrier
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (active) {
            // one bulk copy of the record into each other CTA of the cluster
            if (t == 0) {
#pragma unroll
                for (uint32_t r = 0; r < kFCluster; ++r)
                    if (r != rank) bulk_to_peer(&s.arow[row], (uint32_t)sizeof(ARow), r, &s.abar);
            }
            if (blockIdx.x < kFCluster) {
                // the first cluster also hands the codes and scales to the caller
                if (prm.aq) {
                    uint4 *qg = reinterpret_cast<uint4 *>(prm.aq + row * kbytes + 32 * t);
                    qg[0] = w0;
                    qg[1] = w1;
                }
                if (prm.as && t == 0) prm.as[row] = scale;
            }
        }
    }

    // ---- 4. wait for the other CTAs' rows, this CTA's own rows and the weights.
    // Arriving on the cluster barrier says "every copy into me has landed"; its wait
    // before exit keeps each CTA's rows alive until all copies out of it are done ----
    f_mbar_wait<true>(&s.abar, 0, prm.err);
    __syncthreads();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    f_mbar_wait<false>(&s.wbar, 0, prm.err);

    // ---- 5. the product over this warp's K slice: rows g, g + 8; channels 8 j + g ----
    float acc[4][4];
    int wsum[4] = {0, 0, 0, 0};
    uint32_t wbytes[4] = {0u, 0u, 0u, 0u};             // byte lanes of u_w sums, <= 8 words x 30
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[j][r] = 0.f;
    const int xsw = (g & 1) << 2;                      // rows g and g + 8 share the XOR
    const int s0 = warp * kFSteps;
#pragma unroll
    for (int u = 0; u < kFSteps; ++u) {
        const int gran = 4 * (s0 + u) + tq;
        const uint4 x0v = s.arow[g].q[gran ^ xsw], x1v = s.arow[g + 8].q[gran ^ xsw];
        uint4 wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = s.w[8 * j + g][gran];
#pragma unroll
        for (int q = 0; q < 4; ++q) {                 // four k32 MMA steps per 128 codes
            const uint32_t x0 = (&x0v.x)[q], x1 = (&x1v.x)[q];
            const uint32_t a[4] = {f_ulo(x0), f_ulo(x1), f_uhi(x0), f_uhi(x1)};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t w = (&wv[j].x)[q];
                const uint32_t b[2] = {f_ulo(w), f_uhi(w)};
                wbytes[j] += b[0] + b[1];
                f_mma_e4m3(acc[j], a, b);
            }
        }
        if (u & 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wsum[j] = (int)__dp4a(wbytes[j], 0x01010101u, (unsigned)wsum[j]);   // unsigned bytes
                wbytes[j] = 0u;
            }
        }
    }

    // ---- 6. split-K reduction and epilogue ----
    auto to_int = [](float v) { return __float2int_rn(v * 262144.0f); };   // exact: x 2^18
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s.part[warp][g][j * 8 + tq * 2] = to_int(acc[j][0]);
        s.part[warp][g][j * 8 + tq * 2 + 1] = to_int(acc[j][1]);
        s.part[warp][g + 8][j * 8 + tq * 2] = to_int(acc[j][2]);
        s.part[warp][g + 8][j * 8 + tq * 2 + 1] = to_int(acc[j][3]);
        int v = wsum[j];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if (tq == 0) s.csum[warp][j * 8 + g] = v;
    }
    __syncthreads();
#pragma unroll
    for (int e = threadIdx.x; e < kFMaxM * kFChan; e += kFThreads) {
        const int mm = e / kFChan, cc = e % kFChan;     // cc == lane
        const int64_t c = c0 + cc;
        if (mm < prm.M) {
            // sum q_a q_w = sum u_a u_w - 8 sum u_a - 8 sum u_w + 64 K
            int sacc = 0, su = s.arow[mm].usum;
#pragma unroll
            for (int w = 0; w < kFWarps; ++w) {
                sacc += s.part[w][mm][cc];
                su += s.csum[w][cc];
            }
            const int a = sacc - 8 * su + 64 * (int)K;
            if (YMODE == 2) {
                static_cast<int *>(prm.y)[mm * prm.N + c] = a;
            } else {
                const float v = ((float)a * s.arow[mm].scale) * w_scale;
                if (YMODE == 1) static_cast<float *>(prm.y)[mm * prm.N + c] = v;
                else static_cast<__half *>(prm.y)[mm * prm.N + c] = __float2half_rn(v);
            }
        }
    }
    // no CTA leaves while a copy out of its shared memory may still be reading it
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int IN, int YMODE>
cudaError_t launch_fused_t(const FParams &p, cudaStream_t stream) {
    auto kern = fused_decode_kernel<IN, YMODE>;
    const size_t smem = sizeof(FSmem);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(p.N / kFChan), kFThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int IN>
cudaError_t launch_fused_in(const FParams &p, int y_mode, cudaStream_t stream) {
    switch (y_mode) {
        case 0: return launch_fused_t<IN, 0>(p, stream);
        case 1: return launch_fused_t<IN, 1>(p, stream);
        default: return launch_fused_t<IN, 2>(p, stream);
    }
}

}  // namespace

bool fused_decode_supported(int64_t M, int64_t K, int64_t N) {
    return M >= 1 && M <= kFMaxM && K == kFN && N > 0 && N % (kFChan * kFCluster) == 0;
}

cudaError_t launch_fused_decode(const void *x, int in_type, int64_t M, int64_t ldx, uint64_t seed, uint32_t flags,
                                const uint8_t *wq, const float *sw, int64_t N, void *y, int y_mode, uint8_t *aq,
                                float *as, cudaStream_t stream) {
    const FParams p{x, ldx, M, N, seed, flags, wq, sw, y, aq, as, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    switch (in_type) {
        case IN_BF16: return launch_fused_in<IN_BF16>(p, y_mode, stream);
        case IN_F16: return launch_fused_in<IN_F16>(p, y_mode, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rq
