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
// Data path per K block of 128 codes (persistent kernel; two 128 x 256 fp32
// accumulators in TMEM, all 512 columns, so tile i's epilogue overlaps tile
// i+1's MMAs): TMA brings the packed tiles into a shared-memory ring, converter
// warps widen them into an operand ring in the 128-byte-swizzled K-major layout
// of the MMA descriptors, one thread issues the MMAs.
//
// Two variants share the code:
//  * CTA pairs (M > 128): a cluster of two CTAs on two SMs computes 256 x 256
//    tiles with tcgen05.mma.cta_group::2 (M256 N256 K32).  Each CTA loads and
//    widens its own 128 rows of A and its own half (128 rows) of the W tile, so
//    every SM converts and serves half of B: a third less shared-memory traffic
//    per MAC than one CTA doing 128 x 256 alone.  The
//    leader CTA issues the MMAs; commits multicast to both CTAs' barriers.  The
//    peer's converter warps arrive on the leader's operand barriers through
//    distributed shared memory with a CTA-scope release: their operands stay in
//    the peer's own shared memory and are read by the peer SM's tensor
//    core, and a cluster-scope release there (it waits for the SM's memory
//    traffic to drain) took longer than the K block's MMAs.  Once per tile the
//    epilogues exchange the halves of the per-column offset terms (cluster-scope
//    release, as the peer's threads read them) and release the accumulator to
//    the leader;
//  * single CTAs (64 < M <= 128): 128 x 256 tiles with cta_group::1.
// Roles in each CTA:
//   warp 0    TMA producer: packed A (128 x 64 B) and W (128 or 256 x 64 B)
//             tiles into a ring (mbarrier transaction counts);
//   warp 1    allocates 512 TMEM columns; one lane (of the leader) issues 4 MMAs
//             per K block into the tile's accumulator and commits them to the
//             operand rings' "empty" barriers and, per tile, to "acc full";
//   warps 2-13 converters, three teams of four (team t takes the K blocks g with
//             g % 3 == t, so each warp has three MMA periods for its block: the
//             widening of one block is a chain of shared-memory loads, ALU work
//             and stores that takes several MMA periods).  A team widens all of
//             its block's A and W chunks.  Each team keeps partial per-row code
//             sums and hands them, and the weight scales, to the epilogue through
//             shared memory.  CTA pairs run four teams (warps 2-17, four MMA
//             periods per block; 4 + 4 stages), single CTAs three;
//   last 4 warps epilogue (one per TMEM lane quarter): tcgen05.ld of the fp32
//             accumulator, offset removal, scales (broadcast from shared memory),
//             16-byte stores.
// The order of k inside each 8-code group is permuted the same way for A and W
// (even codes, then odd codes), which leaves every dot product unchanged.
// Every mbarrier wait is bounded: on expiry the CTA raises the library's error
// word, stops, releases its tensor memory and returns.
//
// W4A8 variant (A8; "SpinQuant" page, The architecture: INT8 activations, INT4
// weights, one scale per output channel).  An INT8 code a splits exactly into
// a = 16 h + l with h = a >> 4 in [-8, 7] and l = a & 15 in [0, 15].  Each
// activation row becomes two operand rows of 4-bit values: row 2i holds
// u = h + 8, row 2i+1 holds u = l, both exact E4M3 bytes as above, so an
// operand tile of 128 rows carries 64 activation rows and both accumulators
// stay exact (sum u u_w <= 225 K).  The epilogue combines the two TMEM lanes of
// a row (adjacent lanes of one warp):
//   sum a q_w = 16 (acc_h - 8 sum u_h + c) + (acc_l - 8 sum u_l),
//   c = 64 K - 8 sum u_w (the W4A4 column term),
// which is sum a u_w - 8 sum a with sum a = sum (16 u_h - 128 + l).  The packed
// A tile of a K block is 64 rows x 128 bytes of int8 codes, the same 8 KB as
// 128 rows x 64 bytes of packed nibbles, so the rings are unchanged.
#include "rq_internal.h"

#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>

namespace rq {
namespace {

constexpr int BM = 128, BN = 256, BK = 128;      // per-CTA A rows, tile columns, K block (codes)
constexpr int kTeamWarps = 4;                     // one per TMEM lane quarter
constexpr int kTeamThreads = 32 * kTeamWarps;
constexpr int kEpiWarps = 4;                      // one per TMEM lane quarter
// producer and MMA warps, `teams` converter teams, epilogue warps
constexpr int threads_tc(int teams) { return 32 * (2 + teams * kTeamWarps + kEpiWarps); }
constexpr uint32_t kTmemCols = 2 * BN;            // two 128 x 256 fp32 accumulators
constexpr long long kWaitLimitCycles = 4000000000ll;    // ~2 s at 2 GHz

// TEAMS converter teams: team t converts the K blocks g with g % TEAMS == t.
template <bool PAIR, int TEAMS = 3>
struct Cfg {
    static_assert(TEAMS == 3 || (TEAMS == 4 && PAIR), "four teams only fit the shared memory of CTA pairs");
    static constexpr int kTeams = TEAMS, kConvWarps = TEAMS * kTeamWarps, kThreads = threads_tc(TEAMS);
    static constexpr int NCTA = PAIR ? 2 : 1;
    static constexpr int WROWS = BN / NCTA;         // W rows (output channels) per CTA
    static constexpr int TILE_M = BM * NCTA;        // output rows per tile
    // Stage counts and the team rotation must keep every mbarrier parity wait at
    // most one phase ahead of its barrier: a packed stage is owned by one team
    // (PK_STAGES a multiple of kTeams, so the phase before the one a team waits
    // for is its own finished block), and MMA commits complete in order, so an
    // operand-ring wait is safe with OP_STAGES >= kTeams.
    // The packed ring is the deeper one: it covers the TMA latency from L2/HBM
    // (6 + 3 stages ran the prefill GEMM ~7% faster than 3 + 5).  Four teams need
    // four operand stages, which leaves room for only four packed ones.
    static constexpr int PK_STAGES = TEAMS == 4 ? 4 : (PAIR ? 2 * kTeams : kTeams), OP_STAGES = TEAMS;
    static constexpr int PK_A = BM * BK / 2, PK_W = WROWS * BK / 2;   // packed bytes per stage
    static constexpr int OP_A = BM * BK, OP_W = WROWS * BK;           // e4m3 bytes per stage
    static constexpr int NACH = BM * (BK / 32) / kTeamThreads;       // A chunks per thread and K block
    static constexpr int NWCH = WROWS * (BK / 32) / kTeamThreads;    // W chunks per thread and K block
    static_assert(WROWS * (BK / 32) % kTeamThreads == 0, "W chunks split evenly");
    static_assert(PK_STAGES % kTeams == 0 && OP_STAGES >= kTeams, "parity waits stay one phase ahead at most");
};

template <bool PAIR, int TEAMS = 3, bool AE = false>
struct Smem {
    using C = Cfg<PAIR, TEAMS>;
    static constexpr bool kPair = PAIR;
    alignas(1024) uint8_t opA[C::OP_STAGES][C::OP_A];
    alignas(1024) uint8_t opW[C::OP_STAGES][C::OP_W];
    alignas(128) uint8_t pkA[C::PK_STAGES][AE ? 16 : C::PK_A];   // AE: A goes straight into opA
    alignas(128) uint8_t pkW[C::PK_STAGES][C::PK_W];
    alignas(16) int rowsum[2][BM];       // per tile parity: sum_k u_a (the teams add in; the epilogue clears)
    alignas(16) int colsum[2][BN];       // the same for sum_k u_w, this CTA's W rows
    alignas(16) int colterm[2][BN];      // 64 K - 8 * sum_k u_w, all columns of the tile
    alignas(16) float wscale[2][BN];     // weight scales of the tile's columns
    alignas(8) uint64_t pk_full[C::PK_STAGES];
    uint64_t pk_empty[C::PK_STAGES];
    uint64_t op_full[C::OP_STAGES];      // (leader) both CTAs' converter warps
    uint64_t op_empty[C::OP_STAGES];     // MMA commit (multicast to both CTAs)
    uint64_t acc_full[2], acc_empty[2];  // acc_empty (leader): both CTAs' epilogues
    uint64_t sum_full[2], sum_empty[2];  // own converters -> own epilogue and back
    uint64_t col_full[2];                // colterm complete: own and (pair) the peer's epilogue warps
    uint64_t a_full[C::OP_STAGES];       // AE: this CTA's operand tile of A landed (TMA)
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

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

// Arrive on the barrier at the same offset in CTA `rank` of the cluster (the own
// CTA included), with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cta(const uint64_t *b, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(b)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Arrival on another CTA's barrier with release at CTA scope only: for operands
// that the arriving CTA wrote into its own shared or tensor memory for its own
// SM's tensor core (made visible to it by fence.proxy.async / tcgen05.wait::st
// beforehand).  A cluster-scope release would wait for the SM's memory traffic
// to drain, which costs more than a K block's MMAs.
__device__ __forceinline__ void mbar_arrive_remote_cta_scope(const uint64_t *b, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(b)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}

// CLUSTER: acquire at cluster scope, for barriers that other CTAs (or the pair's
// multicast MMA commits) arrive on; CTA scope otherwise.
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, uint32_t parity) {
    uint32_t ok;
    if constexpr (CLUSTER) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(b)), "r"(parity)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(b)), "r"(parity)
            : "memory");
    }
    return ok != 0;
}

// Bounded wait: returns false (and raises the abort flag and the error word) if
// the phase does not complete in time or another role has aborted.  SLEEP backs
// off with __nanosleep between polls: for the roles with slack (the producer,
// the epilogue), whose polling would otherwise take issue and shared-memory pipe
// slots from the converter warps of the same SM sub-partition.
template <bool CLUSTER = false, bool SLEEP = false, class S>
__device__ __forceinline__ bool mbar_wait(S &s, uint64_t *b, uint32_t parity, int *err) {
    if (mbar_try_wait<CLUSTER>(b, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if constexpr (SLEEP) __nanosleep(128);
        if (mbar_try_wait<CLUSTER>(b, parity)) return true;
        if (s.abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            s.abort_flag = 1;
            atomicExch(err, 1);
            return false;
        }
    }
}

// Warp-wide wait on a barrier that the pair's multicast MMA commit releases: one
// cluster-scope acquire per warp, and __syncwarp orders the other lanes after it.
template <class S>
__device__ __forceinline__ bool warp_wait_commit(S &s, uint64_t *b, uint32_t parity, int lane, int *err) {
    if constexpr (S::kPair) {
        int got = 1;
        if (lane == 0) got = mbar_wait<true>(s, b, parity, err);
        __syncwarp();
        return __shfl_sync(0xffffffffu, got, 0) != 0;
    } else {
        return mbar_wait(s, b, parity, err);
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

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, both K-major, N = 256.
template <bool PAIR>
constexpr uint32_t idesc() {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
           ((uint32_t)(Cfg<PAIR>::TILE_M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, K = 32.
template <bool PAIR>
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    if constexpr (PAIR) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc<PAIR>()), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc<PAIR>()), "r"(accumulate)
            : "memory");
    }
}

// Signal `bar` when the MMAs issued so far complete: in every CTA of the pair.
template <bool PAIR>
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    if constexpr (PAIR) {
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                smem_u32(bar)),
            "h"((uint16_t)3)
            : "memory");
    } else {
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                     : "memory");
    }
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

template <bool PAIR>
__device__ __forceinline__ void cluster_sync() {
    if constexpr (PAIR) {
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
        __syncthreads();
    }
}

// Store NV consecutive outputs of row m from column nb on: raw sums (YMODE 2),
// or acc * sa * sw in fp32 (1) or fp16 (0); groups that would cross N are
// skipped (N * element size is a multiple of 16 bytes).
template <int YMODE, int NV>
__device__ __forceinline__ void store_outputs(void *y, int64_t N, int64_t m, int64_t nb, const int (&acc)[NV],
                                              const float *ws, float sa) {
    const float4 *ws4 = reinterpret_cast<const float4 *>(ws);
    if (YMODE == 2) {
        int *yr = static_cast<int *>(y) + m * N + nb;
#pragma unroll
        for (int j = 0; j < NV; j += 4)
            if (nb + j + 3 < N) *reinterpret_cast<int4 *>(yr + j) = make_int4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    } else if (YMODE == 1) {
        float *yr = static_cast<float *>(y) + m * N + nb;
#pragma unroll
        for (int j = 0; j < NV; j += 4) {
            if (nb + j + 3 >= N) continue;
            const float4 w4 = ws4[j / 4];
            float4 o;
            o.x = ((float)acc[j] * sa) * w4.x;
            o.y = ((float)acc[j + 1] * sa) * w4.y;
            o.z = ((float)acc[j + 2] * sa) * w4.z;
            o.w = ((float)acc[j + 3] * sa) * w4.w;
            *reinterpret_cast<float4 *>(yr + j) = o;
        }
    } else {
        __half *yr = static_cast<__half *>(y) + m * N + nb;
#pragma unroll
        for (int j = 0; j < NV; j += 8) {
            if (nb + j + 7 >= N) continue;
            __align__(16) __half h[8];
            const float4 wa = ws4[j / 4], wb = ws4[j / 4 + 1];
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) h[e2] = __float2half_rn(((float)acc[j + e2] * sa) * wv[e2]);
            *reinterpret_cast<uint4 *>(yr + j) = *reinterpret_cast<const uint4 *>(h);
        }
    }
}

// AE: the activation codes arrive in the operand form (one signed E4M3 byte per
// code, rq_fwht_quant with RQ_E4M3_CODES, whose scales carry each row's code sum
// S_a): lane 1 of warp 0 loads each K block's 128 x 128-byte A tile by TMA with
// the 128-byte swizzle straight into the operand ring (completing on a_full),
// the converters widen only W, to u_w = q_w + 8 as for the packed path, and wait
// for a_full before releasing the operand stage.  Products q_a u_w 2^-18 and
// their sums (|.| <= 120 K 2^-18) are exact; the epilogue subtracts 8 S_a.
template <int YMODE, bool PAIR, bool A8, int TEAMS, bool AE = false>
__global__ void __launch_bounds__(threads_tc(TEAMS), 1)
w4a4_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
               const __grid_constant__ TcParams prm) {
    using C = Cfg<PAIR, TEAMS>;
    using S = Smem<PAIR, TEAMS, AE>;
    constexpr int kTeams = C::kTeams, kConvWarps = C::kConvWarps;
    static_assert(!A8 || PAIR, "the W4A8 variant runs on CTA pairs");
    static_assert(!(A8 && AE), "one activation form");
    extern __shared__ uint8_t smem_raw[];
    // align by offsetting the shared array itself, so the compiler keeps the
    // shared address space (plain LDS/STS instead of generic accesses)
    S &s = *reinterpret_cast<S *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_rank() : 0;
    const int kblocks = (int)(prm.K / BK);
    const int64_t n_tiles_n = (prm.N + BN - 1) / BN;
    const int64_t m_op = A8 ? 2 * prm.M : prm.M;     // operand rows (two per INT8 activation row)
    // Tiles run M-fastest: the CTAs working at the same time cover every row tile
    // of a few column tiles, so those weight columns and all of A stay in L2
    // (row-major order streamed W from DRAM once per row tile).
    const int64_t n_tiles_m = (m_op + C::TILE_M - 1) / C::TILE_M;
    const int64_t n_tiles = n_tiles_n * n_tiles_m;
    const int64_t first_tile = blockIdx.x / C::NCTA, tile_step = gridDim.x / C::NCTA;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::PK_STAGES; ++i) {
            mbar_init(&s.pk_full[i], 1);
            mbar_init(&s.pk_empty[i], kTeamWarps);
        }
        for (int i = 0; i < C::OP_STAGES; ++i) {
            mbar_init(&s.op_full[i], kTeamWarps * C::NCTA);
            mbar_init(&s.op_empty[i], 1);
            mbar_init(&s.a_full[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], kEpiWarps * C::NCTA);
            mbar_init(&s.sum_full[i], kConvWarps);
            mbar_init(&s.sum_empty[i], kEpiWarps);
            mbar_init(&s.col_full[i], kEpiWarps * C::NCTA);
        }
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int i = threadIdx.x; i < 2 * BM; i += blockDim.x) (&s.rowsum[0][0])[i] = 0;
    for (int i = threadIdx.x; i < 2 * BN; i += blockDim.x) (&s.colsum[0][0])[i] = 0;
    if (warp == 1) {
        if constexpr (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&s.tmem_base)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&s.tmem_base)),
                         "r"(kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync<PAIR>();    // barriers initialized and TMEM allocated in both CTAs
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int64_t g = 0;                                   // global K-block counter
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
                // A rows of this CTA: 128 packed rows, or (A8) 64 INT8 rows
                const int m0 = A8 ? (int)(tile % n_tiles_m) * (C::TILE_M / 2) + (int)rank * (BM / 2)
                                  : (int)(tile % n_tiles_m) * C::TILE_M + (int)rank * BM;
                const int n0 = (int)(tile / n_tiles_m) * BN + (int)rank * C::WROWS;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int st = (int)(g % C::PK_STAGES);
                    if (!mbar_wait<false, true>(s, &s.pk_empty[st], (uint32_t)((g / C::PK_STAGES) & 1) ^ 1, prm.err)) { ok = false; break; }
                    mbar_expect_tx(&s.pk_full[st], (AE ? 0 : C::PK_A) + C::PK_W);
                    if constexpr (!AE) tma_load_2d(s.pkA[st], &tmA, &s.pk_full[st], kb * (A8 ? BK : BK / 2), m0);
                    tma_load_2d(s.pkW[st], &tmW, &s.pk_full[st], kb * (BK / 2), n0);
                }
            }
        } else if (AE && lane == 1) {
            // operand-form A: each K block's tile into the operand ring once the
            // MMAs that last read that stage are done
            int64_t g = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
                const int m0 = (int)(tile % n_tiles_m) * C::TILE_M + (int)rank * BM;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int os = (int)(g % C::OP_STAGES);
                    if (!mbar_wait<PAIR, true>(s, &s.op_empty[os], (uint32_t)((g / C::OP_STAGES) & 1) ^ 1, prm.err)) { ok = false; break; }
                    mbar_expect_tx(&s.a_full[os], C::OP_A);
                    tma_load_2d(s.opA[os], &tmA, &s.a_full[os], kb * BK, m0);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader CTA of a pair) ----------------
        if (lane == 0 && rank == 0) {
            int64_t g = 0;
            int it = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step, ++it) {
                const int buf = it & 1;
                // the epilogues must have drained this accumulator (two tiles ago)
                if (!mbar_wait<PAIR>(s, &s.acc_empty[buf], (uint32_t)((it >> 1) & 1) ^ 1, prm.err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + (uint32_t)(buf * BN);
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int st = (int)(g % C::OP_STAGES);
                    if (!mbar_wait<PAIR>(s, &s.op_full[st], (uint32_t)((g / C::OP_STAGES) & 1), prm.err)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = smem_u32(s.opA[st]), w0 = smem_u32(s.opW[st]);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_f8<PAIR>(d, sw128_desc(a0 + 32 * k), sw128_desc(w0 + 32 * k), (kb | k) != 0);
                    mma_commit<PAIR>(&s.op_empty[st]);
                }
                if (ok) mma_commit<PAIR>(&s.acc_full[buf]);
            }
        }
    } else if (warp < 2 + kConvWarps) {
        // ---------------- converters ----------------
        const int tc = threadIdx.x - 64;                  // 0..383
        const int team = (warp - 2) / kTeamWarps;         // K blocks with g % kTeams == team
        // chunk tt + 128 j of a stage = row (tt >> 2) + 32 j, 16-byte chunk tt & 3
        const int tt = tc - kTeamThreads * team;
        const int ch = tt & 3, rq = tt >> 2;
        int64_t g = 0;
        int it = 0;
        bool ok = true;
        for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step, ++it) {
            const int n0 = (int)(tile / n_tiles_m) * BN;
            // the tile's weight scale for column tc, loaded now so that its latency
            // is not on the converters' path at the end of the tile
            const float wsc = (YMODE != 2 && tc < BN && n0 + tc < prm.N) ? prm.sw[n0 + tc] : 0.f;
            // A8: sumA holds the rows' sum of u_h, sumL their sum of u_l
            uint32_t sumA[C::NACH], sumL[A8 ? C::NACH : 1], sumW[C::NWCH];
#pragma unroll
            for (int j = 0; j < C::NACH; ++j) sumA[j] = 0;
#pragma unroll
            for (int j = 0; j < (A8 ? C::NACH : 1); ++j) sumL[j] = 0;
#pragma unroll
            for (int j = 0; j < C::NWCH; ++j) sumW[j] = 0;
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                if ((int)(g % kTeams) != team) continue;
                const int ps = (int)(g % C::PK_STAGES);
                const int os = (int)(g % C::OP_STAGES);
                if (!mbar_wait(s, &s.pk_full[ps], (uint32_t)((g / C::PK_STAGES) & 1), prm.err)) { ok = false; break; }
                uint4 a[AE ? 1 : C::NACH], w[C::NWCH];
                if constexpr (!AE) {
#pragma unroll
                    for (int j = 0; j < C::NACH; ++j) a[j] = reinterpret_cast<const uint4 *>(s.pkA[ps])[tt + kTeamThreads * j];
                }
#pragma unroll
                for (int j = 0; j < C::NWCH; ++j) w[j] = reinterpret_cast<const uint4 *>(s.pkW[ps])[tt + kTeamThreads * j];
                if (!warp_wait_commit(s, &s.op_empty[os], (uint32_t)((g / C::OP_STAGES) & 1) ^ 1, lane, prm.err)) { ok = false; break; }
                // row, chunk ch -> 32 e4m3 bytes = granules 2ch, 2ch+1 of the 128-byte row
                auto emit = [&](uint8_t *base, int row, const uint4 &v, uint32_t &sum) {
                    uint32_t lo[4], hi[4], acc = 0;
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc += widen(wv[i], lo[i], hi[i]);
                    sum = __dp4a(acc, 0x01010101u, sum);
                    uint8_t *rowp = base + row * 128;
                    const int g0 = (2 * ch) ^ (row & 7), g1 = (2 * ch + 1) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(rowp + 16 * g0) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
                    *reinterpret_cast<uint4 *>(rowp + 16 * g1) = make_uint4(lo[2], hi[2], lo[3], hi[3]);
                };
                if constexpr (AE) {
                    // A is in place by TMA (a_full below)
                } else if constexpr (A8) {
                    // INT8 chunk tt + 128 j = row (tt >> 3) + 16 j, codes 16 c .. 16 c + 15
                    // with c = tt & 7 -> granule c of operand rows 2 row (u_h) and
                    // 2 row + 1 (u_l), in the even-then-odd order of the W side
                    const int c = tt & 7;
#pragma unroll
                    for (int j = 0; j < C::NACH; ++j) {
                        const uint4 &v = a[j];
                        const uint32_t p[4] = {__byte_perm(v.x, v.y, 0x6420u), __byte_perm(v.x, v.y, 0x7531u),
                                               __byte_perm(v.z, v.w, 0x6420u), __byte_perm(v.z, v.w, 0x7531u)};
                        uint32_t h[4], l[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            h[i] = ((p[i] >> 4) & 0x0f0f0f0fu) ^ 0x08080808u;   // h + 8 = top nibble, sign bit flipped
                            l[i] = p[i] & 0x0f0f0f0fu;
                        }
                        sumA[j] = __dp4a(h[0] + h[1] + h[2] + h[3], 0x01010101u, sumA[j]);   // byte lanes <= 60
                        sumL[j] = __dp4a(l[0] + l[1] + l[2] + l[3], 0x01010101u, sumL[j]);
                        const int r2 = 2 * ((tt >> 3) + 16 * j);
                        uint8_t *rowp = s.opA[os] + r2 * 128;
                        *reinterpret_cast<uint4 *>(rowp + 16 * (c ^ (r2 & 7))) = make_uint4(h[0], h[1], h[2], h[3]);
                        *reinterpret_cast<uint4 *>(rowp + 128 + 16 * (c ^ ((r2 + 1) & 7))) =
                            make_uint4(l[0], l[1], l[2], l[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C::NACH; ++j) emit(s.opA[os], rq + 32 * j, a[j], sumA[j]);
                }
                if constexpr (AE) {
                    // W as u = q + 8 (one XOR per word, no sums: the activation
                    // row sums arrive with the activation scales), the even codes
                    // of each word first (the operand order of the activation bytes)
#pragma unroll
                    for (int j = 0; j < C::NWCH; ++j) {
                        const int row = rq + 32 * j;
                        uint8_t *rowp = s.opW[os] + row * 128;
                        const uint4 &v = w[j];
                        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
                        uint32_t lo[4], hi[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) widen(wv[i], lo[i], hi[i]);
                        const int g0 = (2 * ch) ^ (row & 7), g1 = (2 * ch + 1) ^ (row & 7);
                        *reinterpret_cast<uint4 *>(rowp + 16 * g0) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
                        *reinterpret_cast<uint4 *>(rowp + 16 * g1) = make_uint4(lo[2], hi[2], lo[3], hi[3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C::NWCH; ++j) emit(s.opW[os], rq + 32 * j, w[j], sumW[j]);
                }
                // AE: this CTA's A tile must be in place before the stage is released to the MMA
                if constexpr (AE) {
                    if (!mbar_wait(s, &s.a_full[os], (uint32_t)((g / C::OP_STAGES) & 1), prm.err)) { ok = false; break; }
                }
                // One proxy fence per thread orders its generic reads of the packed
                // stage before the next TMA refill of it (or the refill can overtake
                // them) and its operand stores before the tensor core's reads; then
                // one lane per warp releases both stages (the operand stage at the
                // leader for a pair).
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.pk_empty[ps]);
                    if (rank == 0) mbar_arrive(&s.op_full[os]);
                    else mbar_arrive_remote_cta_scope(&s.op_full[os], 0);
                }
            }
            if (!ok) break;
            // row sums: the four lanes sharing a row hold its four chunks (A8: the
            // eight lanes sharing an INT8 row hold its eight chunks)
#pragma unroll
            for (int j = 0; j < C::NACH; ++j) {
                sumA[j] += __shfl_xor_sync(0xffffffffu, sumA[j], 1);
                sumA[j] += __shfl_xor_sync(0xffffffffu, sumA[j], 2);
                if constexpr (A8) {
                    sumA[j] += __shfl_xor_sync(0xffffffffu, sumA[j], 4);
                    sumL[j] += __shfl_xor_sync(0xffffffffu, sumL[j], 1);
                    sumL[j] += __shfl_xor_sync(0xffffffffu, sumL[j], 2);
                    sumL[j] += __shfl_xor_sync(0xffffffffu, sumL[j], 4);
                }
            }
#pragma unroll
            for (int j = 0; j < C::NWCH; ++j) {
                sumW[j] += __shfl_xor_sync(0xffffffffu, sumW[j], 1);
                sumW[j] += __shfl_xor_sync(0xffffffffu, sumW[j], 2);
            }
            // add this team's partial sums for the own epilogue, and hand it the
            // weight scales (for a pair, the epilogue passes this CTA's half of
            // the column terms on to the peer)
            const int buf = it & 1;
            if (!mbar_wait(s, &s.sum_empty[buf], (uint32_t)((it >> 1) & 1) ^ 1, prm.err)) { ok = false; break; }
            if constexpr (AE) {
                // the row terms come from the activation row sums (epilogue)
            } else if constexpr (A8) {
                if ((tt & 7) == 0) {
#pragma unroll
                    for (int j = 0; j < C::NACH; ++j) {
                        const int r2 = 2 * ((tt >> 3) + 16 * j);
                        atomicAdd(&s.rowsum[buf][r2], (int)sumA[j]);
                        atomicAdd(&s.rowsum[buf][r2 + 1], (int)sumL[j]);
                    }
                }
            } else if (ch == 0) {
#pragma unroll
                for (int j = 0; j < C::NACH; ++j) atomicAdd(&s.rowsum[buf][rq + 32 * j], (int)sumA[j]);
            }
            if (!AE && ch == 0) {
#pragma unroll
                for (int j = 0; j < C::NWCH; ++j) atomicAdd(&s.colsum[buf][rq + 32 * j], (int)sumW[j]);
            }
            if (YMODE != 2 && tc < BN) s.wscale[buf][tc] = wsc;
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.sum_full[buf]);
        }
    } else {
        // ---------------- epilogue: TMEM -> offset removal -> scales -> global ----------------
        const int e = threadIdx.x - 64 - 32 * kConvWarps;   // 0..127
        const int q = warp & 3;                              // TMEM lane quarter this warp may read
        int it = 0;
        for (int64_t tile = first_tile; tile < n_tiles; tile += tile_step, ++it) {
            const int buf = it & 1;
            const uint32_t par = (uint32_t)((it >> 1) & 1);
            if (!mbar_wait<PAIR, true>(s, &s.acc_full[buf], par, prm.err)) break;
            if (!mbar_wait<false, true>(s, &s.sum_full[buf], par, prm.err)) break;
            // this CTA's column terms (the sums are cleared for the tile after next)
            for (int cl = e; cl < C::WROWS; cl += 32 * kEpiWarps) {
                const int v = AE ? 0 : 64 * (int)prm.K - 8 * s.colsum[buf][cl];
                s.colsum[buf][cl] = 0;
                const int col = (int)rank * C::WROWS + cl;
                s.colterm[buf][col] = v;
                if constexpr (PAIR) {
                    // the peer's epilogue needs this half of the columns too
                    uint32_t remote;
                    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                                 : "=r"(remote)
                                 : "r"(smem_u32(&s.colterm[buf][col])), "r"(rank ^ 1u));
                    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
                }
            }
            // Every epilogue warp of both CTAs arrives once the column terms it wrote
            // are in place (at the peer with a cluster-scope release: generic data
            // read by the peer's threads).  Both epilogues are past this tile's
            // acc_full, so both have finished the tile that last used this buffer.
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s.col_full[buf]);
                if constexpr (PAIR) mbar_arrive_cta(&s.col_full[buf], rank ^ 1u);
            }
            if (!mbar_wait<PAIR, true>(s, &s.col_full[buf], par, prm.err)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // operand rows of this CTA; output row m (A8: two operand rows per row)
            const int64_t m0 = (tile % n_tiles_m) * C::TILE_M + (int64_t)rank * BM, n0 = (tile / n_tiles_m) * BN;
            const int mr = 32 * q + lane;
            const int64_t m = A8 ? (m0 + mr) >> 1 : m0 + mr;
            int rowt;
            float sa;
            if constexpr (AE) {
                // sum_k q_a (q_w + 8) = sum_k q_a q_w + 8 S_a: the pair (scale, S_a)
                // of row m (S_a exact in fp32)
                const float2 p = m < prm.M ? reinterpret_cast<const float2 *>(prm.sa)[m] : make_float2(0.f, 0.f);
                rowt = -8 * (int)p.y;
                sa = p.x;
            } else {
                rowt = -8 * s.rowsum[buf][mr];
                s.rowsum[buf][mr] = 0;
                sa = (YMODE != 2 && m < prm.M) ? prm.sa[m] : 0.f;
            }
            // A8: the u_l lane (odd) takes no column term; its partner adds 16 x its own
            const bool odd = A8 && (lane & 1);
            const int cmask = odd ? 0 : -1;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = 32 * c;
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * BN + col0), r);
                if (A8 || m < prm.M) {
                    int acc[32];
                    const int4 *ct = reinterpret_cast<const int4 *>(&s.colterm[buf][col0]);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const int4 c4 = ct[j / 4];
                        const int cv[4] = {c4.x & cmask, c4.y & cmask, c4.z & cmask, c4.w & cmask};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int u = __float2int_rn(__uint_as_float(r[j + i]) * 262144.0f);   // exact: x 2^18
                            acc[j + i] = u + rowt + cv[i];
                        }
                    }
                    if constexpr (A8) {
                        // the even lane outputs columns col0 .. col0 + 15, the odd lane
                        // the next 16: each sends the partner the half it outputs
                        int out[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int mine = odd ? acc[j + 16] : acc[j];
                            const int recv = __shfl_xor_sync(0xffffffffu, odd ? acc[j] : acc[j + 16], 1);
                            out[j] = odd ? 16 * recv + mine : 16 * mine + recv;
                        }
                        const int cb = col0 + (odd ? 16 : 0);
                        if (m < prm.M) store_outputs<YMODE, 16>(prm.y, prm.N, m, n0 + cb, out, &s.wscale[buf][cb], sa);
                    } else {
                        store_outputs<YMODE, 32>(prm.y, prm.N, m, n0 + col0, acc, &s.wscale[buf][col0], sa);
                    }
                }
            }
            // this accumulator and these offset terms may be reused
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cta(&s.acc_empty[buf], 0);
                else mbar_arrive(&s.acc_empty[buf]);
                mbar_arrive(&s.sum_empty[buf]);
            }
        }
    }

    __syncwarp();            // lanes that skipped a single-lane role wait for it here
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync<PAIR>();    // all MMAs done and all TMEM reads finished in both CTAs
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if constexpr (PAIR) {
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
        } else {
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
        }
    }
}

// ---------------------------------------------------------------------------
// W4A8 with one weight scale per group of 128 codes along K ("SpinQuant" page,
// The architecture: per-group scales), for more than 64 tokens:
//   y[m][c] = sa[m] * sum_g sw[c][g] * sum_{k in g} a[m][k] q[c][k].
// The group scale multiplies each K block's exact partial, so a block's product
// cannot stay in one running accumulator as in the per-channel kernel.  Here:
//  * codes widen to E4M3 with their sign (sign bit plus |q| <= 8 as u 2^-9, all
//    exact), so a partial needs no offset terms; INT8 activations split as in
//    the A8 variant (a = 16 h + l: row 2i holds h with its sign, row 2i+1 l);
//  * the MMA (CTA pairs, M256 N128 K32) writes each K block into a fresh
//    partial in a 4-deep TMEM ring (all 512 columns);
//  * the epilogue warps (four per TMEM lane quarter, 32 columns each) read a
//    partial, release it, and add sw[c][g] x partial into running sums kept in
//    registers (32 per thread), so each block costs one TMEM load per warp and
//    no store.  The release is a CTA-scope arrive on the leader's barrier: the
//    warp only read tensor memory (ordered by tcgen05.fence), and a cluster-scope
//    release per warp and block stalled the epilogue on memory barriers.  Two
//    converter teams take alternate K blocks.  After the last block the two
//    rows of an activation row (adjacent TMEM lanes) combine as 16 S_h + S_l,
//    times 2^18 and sa[m];
//  * the tile's group scales (128 columns x K/128 groups, K <= 8192) are staged
//    in shared memory by the epilogue threads with cp.async, one tile ahead,
//    transposed to [group][column] so that a block's 32 columns are 8 vector
//    loads.  Barriers sc_full (the copies landed) and sc_empty (every epilogue
//    warp is done with a buffer) order the two buffers; every wait is bounded.
// ---------------------------------------------------------------------------
constexpr int GBN = 128;                   // tile columns
constexpr int GWROWS = GBN / 2;            // W rows (output channels) per CTA of the pair
constexpr int GPK = 4, GOP = 4, GPR = 4;   // packed stages, operand stages, TMEM partial ring
constexpr int GTEAMS = 2;                  // converter teams, taking alternate K blocks
constexpr int GEPI = 16;                   // epilogue warps: four per TMEM lane quarter, 32 columns each
constexpr int GTHREADS = 32 * (2 + GTEAMS * kTeamWarps + GEPI);
constexpr int GMAXG = 64;                  // groups staged per column: K <= 8192
static_assert(GPR * GBN <= 512, "TMEM budget");
static_assert(GPK % GTEAMS == 0 && GOP >= GTEAMS, "parity waits stay one phase ahead at most");

struct GSmem {
    static constexpr bool kPair = true;
    alignas(1024) uint8_t opA[GOP][BM * BK];            // 128 operand rows of E4M3
    alignas(1024) uint8_t opW[GOP][GWROWS * BK];        // 64 W rows of E4M3
    alignas(128) uint8_t pkA[GPK][(BM / 2) * BK];       // 64 INT8 rows x 128 bytes
    alignas(128) uint8_t pkW[GPK][GWROWS * BK / 2];     // 64 packed W rows x 64 bytes
    alignas(16) float gsc[2][GMAXG * GBN];              // group scales [g][column], two tiles
    alignas(8) uint64_t pk_full[GPK], pk_empty[GPK];
    uint64_t op_full[GOP], op_empty[GOP];               // op_full at the leader: both CTAs' teams
    uint64_t p_full[GPR], p_empty[GPR];                 // p_empty at the leader: both CTAs' epilogues
    uint64_t sc_full[2], sc_empty[2];                   // own epilogue threads / warps
    uint64_t a_full[GOP];                               // AE: this CTA's operand tile of A landed (TMA)
    uint32_t tmem_base;
    volatile int abort_flag;
};

struct GParams {
    const float *sa, *sw;   // sw: [N][K/128]
    void *y;
    int64_t M, N, K;
    int *err;
};

// kind::f8f6f4, E4M3 x E4M3 -> F32, K-major, M = 256 (CTA pair), N = 128.
constexpr uint32_t idesc_pair_n128() { return (1u << 4) | ((uint32_t)(GBN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24); }

__device__ __forceinline__ void mma_f8_pair_n128(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc_pair_n128()), "r"(acc)
        : "memory");
}

// 16 columns of the warp's 32 TMEM lanes, one register each, behind its wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Byte lanes holding 4-bit two's-complement codes (0..15) -> E4M3 bytes of the
// same signed value times 2^-9: |q| <= 8 in bits 0..3, the sign in bit 7.
__device__ __forceinline__ uint32_t nib_to_e4m3_signed(uint32_t x) {
    const uint32_t one = (x >> 3) & 0x01010101u;                  // 1 in the negative lanes
    return (x ^ (one * 0x8fu)) + one;                              // 0x80 | (15 - x) + 1 there
}

// Store 16 final values of row m from column nb on (fp16 or fp32); N is a
// multiple of 128.
template <int YMODE>
__device__ __forceinline__ void store16_f(void *y, int64_t N, int64_t m, int64_t nb, const float (&v)[16]) {
    if (YMODE == 1) {
        float4 *yr = reinterpret_cast<float4 *>(static_cast<float *>(y) + m * N + nb);
#pragma unroll
        for (int j = 0; j < 4; ++j) yr[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
        uint4 *yr = reinterpret_cast<uint4 *>(static_cast<__half *>(y) + m * N + nb);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            __align__(16) __half h[8];
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) h[e2] = __float2half_rn(v[8 * j + e2]);
            yr[j] = *reinterpret_cast<const uint4 *>(h);
        }
    }
}

// AE: INT4 activation codes in the product's operand form (rq_fwht_quant with
// RQ_E4M3_CODES: signed E4M3 bytes, scales as (scale, code sum) pairs).  Lane 1
// of warp 0 loads each K block's 128 x 128-byte A tile by TMA straight into the
// operand ring (completing on a_full), the converters widen only W, and each
// TMEM lane is one activation row (no INT8 halves): tiles of 256 activation
// rows per pair, half the MMA rows and epilogue work per output of the INT8
// path.  The sums are not needed: the weights widen with their sign.
template <int YMODE, bool AE = false>
__global__ void __launch_bounds__(GTHREADS, 1)
w4a8_group_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ GParams prm) {
    constexpr int kConvWarps = GTEAMS * kTeamWarps;
    constexpr int PK_A = (BM / 2) * BK, PK_W = GWROWS * BK / 2;
    extern __shared__ uint8_t smem_raw[];
    GSmem &s = *reinterpret_cast<GSmem *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int kblocks = (int)(prm.K / BK);                    // = groups
    const int64_t n_tiles_n = prm.N / GBN;
    constexpr int kRowsPerTile = AE ? 2 * BM : BM;                  // activation rows per tile (pair)
    const int64_t n_tiles_m = (prm.M + kRowsPerTile - 1) / kRowsPerTile;
    const int64_t n_tiles = n_tiles_n * n_tiles_m;                  // run M-fastest (L2 reuse of W)
    const int64_t first_tile = blockIdx.x / 2, tile_step = gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < GPK; ++i) {
            mbar_init(&s.pk_full[i], 1);
            mbar_init(&s.pk_empty[i], kTeamWarps);
        }
        for (int i = 0; i < GOP; ++i) {
            mbar_init(&s.op_full[i], kTeamWarps * 2);
            mbar_init(&s.op_empty[i], 1);
        }
        for (int i = 0; i < GPR; ++i) {
            mbar_init(&s.p_full[i], 1);
            mbar_init(&s.p_empty[i], GEPI * 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.sc_full[i], GBN);      // the 128 staging threads
            mbar_init(&s.sc_empty[i], GEPI);
        }
        for (int i = 0; i < GOP; ++i) mbar_init(&s.a_full[i], 1);
        s.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s.tmem_base)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync<true>();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int64_t g = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
                const int m0 = (int)(tile % n_tiles_m) * BM + (int)rank * (BM / 2);   // INT8 rows
                const int n0 = (int)(tile / n_tiles_m) * GBN + (int)rank * GWROWS;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int st = (int)(g % GPK);
                    if (!mbar_wait<false, true>(s, &s.pk_empty[st], (uint32_t)((g / GPK) & 1) ^ 1, prm.err)) { ok = false; break; }
                    mbar_expect_tx(&s.pk_full[st], (AE ? 0 : PK_A) + PK_W);
                    if constexpr (!AE) tma_load_2d(s.pkA[st], &tmA, &s.pk_full[st], kb * BK, m0);
                    tma_load_2d(s.pkW[st], &tmW, &s.pk_full[st], kb * (BK / 2), n0);
                }
            }
        } else if (AE && lane == 1) {
            // operand-form A: each K block's tile into the operand ring once the
            // MMAs that last read that stage are done
            int64_t g = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
                const int m0 = (int)(tile % n_tiles_m) * (2 * BM) + (int)rank * BM;
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int os = (int)(g % GOP);
                    if (!mbar_wait<true, true>(s, &s.op_empty[os], (uint32_t)((g / GOP) & 1) ^ 1, prm.err)) { ok = false; break; }
                    mbar_expect_tx(&s.a_full[os], BM * BK);
                    tma_load_2d(s.opA[os], &tmA, &s.a_full[os], kb * BK, m0);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader CTA): one fresh partial per K block ----------------
        if (lane == 0 && rank == 0) {
            int64_t g = 0;
            bool ok = true;
            for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
                for (int kb = 0; kb < kblocks; ++kb, ++g) {
                    const int pr = (int)(g % GPR), st = (int)(g % GOP);
                    if (!mbar_wait<true>(s, &s.p_empty[pr], (uint32_t)((g / GPR) & 1) ^ 1, prm.err)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    if (!mbar_wait<true>(s, &s.op_full[st], (uint32_t)((g / GOP) & 1), prm.err)) { ok = false; break; }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + (uint32_t)(pr * GBN);
                    const uint32_t a0 = smem_u32(s.opA[st]), w0 = smem_u32(s.opW[st]);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        mma_f8_pair_n128(d, sw128_desc(a0 + 32 * k), sw128_desc(w0 + 32 * k), k != 0);
                    mma_commit<true>(&s.op_empty[st]);
                    mma_commit<true>(&s.p_full[pr]);
                }
            }
        }
    } else if (warp < 2 + kConvWarps) {
        // ---------------- converters: signed E4M3 ----------------
        const int tc = threadIdx.x - 64;
        const int team = (warp - 2) / kTeamWarps;
        const int tt = tc - kTeamThreads * team;
        const int ch = tt & 3, rq = tt >> 2;        // W: row rq + 32 j (j < 2), 16-byte chunk ch
        const int c8 = tt & 7, r8 = tt >> 3;        // A: INT8 row r8 + 16 j (j < 4), 16-code chunk c8
        int64_t g = 0;
        bool ok = true;
        for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step) {
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                if ((int)(g % GTEAMS) != team) continue;
                const int ps = (int)(g % GPK), os = (int)(g % GOP);
                if (!mbar_wait(s, &s.pk_full[ps], (uint32_t)((g / GPK) & 1), prm.err)) { ok = false; break; }
                uint4 a[AE ? 1 : 4], w[2];
                if constexpr (!AE) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[j] = reinterpret_cast<const uint4 *>(s.pkA[ps])[tt + kTeamThreads * j];
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) w[j] = reinterpret_cast<const uint4 *>(s.pkW[ps])[tt + kTeamThreads * j];
                if (!warp_wait_commit(s, &s.op_empty[os], (uint32_t)((g / GOP) & 1) ^ 1, lane, prm.err)) { ok = false; break; }
#pragma unroll
                for (int j = 0; j < (AE ? 0 : 4); ++j) {
                    const uint4 &v = a[j];
                    const uint32_t p[4] = {__byte_perm(v.x, v.y, 0x6420u), __byte_perm(v.x, v.y, 0x7531u),
                                           __byte_perm(v.z, v.w, 0x6420u), __byte_perm(v.z, v.w, 0x7531u)};
                    uint32_t h[4], l[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        h[i] = nib_to_e4m3_signed((p[i] >> 4) & 0x0f0f0f0fu);   // h = a >> 4, a 4-bit code
                        l[i] = p[i] & 0x0f0f0f0fu;                              // l = a & 15 >= 0
                    }
                    const int r2 = 2 * (r8 + 16 * j);
                    uint8_t *rowp = s.opA[os] + r2 * 128;
                    *reinterpret_cast<uint4 *>(rowp + 16 * (c8 ^ (r2 & 7))) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4 *>(rowp + 128 + 16 * (c8 ^ ((r2 + 1) & 7))) = make_uint4(l[0], l[1], l[2], l[3]);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t wv[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        lo[i] = nib_to_e4m3_signed(wv[i] & 0x0f0f0f0fu);          // even codes
                        hi[i] = nib_to_e4m3_signed((wv[i] >> 4) & 0x0f0f0f0fu);   // odd codes
                    }
                    const int row = rq + 32 * j;
                    uint8_t *rowp = s.opW[os] + row * 128;
                    const int g0 = (2 * ch) ^ (row & 7), g1 = (2 * ch + 1) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(rowp + 16 * g0) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
                    *reinterpret_cast<uint4 *>(rowp + 16 * g1) = make_uint4(lo[2], hi[2], lo[3], hi[3]);
                }
                // AE: this CTA's A tile must be in place before the stage is released to the MMA
                if constexpr (AE) {
                    if (!mbar_wait(s, &s.a_full[os], (uint32_t)((g / GOP) & 1), prm.err)) { ok = false; break; }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.pk_empty[ps]);
                    if (rank == 0) mbar_arrive(&s.op_full[os]);
                    else mbar_arrive_remote_cta_scope(&s.op_full[os], 0);
                }
            }
        }
    } else {
        // ---------------- epilogue: scale and add the partials, then combine and store ----------------
        const int e = threadIdx.x - 64 - 32 * kConvWarps;   // 0..511; threads e < 128 stage column e's scales
        const int q = warp & 3;                              // TMEM lane quarter
        const int part = e >> 7;                             // columns 32 part .. 32 part + 31
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const bool odd = (lane & 1) != 0;
        const int G = kblocks;
        // copy the group scales of `tile`'s column e into buffer b (transposed to [g][column]);
        // the thread's arrival on sc_full[b] fires when its copies have landed
        auto stage = [&](int64_t tile, int b) {
            const float *src = prm.sw + ((tile / n_tiles_m) * GBN + e) * (int64_t)G;
            float *dst = s.gsc[b] + e;
            for (int gg = 0; gg < G; ++gg)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst + gg * GBN)), "l"(src + gg)
                             : "memory");
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&s.sc_full[b]))
                         : "memory");
        };
        int64_t g = 0;
        int it = 0;
        bool ok = true;
        if (first_tile < n_tiles && e < GBN) {
            if (!mbar_wait<false, true>(s, &s.sc_empty[0], 1u, prm.err)) ok = false;   // fresh: passes at once
            else stage(first_tile, 0);
        }
        for (int64_t tile = first_tile; tile < n_tiles && ok; tile += tile_step, ++it) {
            const int b = it & 1;
            if (!mbar_wait<false, true>(s, &s.sc_full[b], (uint32_t)((it >> 1) & 1), prm.err)) break;
            // stage the next tile into the other buffer once every epilogue warp is done with it
            const int64_t nt = tile + tile_step;
            if (nt < n_tiles && e < GBN) {
                if (!mbar_wait<false, true>(s, &s.sc_empty[b ^ 1], (uint32_t)(((it + 1) >> 1) & 1) ^ 1, prm.err)) break;
                stage(nt, b ^ 1);
            }
            const int64_t m0 = (tile % n_tiles_m) * (2 * BM) + (int64_t)rank * BM;   // operand rows
            // activation row: one per TMEM lane (AE), or one per two lanes (INT8 halves)
            const int64_t m = AE ? m0 + 32 * q + lane : (m0 + 32 * q + lane) >> 1;
            const int64_t n0 = (tile / n_tiles_m) * GBN;
            // x 2^18: partials are 2^-18 units; AE scales are (scale, code sum) pairs
            const float sa = m < prm.M ? prm.sa[AE ? 2 * m : m] * 262144.0f : 0.f;
            float acc[32];   // the running sums of this thread's row, columns 32 part .. 32 part + 31
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = 0.f;
            for (int kb = 0; kb < kblocks; ++kb, ++g) {
                const int pr = (int)(g % GPR);
                if (!mbar_wait<true, false>(s, &s.p_full[pr], (uint32_t)((g / GPR) & 1), prm.err)) { ok = false; break; }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const float4 *sc4 = reinterpret_cast<const float4 *>(s.gsc[b] + kb * GBN + 32 * part);
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // two 16-column halves: fewer live registers
                    uint32_t pv[16];
                    tmem_ld16(tmem + lane_base + (uint32_t)(pr * GBN + 32 * part + 16 * h), pv);
                    if (h == 1) {
                        // the partial may be overwritten: it was only read (tensor memory, ordered
                        // by the fence), so a CTA-scope release is enough, as for the operands
                        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive_remote_cta_scope(&s.p_empty[pr], 0);
                    }
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 w4 = sc4[(16 * h + j) / 4];
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            acc[16 * h + j + i] = fmaf(wv[i], __uint_as_float(pv[j + i]), acc[16 * h + j + i]);
                    }
                }
            }
            if (ok && AE) {
                // one activation row per lane: all 32 columns
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float out[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) out[j] = acc[16 * h + j] * sa;
                    if (m < prm.M) store16_f<YMODE>(prm.y, prm.N, m, n0 + 32 * part + 16 * h, out);
                }
            } else if (ok) {
                // rows 2i (h) and 2i+1 (l) are lanes 2i, 2i+1: the even lane outputs the
                // chunk's first 16 columns, the odd lane the next 16
                float out[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float mine = odd ? acc[j + 16] : acc[j];
                    const float recv = __shfl_xor_sync(0xffffffffu, odd ? acc[j] : acc[j + 16], 1);
                    out[j] = (odd ? fmaf(16.f, recv, mine) : fmaf(16.f, mine, recv)) * sa;
                }
                if (m < prm.M) store16_f<YMODE>(prm.y, prm.N, m, n0 + 32 * part + (odd ? 16 : 0), out);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.sc_empty[b]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy into shared memory outlives the CTA
    }

    __syncwarp();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync<true>();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
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

bool make_map(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int box_bytes, int box_rows,
              CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SM count of the current device (0 on error).
int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// A8: a_q holds M rows of K int8 codes (TMA boxes of 64 rows x 128 bytes), and a
// tile spans 128 activation rows.
template <int YMODE, bool PAIR, bool A8 = false, int TEAMS = 3, bool AE = false>
cudaError_t launch_mode(const GemmArgs &g, const TcParams &p, cudaStream_t stream) {
    using C = Cfg<PAIR, TEAMS>;
    CUtensorMap ta, tw;
    // AE: 128 rows x 128 bytes of operand-form codes, with the 128-byte swizzle of
    // the MMA's K-major operand layout
    const bool a_ok = AE ? make_map(&ta, g.a_q, g.M, g.K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B)
                         : (A8 ? make_map(&ta, g.a_q, g.M, g.K, BK, BM / 2, CU_TENSOR_MAP_SWIZZLE_NONE)
                               : make_map(&ta, g.a_q, g.M, g.K / 2, BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE));
    if (!a_ok || !make_map(&tw, g.w_q, g.N, g.K / 2, BK / 2, C::WROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kern = w4a4_tc_kernel<YMODE, PAIR, A8, TEAMS, AE>;
    const size_t smem = sizeof(Smem<PAIR, TEAMS, AE>) + 1024;
    // set on every launch: the attribute is per device, and a process may use several
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const int64_t m_op = A8 ? 2 * p.M : p.M;
    const int64_t tiles = ((p.N + BN - 1) / BN) * ((m_op + C::TILE_M - 1) / C::TILE_M);
    // persistent: one CTA per SM (one pair per two SMs)
    const int64_t units = tiles < sms / C::NCTA ? tiles : sms / C::NCTA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * C::NCTA));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::NCTA;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tw, p);
}

// Converter teams for CTA pairs: four.  Four teams give each warp four MMA
// periods per K block but leave room for only four packed stages, a ring depth
// that covers the TMA latency while the operands come from L2.  With tiles walked
// M-fastest the CTAs working at once share their weight columns in L2 at every
// size measured: 2048 x 4096 -> 14336 102.4 us (three teams ~106 us), 4096 x
// 8192 -> 28672 676 us (three teams 739 us).

template <int YMODE, bool AE = false>
cudaError_t launch_group_mode(const CUtensorMap &ta, const CUtensorMap &tw, const GParams &p, cudaStream_t stream) {
    auto kern = w4a8_group_tc_kernel<YMODE, AE>;
    const size_t smem = sizeof(GSmem) + 1024;
    // set on every launch: the attribute is per device, and a process may use several
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorUnknown;
    const int64_t rows_per_tile = AE ? 2 * BM : BM;
    const int64_t tiles = (p.N / GBN) * ((p.M + rows_per_tile - 1) / rows_per_tile);
    const int64_t units = tiles < sms / 2 ? tiles : sms / 2;   // persistent CTA pairs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * 2));
    cfg.blockDim = dim3(GTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tw, p);
}

}  // namespace

bool make_tma_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int box_bytes, int box_rows,
                     CUtensorMapSwizzle swizzle) {
    return make_map(map, base, rows, row_bytes, box_bytes, box_rows, swizzle);
}

int device_sm_count() { return sm_count(); }

bool w4a4_gemm_tc_supported(const GemmArgs &g) { return g.M > 64 && g.K % BK == 0 && g.K <= 65536; }

cudaError_t launch_w4a4_gemm_tc(const GemmArgs &g, cudaStream_t stream) {
    TcParams p{g.a_scales, g.w_scales, g.y, g.M, g.N, g.K, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    const bool pair = g.M > BM;   // tiles of 256 rows on SM pairs; one SM for M <= 128
    const bool t4 = pair;         // four converter teams on pairs (single CTAs: no room)
    if (g.a_e4m3) {
        switch (g.y_mode * 2 + (pair ? 1 : 0)) {
            case 0: return launch_mode<0, false, false, 3, true>(g, p, stream);
            case 1: return launch_mode<0, true, false, 4, true>(g, p, stream);
            case 2: return launch_mode<1, false, false, 3, true>(g, p, stream);
            case 3: return launch_mode<1, true, false, 4, true>(g, p, stream);
            case 4: return launch_mode<2, false, false, 3, true>(g, p, stream);
            default: return launch_mode<2, true, false, 4, true>(g, p, stream);
        }
    }
    switch (g.y_mode * 3 + (pair ? (t4 ? 2 : 1) : 0)) {
        case 0: return launch_mode<0, false>(g, p, stream);
        case 1: return launch_mode<0, true>(g, p, stream);
        case 2: return launch_mode<0, true, false, 4>(g, p, stream);
        case 3: return launch_mode<1, false>(g, p, stream);
        case 4: return launch_mode<1, true>(g, p, stream);
        case 5: return launch_mode<1, true, false, 4>(g, p, stream);
        case 6: return launch_mode<2, false>(g, p, stream);
        case 7: return launch_mode<2, true>(g, p, stream);
        default: return launch_mode<2, true, false, 4>(g, p, stream);
    }
}

bool w4a8_gemm_tc_supported(int64_t M, int64_t N, int64_t K, int y_mode) {
    const int64_t elem = y_mode == 0 ? 2 : 4;
    return M > 64 && K % BK == 0 && K <= 65536 && (N * elem) % 16 == 0;
}

bool w4a8_group_tc_supported(int64_t M, int64_t N, int64_t K, int y_mode) {
    return M > 64 && K % BK == 0 && K / BK <= GMAXG && N % GBN == 0 && y_mode != 2;
}

cudaError_t launch_w4a8_group_tc(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                                 int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream) {
    const GParams p{sa, sw, y, M, N, K, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    CUtensorMap ta, tw;
    if (!make_map(&ta, aq, M, K, BK, BM / 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tw, wq, N, K / 2, BK / 2, GWROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    return y_mode == 1 ? launch_group_mode<1>(ta, tw, p, stream) : launch_group_mode<0>(ta, tw, p, stream);
}

cudaError_t launch_w4a4_group_tc(const uint8_t *aq_e4m3, const float *sa2, const uint8_t *wq, const float *sw,
                                 int64_t M, int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream) {
    const GParams p{sa2, sw, y, M, N, K, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    CUtensorMap ta, tw;
    // 128 rows x 128 bytes of operand-form codes with the 128-byte swizzle of the
    // MMA's K-major operand layout
    if (!make_map(&ta, aq_e4m3, M, K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tw, wq, N, K / 2, BK / 2, GWROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    return y_mode == 1 ? launch_group_mode<1, true>(ta, tw, p, stream) : launch_group_mode<0, true>(ta, tw, p, stream);
}

cudaError_t launch_w4a8_gemm_tc(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                                int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream) {
    const GemmArgs g{reinterpret_cast<const uint8_t *>(aq), sa, wq, sw, M, N, K, y, y_mode};
    TcParams p{sa, sw, y, M, N, K, error_word_device_ptr()};
    if (!p.err) return cudaErrorUnknown;
    // M > 64: at least 130 operand rows, so always CTA pairs, with four teams
    const bool t4 = true;
    switch (y_mode * 2 + (t4 ? 1 : 0)) {
        case 0: return launch_mode<0, true, true>(g, p, stream);
        case 1: return launch_mode<0, true, true, 4>(g, p, stream);
        case 2: return launch_mode<1, true, true>(g, p, stream);
        case 3: return launch_mode<1, true, true, 4>(g, p, stream);
        case 4: return launch_mode<2, true, true>(g, p, stream);
        default: return launch_mode<2, true, true, 4>(g, p, stream);
    }
}

}  // namespace rq
