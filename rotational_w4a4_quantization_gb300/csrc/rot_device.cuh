// rot_device.cuh -- device helpers shared by the rotation kernels: SplitMix64
// signs, fp32 pairs in 64-bit registers with packed f32x2 arithmetic, the
// butterflies of the Sylvester Hadamard network, row absmax, INT4 packing, and
// the three-phase layout of a 4096-element row (two warps, 64 values per
// thread).  Internal linkage: every translation unit gets its own copy.
#pragma once

#include "rq_internal.h"

#include <cuda_fp16.h>

#include <cstdint>

namespace rq {
namespace {

__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    // SplitMix64 (Steele, Lea, Flood 2014): output i is the mix of seed + (i+1)*gamma.
    uint64_t z = seed + (i + 1ull) * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// ---- fp32 pairs in 64-bit registers (low word = even element) ----
using pair_t = unsigned long long;

__device__ __forceinline__ pair_t add2(pair_t a, pair_t b) {
    pair_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ pair_t sub2(pair_t a, pair_t b) {
    pair_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ pair_t fma2(pair_t a, pair_t b, pair_t c) {
    pair_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ pair_t mk2(float lo, float hi) {
    pair_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float lo2(pair_t p) { return __uint_as_float((uint32_t)p); }
__device__ __forceinline__ float hi2(pair_t p) { return __uint_as_float((uint32_t)(p >> 32)); }
// butterfly inside a pair: (x, y) -> (x + y, x - y)
__device__ __forceinline__ pair_t bfly_in(pair_t p) {
    pair_t r;
    asm("{\n\t.reg .f32 x, y, s, d;\n\t"
        "mov.b64 {x, y}, %1;\n\t"
        "add.rn.f32 s, x, y;\n\t"
        "sub.rn.f32 d, x, y;\n\t"
        "mov.b64 %0, {s, d};\n\t}"
        : "=l"(r) : "l"(p));
    return r;
}
// bf16x2 word (x0 low, x1 high) -> (x0 + x1, x0 - x1) in fp32, the first
// butterfly stage fused with the widening.
__device__ __forceinline__ pair_t bf16w_bfly(uint32_t w) {
    pair_t r;
    asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 x1, s, d;\n\t"
        "mov.b32 {l, h}, %1;\n\t"
        "and.b32 x1, %1, 0xffff0000;\n\t"
        "add.rn.f32.bf16 s, l, x1;\n\t"
        "sub.rn.f32.bf16 d, l, x1;\n\t"
        "mov.b64 %0, {s, d};\n\t}"
        : "=l"(r) : "r"(w));
    return r;
}

// max |y| over the values of v: eight independent running maxima and a tree at the
// end (a single running maximum is a serial chain as long as v).
template <int NP>
__device__ __forceinline__ float pairs_absmax(const pair_t (&v)[NP]) {
    constexpr int A = NP < 8 ? NP : 8;
    float m[A];
#pragma unroll
    for (int j = 0; j < A; ++j) m[j] = fmaxf(fabsf(lo2(v[j])), fabsf(hi2(v[j])));
#pragma unroll
    for (int i = A; i < NP; ++i) m[i % A] = fmaxf(m[i % A], fmaxf(fabsf(lo2(v[i])), fabsf(hi2(v[i]))));
#pragma unroll
    for (int w = A / 2; w >= 1; w /= 2)
#pragma unroll
        for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
    return m[0];
}

// Butterflies over register-element bit rb >= 1 of v (pairs pi and pi ^ 2^(rb-1)).
template <int NP>
__device__ __forceinline__ void butterfly_pairs(pair_t (&v)[NP], int rb) {
    const int st = 1 << (rb - 1);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        if (!(i & st)) {
            const pair_t a = v[i], b = v[i + st];
            v[i] = add2(a, b);
            v[i + st] = sub2(a, b);
        }
    }
}

// One chunk (8 elements, 4 pairs) from its raw granule(s): signs (bit 15 / bit 31
// of mask word k flip element 2k / 2k+1; msel = ~0 applies them, 0 skips them,
// one three-input logic op either way), widening, and the in-pair butterfly.
template <int IN>
__device__ __forceinline__ void convert_chunk(const uint4 *g, uint4 m, uint32_t msel, pair_t *out) {
    const uint32_t mm[4] = {m.x & msel, m.y & msel, m.z & msel, m.w & msel};
    if constexpr (IN == IN_F32) {
        const uint32_t w[8] = {g[0].x, g[0].y, g[0].z, g[0].w, g[1].x, g[1].y, g[1].z, g[1].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t e0 = w[2 * k] ^ (mm[k] << 16);
            const uint32_t e1 = w[2 * k + 1] ^ (mm[k] & 0x80000000u);
            out[k] = bfly_in(mk2(__uint_as_float(e0), __uint_as_float(e1)));
        }
    } else {
        const uint32_t w[4] = {g[0].x, g[0].y, g[0].z, g[0].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t x = w[k] ^ mm[k];
            if constexpr (IN == IN_BF16) {
                out[k] = bf16w_bfly(x);
            } else {
                const __half2 h = *reinterpret_cast<const __half2 *>(&x);
                const float2 f = __half22float2(h);
                out[k] = bfly_in(mk2(f.x, f.y));
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

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
// The operand form of four codes, each the low byte of a word (two's complement,
// |q| <= 7): one E4M3 byte per code with the code's sign and |q| as |q| 2^-9.
// Gather the bytes, then turn each negative one into sign and magnitude (a
// selector nibble with bit 3 set replicates the sign of its byte, so `neg`
// holds 0xff in the bytes of negative codes).  The four codes are also added to
// `sum` (a signed byte dot product with ones): the operand form carries each
// row's code sum, the offset term of the W4A4 product.
__device__ __forceinline__ uint32_t e4m3_word_sum(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, int &sum) {
    const uint32_t x = prmt_b32(prmt_b32(c0, c1, 0x0040u), prmt_b32(c2, c3, 0x0040u), 0x5410u);
    sum = __dp4a((int)x, 0x01010101, sum);
    const uint32_t neg = prmt_b32(x, 0u, 0xba98u);
    return (x ^ (neg & 0x7f7f7f7fu)) + (neg & 0x01010101u);
}

__device__ __forceinline__ int k4_chunk1(int t, int s) {
    return (t & 7) | (s << 3) | (((t >> 3) & 3) << 6) | ((t >> 5) << 8);
}
__device__ __forceinline__ int k4_chunk2(int t, int s) { return (t & 63) | (s << 6); }
__device__ __forceinline__ int k4_chunk3(int t, int s) { return (t << 3) | s; }
__device__ __forceinline__ int k4_pos1(int c, int h) { return (2 * c + h) ^ ((c >> 2) & 1); }
__device__ __forceinline__ int k4_pos2(int c, int h) {
    return (2 * c + h) ^ ((((c >> 2) ^ (c >> 5)) & 1) | (((c >> 3) & 1) << 1) | (((c >> 4) & 1) << 2));
}

// Per-thread parts of the maps above (t = 0..63).  The swizzle XORs of the first
// transpose and of the second one's write side take thread bits only, so those
// granule positions are a thread base plus 16 s or 128 s; the second transpose's
// read side XORs slot bit 2 as well, leaving one XOR with a thread constant per
// access:
//   k4_chunk1(t, s)           == c1 + 8 s
//   k4_pos1(k4_chunk1(t,s),h) == (w1 ^ h) + 16 s
//   k4_pos1(k4_chunk2(t,s),h) == (r1 ^ h) + 128 s
//   k4_pos2(k4_chunk2(t,s),h) == (w2 ^ h) + 128 s
//   k4_pos2(k4_chunk3(t,s),h) == 16 t + (k4_k3(s, h) ^ m3)
struct K4Addr {
    int c1, w1, r1, w2, m3;
};
__device__ __forceinline__ K4Addr k4_addr(int t) {
    const int x2 = (t >> 2) & 1;
    K4Addr a;
    a.c1 = k4_chunk1(t, 0);
    a.w1 = 2 * a.c1 + x2;
    a.r1 = 2 * t + x2;
    a.w2 = (2 * t) ^ ((((t >> 2) ^ (t >> 5)) & 1) | (((t >> 3) & 1) << 1) | (((t >> 4) & 1) << 2));
    a.m3 = x2 | ((t & 1) << 1) | (((t >> 1) & 1) << 2);
    return a;
}
__host__ __device__ constexpr int k4_k3(int s, int h) { return (2 * s + h) ^ ((s >> 2) & 1); }

}  // namespace
}  // namespace rq
