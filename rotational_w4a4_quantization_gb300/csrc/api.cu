// api.cu -- the C ABI (include/rq.h): host-side argument checks, dispatch to the
// kernels, status codes.  Nothing here allocates device memory.
#include "../../include/rq.h"
#include "rq_internal.h"

#include <cstdint>

namespace rq {

cudaError_t launch_w4a4_gemm_small(const GemmArgs &g, cudaStream_t stream);
cudaError_t launch_w4a4_gemm_tc(const GemmArgs &g, cudaStream_t stream);
bool w4a4_gemm_tc_supported(const GemmArgs &g);

namespace {
__device__ int g_error_word;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }
int log2i(int64_t n) {
    int l = 0;
    while ((int64_t(1) << l) < n) ++l;
    return l;
}
int elem_size(rq_dtype t) {
    switch (t) {
        case RQ_F32: return 4;
        case RQ_BF16: return 2;
        case RQ_F16: return 2;
        case RQ_I32: return 4;
    }
    return 0;
}
bool is_rot_input(rq_dtype t) { return t == RQ_F32 || t == RQ_BF16 || t == RQ_F16; }
}  // namespace

int *error_word_device_ptr() {
    int *p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_error_word) != cudaSuccess) return nullptr;
    return p;
}

cudaError_t read_and_clear_error_word(int *value, cudaStream_t stream) {
    int *p = error_word_device_ptr();
    if (!p) return cudaErrorUnknown;
    cudaError_t e = cudaMemcpyAsync(value, p, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*value != 0) {
        const int zero = 0;
        e = cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
    }
    return e;
}

cudaError_t launch_w4a4_gemm(const GemmArgs &g, cudaStream_t stream) {
    if (w4a4_gemm_tc_supported(g)) return launch_w4a4_gemm_tc(g, stream);                 // M > 64
    if (w4a4_gemm_decode_tc_supported(g)) return launch_w4a4_gemm_decode_tc(g, stream);   // M <= 64
    return launch_w4a4_gemm_small(g, stream);   // N not a multiple of 128, or K > 8192
}

}  // namespace rq

extern "C" {

rq_status rq_fwht_quant(const void *x, rq_dtype x_dtype, int64_t rows, int64_t n, int64_t ld_x,
                        uint64_t seed, uint32_t flags, uint8_t *q, float *scales, float *y,
                        void *stream) {
    if (rows < 0 || n <= 0) return RQ_ERR_INVALID_ARG;
    if (!rq::is_rot_input(x_dtype)) return RQ_ERR_UNSUPPORTED;
    int km = 0, klb = 0;   // n = km 2^klb with a Hadamard block of order km (not a power of two)
    const bool kron = !rq::pow2(n) && rq::kron_block_of(n, &km, &klb);
    if (!kron && (!rq::pow2(n) || n < RQ_MIN_N || n > RQ_MAX_N)) return RQ_ERR_UNSUPPORTED;
    if (ld_x < n) return RQ_ERR_INVALID_ARG;
    if (flags & ~uint32_t(RQ_SIGNS_FIRST | RQ_INT8_CODES | RQ_GROUP_SCALES | RQ_E4M3_CODES | RQ_INT4_BYTES))
        return RQ_ERR_INVALID_ARG;
    const uint32_t modes = flags & uint32_t(RQ_INT8_CODES | RQ_GROUP_SCALES | RQ_E4M3_CODES | RQ_INT4_BYTES);
    if (modes & (modes - 1)) return RQ_ERR_INVALID_ARG;   // at most one code mode
    // INT8, INT4-in-bytes and per-group codes: n = m 2^k, n = 128, and powers of two
    // from 256 on (the kernels whose threads end with whole 32-element runs of a
    // row); E4M3 operand codes: n = 128 and powers of two from 256 on
    if (modes && !kron && n < 256 && n != 128) return RQ_ERR_UNSUPPORTED;   // n = 128: the head-sized kernel
    if ((flags & RQ_E4M3_CODES) && kron) return RQ_ERR_UNSUPPORTED;
    if (rows == 0) return RQ_OK;
    if (!x || !q || !scales) return RQ_ERR_INVALID_ARG;
    if (!rq::aligned16(x) || !rq::aligned16(q) || !rq::aligned16(scales) || (y && !rq::aligned16(y)))
        return RQ_ERR_MISALIGNED;
    if ((ld_x * rq::elem_size(x_dtype)) % 16 != 0) return RQ_ERR_MISALIGNED;
    rq::RotJob job{x, ld_x, rows, q, scales, y};
    cudaError_t e = kron ? rq::launch_fwht_kron(job, km, klb, (int)x_dtype, seed, flags,
                                                static_cast<cudaStream_t>(stream))
                         : rq::launch_fwht_quant(&job, 1, rq::log2i(n), (int)x_dtype, seed, flags,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_w4a4_gemm(const uint8_t *a_q, const float *a_scales, const uint8_t *w_q,
                       const float *w_scales, int64_t M, int64_t N, int64_t K, uint64_t seed,
                       uint32_t flags, void *y, rq_dtype y_dtype, void *stream) {
    (void)seed;  // the rotation is already folded into w_q
    if (M < 0 || N < 0 || K <= 0) return RQ_ERR_INVALID_ARG;
    if (flags & ~uint32_t(RQ_A_E4M3 | RQ_GROUP_SCALES)) return RQ_ERR_INVALID_ARG;
    const bool a_e4m3 = (flags & RQ_A_E4M3) != 0;
    const bool group = (flags & RQ_GROUP_SCALES) != 0;
    if (a_e4m3 && M > 0 && M <= 64) return RQ_ERR_UNSUPPORTED;   // the operand form feeds the tensor-core kernel
    if (K % 128 != 0 || K > 65536) return RQ_ERR_UNSUPPORTED;
    if (y_dtype != RQ_F16 && y_dtype != RQ_F32 && y_dtype != RQ_I32) return RQ_ERR_UNSUPPORTED;
    // per-group weight scales: the group kernel, on operand-form activations only
    if (group && (!a_e4m3 || y_dtype == RQ_I32 || N % 128 != 0 || K > 8192)) return RQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return RQ_OK;
    const bool need_scales = y_dtype != RQ_I32;
    const bool need_a = need_scales || a_e4m3;   // the operand form's row code sums sit in a_scales
    if (!a_q || !w_q || !y || (need_a && !a_scales) || (need_scales && !w_scales)) return RQ_ERR_INVALID_ARG;
    if (!rq::aligned16(a_q) || !rq::aligned16(w_q) || !rq::aligned16(y)) return RQ_ERR_MISALIGNED;
    if ((need_a && !rq::aligned16(a_scales)) || (need_scales && !rq::aligned16(w_scales))) return RQ_ERR_MISALIGNED;
    if ((N * rq::elem_size(y_dtype)) % 16 != 0) return RQ_ERR_MISALIGNED;
    if (group) {
        cudaError_t e = rq::launch_w4a4_group_tc(a_q, a_scales, w_q, w_scales, M, N, K, y, y_dtype == RQ_F16 ? 0 : 1,
                                                 static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
    }
    rq::GemmArgs g{a_q, a_scales, w_q, w_scales, M, N, K, y,
                   y_dtype == RQ_F16 ? 0 : (y_dtype == RQ_F32 ? 1 : 2), a_e4m3};
    cudaError_t e = rq::launch_w4a4_gemm(g, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_kv_rotate_quant(const void *k, const void *v, rq_dtype dtype, int64_t tokens,
                             int64_t heads, int64_t head_dim, uint64_t seed, uint32_t flags,
                             uint8_t *kq, float *ks, uint8_t *vq, float *vs, void *stream) {
    if (tokens < 0 || heads <= 0 || head_dim <= 0) return RQ_ERR_INVALID_ARG;
    if (!k && !v) return RQ_ERR_INVALID_ARG;
    if (!rq::is_rot_input(dtype)) return RQ_ERR_UNSUPPORTED;
    if (!rq::pow2(head_dim) || head_dim < RQ_MIN_N || head_dim > 256) return RQ_ERR_UNSUPPORTED;
    if (flags & ~uint32_t(RQ_SIGNS_FIRST)) return RQ_ERR_INVALID_ARG;
    if (tokens == 0) return RQ_OK;
    if ((k && (!kq || !ks)) || (v && (!vq || !vs))) return RQ_ERR_INVALID_ARG;
    const void *ptrs[6] = {k, v, kq, ks, vq, vs};
    for (const void *p : ptrs)
        if (p && !rq::aligned16(p)) return RQ_ERR_MISALIGNED;
    const int64_t rows = tokens * heads;
    rq::RotJob jobs[2];
    int nj = 0;
    if (k) jobs[nj++] = rq::RotJob{k, head_dim, rows, kq, ks, nullptr};
    if (v) jobs[nj++] = rq::RotJob{v, head_dim, rows, vq, vs, nullptr};
    cudaError_t e = rq::launch_fwht_quant(jobs, nj, rq::log2i(head_dim), (int)dtype, seed, flags,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_fwht_quant_gemm(const void *x, rq_dtype x_dtype, int64_t M, int64_t K, int64_t ld_x,
                             uint64_t seed, uint32_t flags, const uint8_t *w_q, const float *w_scales,
                             int64_t N, void *y, rq_dtype y_dtype, uint8_t *a_q, float *a_scales,
                             void *stream) {
    if (M < 0 || N < 0 || K <= 0) return RQ_ERR_INVALID_ARG;
    if (flags & ~uint32_t(RQ_SIGNS_FIRST)) return RQ_ERR_INVALID_ARG;
    if (x_dtype != RQ_BF16 && x_dtype != RQ_F16) return RQ_ERR_UNSUPPORTED;
    if (y_dtype != RQ_F16 && y_dtype != RQ_F32 && y_dtype != RQ_I32) return RQ_ERR_UNSUPPORTED;
    if (ld_x < K) return RQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return RQ_OK;
    if (!rq::fused_decode_supported(M, K, N)) return RQ_ERR_UNSUPPORTED;
    const bool need_scales = y_dtype != RQ_I32;
    if (!x || !w_q || !y || (need_scales && !w_scales)) return RQ_ERR_INVALID_ARG;
    const void *ptrs[6] = {x, w_q, y, w_scales, a_q, a_scales};
    for (const void *p : ptrs)
        if (p && !rq::aligned16(p)) return RQ_ERR_MISALIGNED;
    if ((ld_x * rq::elem_size(x_dtype)) % 16 != 0) return RQ_ERR_MISALIGNED;
    if ((N * rq::elem_size(y_dtype)) % 16 != 0) return RQ_ERR_MISALIGNED;
    const int y_mode = y_dtype == RQ_F16 ? 0 : (y_dtype == RQ_F32 ? 1 : 2);
    cudaError_t e = rq::launch_fused_decode(x, (int)x_dtype, M, ld_x, seed, flags, w_q, w_scales, N, K, y, y_mode,
                                            a_q, a_scales, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_attn_decode(const void *q, rq_dtype q_dtype, int64_t M, int64_t heads, int64_t head_dim,
                         const uint8_t *kq, const float *ks, const uint8_t *vq, const float *vs, int64_t tokens,
                         uint64_t seed, uint32_t flags, float softmax_scale, float *out, void *stream) {
    if (M < 0 || heads < 0 || head_dim <= 0 || tokens < 0) return RQ_ERR_INVALID_ARG;
    if (flags & ~uint32_t(RQ_SIGNS_FIRST | RQ_ATTN_ROTATED_OUT)) return RQ_ERR_INVALID_ARG;
    if (!rq::is_rot_input(q_dtype)) return RQ_ERR_UNSUPPORTED;
    if (!rq::attn_decode_supported(head_dim)) return RQ_ERR_UNSUPPORTED;
    if (M == 0 || heads == 0) return RQ_OK;
    if (tokens < 1) return RQ_ERR_INVALID_ARG;   // a softmax over no tokens is undefined
    if (!q || !kq || !ks || !vq || !vs || !out) return RQ_ERR_INVALID_ARG;
    if (!rq::aligned16(q) || !rq::aligned16(kq) || !rq::aligned16(vq) || !rq::aligned16(out))
        return RQ_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(ks) & 3u) || (reinterpret_cast<uintptr_t>(vs) & 3u)) return RQ_ERR_MISALIGNED;
    if (heads > 65535 / 8 || M > 65535) return RQ_ERR_UNSUPPORTED;   // grid limits: 8 CTAs per head, M rows
    cudaError_t e = rq::launch_attn_decode(q, (int)q_dtype, M, heads, head_dim, kq, ks, vq, vs, tokens, seed, flags,
                                           softmax_scale, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_w4a8_gemm(const int8_t *a_q, const float *a_scales, const uint8_t *w_q, const float *w_scales,
                       int64_t M, int64_t N, int64_t K, int64_t group, void *y, rq_dtype y_dtype, void *stream) {
    if (M < 0 || N < 0 || K <= 0 || group <= 0) return RQ_ERR_INVALID_ARG;
    if (K % 128 != 0 || (group != 128 && group != K)) return RQ_ERR_UNSUPPORTED;
    if (y_dtype != RQ_F16 && y_dtype != RQ_F32 && !(y_dtype == RQ_I32 && group == K)) return RQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return RQ_OK;
    if (!a_q || !w_q || !y || (y_dtype != RQ_I32 && (!a_scales || !w_scales))) return RQ_ERR_INVALID_ARG;
    if (!rq::aligned16(a_q) || !rq::aligned16(w_q) || !rq::aligned16(y)) return RQ_ERR_MISALIGNED;
    if ((a_scales && (reinterpret_cast<uintptr_t>(a_scales) & 3u)) ||
        (w_scales && (reinterpret_cast<uintptr_t>(w_scales) & 3u)))
        return RQ_ERR_MISALIGNED;
    if ((M + 31) / 32 > 65535) return RQ_ERR_UNSUPPORTED;
    const int y_mode = y_dtype == RQ_F16 ? 0 : (y_dtype == RQ_F32 ? 1 : 2);
    cudaError_t e = rq::launch_w4a8_gemm(a_q, a_scales, w_q, w_scales, M, N, K, group, y, y_mode,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_selftest_wait_timeout(int64_t limit_cycles, void *stream) {
    if (limit_cycles < 1000 || limit_cycles > 4000000000ll) return RQ_ERR_INVALID_ARG;
    cudaError_t e = rq::launch_wait_timeout_selftest((long long)limit_cycles, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_probe_f8_mma(int64_t mmas_per_sm, int32_t *ctas, void *stream) {
    if (mmas_per_sm < 1 || mmas_per_sm > (int64_t(1) << 30)) return RQ_ERR_INVALID_ARG;
    int n = 0;
    cudaError_t e = rq::launch_f8_mma_probe((long long)mmas_per_sm, &n, static_cast<cudaStream_t>(stream));
    if (ctas) *ctas = n;
    return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

rq_status rq_sync_status(void *stream) {
    int word = 0;
    cudaError_t e = rq::read_and_clear_error_word(&word, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return RQ_ERR_CUDA;
    return word != 0 ? RQ_ERR_TIMEOUT : RQ_OK;
}

const char *rq_status_string(rq_status s) {
    switch (s) {
        case RQ_OK: return "RQ_OK";
        case RQ_ERR_INVALID_ARG: return "RQ_ERR_INVALID_ARG";
        case RQ_ERR_UNSUPPORTED: return "RQ_ERR_UNSUPPORTED";
        case RQ_ERR_MISALIGNED: return "RQ_ERR_MISALIGNED";
        case RQ_ERR_CUDA: return "RQ_ERR_CUDA";
        case RQ_ERR_TIMEOUT: return "RQ_ERR_TIMEOUT";
    }
    return "RQ_ERR_UNKNOWN";
}

uint32_t rq_version(void) { return (1u << 16) | 0u; }

}  // extern "C"
