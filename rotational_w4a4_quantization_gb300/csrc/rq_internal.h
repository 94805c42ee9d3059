// rq_internal.h -- declarations shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace rq {

// Element types of rotation inputs (values match rq_dtype).
enum InType : int { IN_F32 = 0, IN_BF16 = 1, IN_F16 = 2 };

// One rotation+quantization job: `rows` rows of `n` elements, row stride `ld`
// elements, written to packed codes q (row stride n/2 bytes), fp32 scales and
// optionally fp32 rotated rows y.
struct RotJob {
    const void *x;
    int64_t ld;
    int64_t rows;
    uint8_t *q;
    float *scales;
    float *y;
};

// Launch the rotation+quant kernel over up to two jobs of the same n and dtype
// (the KV path passes K and V as two jobs of one launch).
cudaError_t launch_fwht_quant(const RotJob *jobs, int njobs, int log_n, int in_type,
                              uint64_t seed, uint32_t flags, cudaStream_t stream);

// Row lengths n = m 2^k (m in {12, 20, 28}, 2^k in [32, 1024]): R = diag(s) (H_m (x)
// H_{2^k}) / sqrt(n) with Paley blocks H_m.  kron_block_of reports m and k.
bool kron_block_of(int64_t n, int *m, int *logb);
cudaError_t launch_fwht_kron(const RotJob &job, int m, int logb, int in_type, uint64_t seed, uint32_t flags,
                             cudaStream_t stream);

// y_mode: 0 = fp16 out, 1 = fp32 out, 2 = raw int32 accumulators.
struct GemmArgs {
    const uint8_t *a_q;
    const float *a_scales;
    const uint8_t *w_q;
    const float *w_scales;
    int64_t M, N, K;
    void *y;
    int y_mode;
    bool a_e4m3;    // a_q holds one E4M3 operand byte per code ([M][K]), not packed nibbles
};

cudaError_t launch_w4a4_gemm(const GemmArgs &args, cudaStream_t stream);

// Decode-sized products on the tensor cores (M <= 64 tokens, N a multiple of
// 128, K a multiple of 128 up to 8192): weights in tensor memory, split along K
// over a thread-block cluster.
bool w4a4_gemm_decode_tc_supported(const GemmArgs &args);
cudaError_t launch_w4a4_gemm_decode_tc(const GemmArgs &args, cudaStream_t stream);

// Host helpers shared by the tensor-core kernels: a 2-D TMA map over a byte
// matrix (rows x row_bytes, row stride row_bytes) with boxes of box_rows x
// box_bytes; the SM count of the current device (0 on error).
bool make_tma_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t row_bytes, int box_bytes, int box_rows,
                     CUtensorMapSwizzle swizzle);
int device_sm_count();

// Fused decode path (rotation + quantization + W4A4 product in one launch):
// M <= 16 tokens, K in {1024, 2048, 4096, 8192}, N a multiple of 128.
bool fused_decode_supported(int64_t M, int64_t K, int64_t N);
cudaError_t launch_fused_decode(const void *x, int in_type, int64_t M, int64_t ldx, uint64_t seed, uint32_t flags,
                                const uint8_t *wq, const float *sw, int64_t N, int64_t K, void *y, int y_mode,
                                uint8_t *aq, float *as, cudaStream_t stream);

// Attention of decode queries over the rotated INT4 KV cache.
bool attn_decode_supported(int64_t head_dim);
cudaError_t launch_attn_decode(const void *q, int in_type, int64_t M, int64_t heads, int64_t head_dim,
                               const uint8_t *kq, const float *ks, const uint8_t *vq, const float *vs,
                               int64_t tokens, uint64_t seed, uint32_t flags, float softmax_scale, float *out,
                               cudaStream_t stream);

// W4A8 product: INT8 activations, INT4 weights, per-channel (group == K) or
// per-group (group == 128) weight scales.  Per-channel scales with more than 64
// tokens run on the tensor cores (launch_w4a8_gemm_tc), the rest on mma.sync.
bool w4a8_gemm_tc_supported(int64_t M, int64_t N, int64_t K, int y_mode);
cudaError_t launch_w4a8_gemm_tc(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                                int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream);
// Per-group (128) weight scales with more than 64 tokens on the tensor cores:
// N a multiple of 128, K <= 8192, fp16 or fp32 out.
bool w4a8_group_tc_supported(int64_t M, int64_t N, int64_t K, int y_mode);
cudaError_t launch_w4a8_group_tc(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                                 int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream);
// The same kernel for INT4 activations in the product's operand form
// ([M][K] signed E4M3 bytes, sa2 the [M][2] (scale, code sum) pairs): the W4A4
// product with per-group (128) weight scales, under the same shape limits.
cudaError_t launch_w4a4_group_tc(const uint8_t *aq_e4m3, const float *sa2, const uint8_t *wq, const float *sw,
                                 int64_t M, int64_t N, int64_t K, void *y, int y_mode, cudaStream_t stream);
cudaError_t launch_w4a8_gemm(const int8_t *aq, const float *sa, const uint8_t *wq, const float *sw, int64_t M,
                             int64_t N, int64_t K, int64_t group, void *y, int y_mode, cudaStream_t stream);

// One thread waits on a barrier that nothing arrives on, with the rotation
// kernels' bounded wait and the given limit: raises the error word on expiry.
cudaError_t launch_wait_timeout_selftest(long long limit_cycles, cudaStream_t stream);

// Tensor-pipe rate probe: one CTA per SM issues `mmas_per_sm` M128 N256 K32
// kind::f8f6f4 MMAs; *ctas receives the grid size.
cudaError_t launch_f8_mma_probe(long long mmas_per_sm, int *ctas, cudaStream_t stream);

// Device-resident error word set by bounded waits that gave up.
cudaError_t read_and_clear_error_word(int *value, cudaStream_t stream);
int *error_word_device_ptr();

}  // namespace rq
