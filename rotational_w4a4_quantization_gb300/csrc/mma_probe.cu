// mma_probe.cu -- rate of the tensor pipe that the W4A4 kernels use (sm_103a).
//
// The W4A4 products run on tcgen05.mma kind::f8f6f4 (E4M3 operands, fp32
// accumulators in tensor memory).  This probe measures that pipe alone: one CTA
// per SM, one thread issuing back-to-back M128 N256 K32 MMAs on operands that sit
// in shared memory (zeros; no data movement), then one commit and a bounded wait.
// The rate it shows, at the clocks of the run that times it, is the ceiling of a
// GEMM that keeps the pipe fed; the GEMM's own rate is reported against it
// alongside the dense peak derived from the measured bf16 GEMM.
#include "rq_internal.h"

#include <cstdint>

namespace rq {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeOperandBytes = 65536;          // A (32 KB) and B (32 KB) regions
constexpr long long kProbeWaitLimit = 4000000000ll;   // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t probe_smem(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// K-major, 128-byte-swizzled operand descriptor (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t probe_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__global__ void __launch_bounds__(kProbeThreads, 1) f8_mma_probe_kernel(long long mmas, int *err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t done;
    uint8_t *ops = smem_raw + ((1024u - (probe_smem(smem_raw) & 1023u)) & 1023u);
    for (int i = threadIdx.x; i < kProbeOperandBytes / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(ops)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(probe_smem(&done)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(probe_smem(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // zeros visible to the tensor core
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    if (threadIdx.x == 0) {
        // kind::f8f6f4, A = B = E4M3, D = F32, K-major, N = 256, M = 128
        constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
        const uint32_t a0 = probe_smem(ops), b0 = probe_smem(ops + kProbeOperandBytes / 2);
        for (long long i = 0; i < mmas; ++i) {
            const uint32_t k = (uint32_t)(i & 3);
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                "l"(probe_desc(a0 + 32 * k)), "l"(probe_desc(b0 + 32 * k)), "r"(idesc), "r"((uint32_t)(i != 0))
                : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         probe_smem(&done))
                     : "memory");
        uint32_t ok = 0;
        const long long t0 = clock64();
        while (!ok) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], 0;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(probe_smem(&done))
                : "memory");
            if (!ok && clock64() - t0 > kProbeWaitLimit) {
                atomicExch(err, 1);
                break;
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
    }
}

}  // namespace

cudaError_t launch_f8_mma_probe(long long mmas_per_sm, int *ctas, cudaStream_t stream) {
    int *err = error_word_device_ptr();
    if (!err) return cudaErrorUnknown;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int smem = kProbeOperandBytes + 1024;
    e = cudaFuncSetAttribute(f8_mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    f8_mma_probe_kernel<<<sms, kProbeThreads, smem, stream>>>(mmas_per_sm, err);
    if (ctas) *ctas = sms;
    return cudaGetLastError();
}

}  // namespace rq
