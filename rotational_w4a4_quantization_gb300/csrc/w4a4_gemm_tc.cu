// w4a4_gemm_tc.cu -- placeholder until the tensor-core kernel lands.
#include "rq_internal.h"

namespace rq {
bool w4a4_gemm_tc_supported(const GemmArgs &) { return false; }
cudaError_t launch_w4a4_gemm_tc(const GemmArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace rq
