// bwd_tc.cu - bf16 backward on the 5th-generation tensor cores (not yet enabled:
// bf16 backward currently runs on the CUDA-core kernels of attn_simt.cu).
#include "common.cuh"

namespace sdpa_impl {

bool bwd_tc_supported(int, int) { return false; }

cudaError_t launch_bwd_tc(const BwdParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sdpa_impl
