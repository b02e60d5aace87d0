// fwd_tc_direct.cu - the bf16 tensor-core prefill forward with an additive mask
// that the softmax threads read from global memory (rows not a multiple of 4 keys).
#include "fwd_tc_kernel.cuh"

namespace sdpa_impl {

cudaError_t launch_fwd_tc_direct_mask(const FwdParams& p, cudaStream_t st) {
  return launch_mask_mode<kMaskDirect>(p, st);
}

}  // namespace sdpa_impl
