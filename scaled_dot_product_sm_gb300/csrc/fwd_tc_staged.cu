// fwd_tc_staged.cu - the bf16 tensor-core prefill forward with an additive mask
// staged in shared memory by TMA (rows of a multiple of 4 keys).
#include "fwd_tc_kernel.cuh"

namespace sdpa_impl {

cudaError_t launch_fwd_tc_staged_mask(const FwdParams& p, cudaStream_t st) {
  return launch_mask_mode<kMaskStaged>(p, st);
}

}  // namespace sdpa_impl
