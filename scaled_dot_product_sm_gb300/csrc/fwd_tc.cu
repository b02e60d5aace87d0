// fwd_tc.cu - the bf16 tensor-core prefill forward's entry point and its
// instantiations without an additive mask (the kernel is in fwd_tc_kernel.cuh).
#include "fwd_tc_kernel.cuh"

namespace sdpa_impl {

cudaError_t launch_fwd_tc_direct_mask(const FwdParams& p, cudaStream_t st);   // fwd_tc_direct.cu
cudaError_t launch_fwd_tc_staged_mask(const FwdParams& p, cudaStream_t st);   // fwd_tc_staged.cu

bool fwd_tc_supported(int E, int Ev) { return (E == 64 || E == 128) && (Ev == 64 || Ev == 128); }

cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t st) {
  if (!p.mask) return launch_mask_mode<kMaskNone>(p, st);
  // the mask base is 16-byte aligned (checked at the boundary); rows of a multiple
  // of 4 keys are 16-byte multiples, as TMA needs
  return (p.S & 3) == 0 ? launch_fwd_tc_staged_mask(p, st) : launch_fwd_tc_direct_mask(p, st);
}

}  // namespace sdpa_impl
