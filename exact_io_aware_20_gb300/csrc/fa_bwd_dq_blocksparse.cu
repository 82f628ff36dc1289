// Deterministic dQ under a block mask (block-sparse attention); the kernel is
// in fa_bwd_dq_kernel.cuh, instantiated here with its key-tile list.
#include "fa_bwd_dq_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_dq_blocksparse(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr == nullptr) return cudaErrorInvalidValue;
  return launch_bwd_dq_for<true>(pr, a, stream);
}

}  // namespace fa
