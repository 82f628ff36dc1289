// Backward pass under a block mask (block-sparse attention); the kernels are
// in fa_bwd_kernel.cuh, instantiated here with their step lists.
#include "fa_bwd_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_blocksparse(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr == nullptr) return cudaErrorInvalidValue;
  return launch_bwd_for<true>(pr, a, stream);
}

}  // namespace fa
