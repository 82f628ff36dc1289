// Forward pass under a block mask (block-sparse attention); the kernel is in
// fa_fwd_kernel.cuh, instantiated here with its tile list.
#include "fa_fwd_kernel.cuh"

namespace fa {

cudaError_t launch_fwd_blocksparse(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr == nullptr || a.pack || a.splits > 1) return cudaErrorInvalidValue;
  return launch_fwd_for<true>(pr, a, stream);
}

}  // namespace fa
