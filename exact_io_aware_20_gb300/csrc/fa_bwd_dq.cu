// Deterministic dQ, dense; the kernel is in fa_bwd_dq_kernel.cuh.
#include "fa_bwd_dq_kernel.cuh"

namespace fa {

cudaError_t launch_bwd_dq(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr != nullptr) return launch_bwd_dq_blocksparse(pr, a, stream);
  return launch_bwd_dq_for<false>(pr, a, stream);
}

}  // namespace fa
