// Forward pass, dense (causal or not, with or without key-axis splits); the
// kernel is in fa_fwd_kernel.cuh.
#include "fa_fwd_kernel.cuh"

namespace fa {

int fwd_key_tile(int) { return 128; }

cudaError_t launch_fwd(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr != nullptr) return launch_fwd_blocksparse(pr, a, stream);
  return launch_fwd_for<false>(pr, a, stream);
}

}  // namespace fa
