// Backward pass, dense; the kernels are in fa_bwd_kernel.cuh.
#include "fa_bwd_kernel.cuh"

namespace fa {

int bwd_query_tile(int d) { return d == 256 ? 64 : 128; }

int bwd_list_cap(int d) {
  switch (d) {
    case 64: return Cfg64::kListCap;
    case 128: return Cfg128::kListCap;
    default: return Cfg256::kListCap;
  }
}

cudaError_t launch_bwd(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (a.mask.ptr != nullptr) return launch_bwd_blocksparse(pr, a, stream);
  if (pr.d == 128 && !a.deterministic) return launch_bwd_fused(pr, a, stream);
  if (pr.d == 256) return launch_bwd_pair(pr, a, stream);
  return launch_bwd_for<false>(pr, a, stream);
}

}  // namespace fa
