#include "fa_internal.h"
namespace fa {
cudaError_t launch_bwd(const Problem&, const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}
