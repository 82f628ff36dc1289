// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// fa_bwd needs scratch (the fp32 row vector D and the fp32 dQ accumulator)
// and asks the caller for it.  Some callers have no way to provide it: a
// plugin whose host interface hands over only input and output buffers, or
// a process whose device memory is fixed at start-up and which must not call
// cudaMalloc (or any allocating library routine) afterwards.  This entry
// point takes its scratch from a fixed array in the library's own device
// memory instead, so it allocates nothing at call time.
//
// Costs and rules of that array:
//  - it is kFaNoallocScratchBytes (64 MiB) on every GPU that loads the
//    library, held until the process exits;
//  - problems whose scratch (fa_bwd_workspace_size) is larger are rejected
//    with FA_ERR_WORKSPACE before anything is enqueued;
//  - all calls share it and it keeps the last call's contents; the backward
//    preprocess rewrites D and zeroes the dQ accumulator at the start of
//    every call, so no stale value is read;
//  - calls whose work overlaps on the GPU (two streams, or two host threads)
//    race on it: the caller must order them;
//  - the first call on each device looks up the array's device address with
//    that device current (cudaGetSymbolAddress), so make that first call
//    before any stream capture.
#include <mutex>

#include "fa.h"

namespace {

constexpr size_t kFaNoallocScratchBytes = static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES);

// The scratch itself.  In host code this name is only a host-side stand-in
// for the device symbol: its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kFaNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64];   // device address of the array, per device

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int N, int d, int causal, float scale,
                              int dtype, fa_stream_t stream) {
  const size_t need = fa_bwd_workspace_size(B, H, Hkv, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kFaNoallocScratchBytes) return FA_ERR_WORKSPACE;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? FA_ERR_CUDA : FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess) return FA_ERR_CUDA;
      g_scratch_ptr[dev] = ptr;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, d, causal, scale, dtype,
                scratch, kFaNoallocScratchBytes, stream);
}
