// C-ABI layer of libfa_gb300.so: argument validation, variant dispatch,
// tensor-map encoding and error reporting.  See include/fa.h for the contract.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Device-side error word; kernels receive its address and set bit 0 when a
// bounded wait expired.
__device__ unsigned int g_device_error = 0;

namespace {

thread_local char g_cuda_msg[256] = "no CUDA error recorded";

int cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_cuda_msg, sizeof(g_cuda_msg), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return FA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

void load_encoder() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                  cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
    g_encode_err = cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Per-device answer to "is this an sm_103 device?", cached.
int g_dev_ok[64];   // 0 = unknown, 1 = yes, 2 = no
std::mutex g_dev_mu;

unsigned int* g_err_ptr[64];

// Checks that the current device is an sm_103 part and returns the device
// address of its error word in *err (both cached per device).
int check_device(unsigned int** err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major == 10 && minor == 3) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_device_error);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
      g_err_ptr[dev] = static_cast<unsigned int*>(ptr);
      g_dev_ok[dev] = 1;
    } else {
      g_dev_ok[dev] = 2;
    }
  }
  if (g_dev_ok[dev] != 1) return FA_ERR_UNSUPPORTED;
  *err = g_err_ptr[dev];
  return FA_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int validate(int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
             Problem* pr) {
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARG;
  if (B > 65535 || H > 65535) return FA_ERR_INVALID_ARG;   // grid y/z limits
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  // Every tensor-map dimension and every flat index must fit the kernels'
  // 32-bit coordinates.
  const long long rows_q = static_cast<long long>(B) * H * Nq;
  const long long rows_k = static_cast<long long>(B) * Hkv * Nk;
  if (static_cast<long long>(B) * H > INT32_MAX || rows_q > (1ll << 31) - 1 ||
      rows_k > (1ll << 31) - 1 || static_cast<long long>(Nq) * d > INT32_MAX ||
      static_cast<long long>(Nk) * d > INT32_MAX)
    return FA_ERR_INVALID_ARG;
  pr->B = B;
  pr->H = H;
  pr->Hkv = Hkv;
  pr->Nq = Nq;
  pr->Nk = Nk;
  pr->d = d;
  pr->causal = causal;
  pr->bf16 = dtype == FA_BF16 ? 1 : 0;
  pr->scale = scale;
  pr->err = nullptr;
  return FA_OK;
}

}  // namespace

namespace {
// Encoded tensor maps, kept per (base address, shape, strides, box): encoding
// is a driver call of about a microsecond, and a training loop passes the
// same buffers call after call.  A fixed number of entries, replaced round
// robin; the map itself holds only the address and the geometry, so an entry
// is valid on any device.
struct TmapKey {
  int kind;                      // 0: 16-bit 4-D view, 1: fp32 3-D array
  const void* base;
  long long dims[4], strides[3];
  int box[2];
  bool operator==(const TmapKey& o) const {
    return kind == o.kind && base == o.base && box[0] == o.box[0] && box[1] == o.box[1] &&
           std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
           std::memcmp(strides, o.strides, sizeof(strides)) == 0;
  }
};
constexpr int kTmapCacheSize = 128;
struct TmapCache {
  std::mutex mu;
  TmapKey key[kTmapCacheSize];
  CUtensorMap map[kTmapCacheSize];
  int used = 0, next = 0;
};
TmapCache g_tmaps;

bool tmap_lookup(const TmapKey& k, CUtensorMap* out) {
  std::lock_guard<std::mutex> lk(g_tmaps.mu);
  for (int i = 0; i < g_tmaps.used; ++i)
    if (g_tmaps.key[i] == k) {
      *out = g_tmaps.map[i];
      return true;
    }
  return false;
}

void tmap_store(const TmapKey& k, const CUtensorMap& m) {
  std::lock_guard<std::mutex> lk(g_tmaps.mu);
  const int slot = g_tmaps.next;
  g_tmaps.key[slot] = k;
  g_tmaps.map[slot] = m;
  g_tmaps.next = (slot + 1) % kTmapCacheSize;
  if (g_tmaps.used < kTmapCacheSize) ++g_tmaps.used;
}
}  // namespace

cudaError_t make_tmap_4d(CUtensorMap* map, const void* base, int cols, int rows, int heads,
                         int batch, const Strides& st, int box_cols, int box_rows) {
  TmapKey key{};
  key.kind = 0;
  key.base = base;
  key.dims[0] = cols;
  key.dims[1] = rows;
  key.dims[2] = heads;
  key.dims[3] = batch;
  key.strides[0] = st.n;
  key.strides[1] = st.h;
  key.strides[2] = st.b;
  key.box[0] = box_cols;
  key.box[1] = box_rows;
  if (tmap_lookup(key, map)) return cudaSuccess;
  std::call_once(g_encode_once, load_encoder);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  tmap_store(key, *map);
  return cudaSuccess;
}

cudaError_t make_tmap_f32_3d(CUtensorMap* map, const float* base, int cols, int rows, int planes,
                             int box_cols, int box_rows) {
  TmapKey key{};
  key.kind = 1;
  key.base = base;
  key.dims[0] = cols;
  key.dims[1] = rows;
  key.dims[2] = planes;
  key.box[0] = box_cols;
  key.box[1] = box_rows;
  if (tmap_lookup(key, map)) return cudaSuccess;
  std::call_once(g_encode_once, load_encoder);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4,
                           static_cast<cuuint64_t>(cols) * rows * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  tmap_store(key, *map);
  return cudaSuccess;
}

namespace {
struct TimingState {
  std::mutex mu;
  std::vector<cudaEvent_t> start, stop;
  std::vector<int> kind;     // kind of each used slot
  bool enabled = false;
};
TimingState g_timing;
}  // namespace

int timing_begin(int kind, cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  if (!g_timing.enabled || g_timing.kind.size() >= g_timing.start.size()) return -1;
  const int slot = static_cast<int>(g_timing.kind.size());
  g_timing.kind.push_back(kind);
  cudaEventRecord(g_timing.start[slot], stream);
  return slot;
}

void timing_end(int slot, cudaStream_t stream) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_timing.mu);
  if (slot < static_cast<int>(g_timing.stop.size())) cudaEventRecord(g_timing.stop[slot], stream);
}

// One thread waits, through the attention kernels' bounded wait, on a
// barrier that nothing completes; the expired wait is reported exactly as in
// those kernels (bit 0 of the error word).
__global__ void expired_wait_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t never_done;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never_done), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool completed = mbar_wait_limit(smem_u32(&never_done), 0, &abort_flag, limit_ns);
    if (!completed && abort_flag == 2) atomicOr(err, kErrTimeout);
  }
}

// Throughput of the exponential unit: every thread runs eight independent
// chains x <- 2^(-x) (values stay in [1/2, 1]) through ex2.approx, the
// instruction the softmax warps use; the chains' results are kept alive
// through a store that never happens for these inputs.
__global__ void __launch_bounds__(256) ex2_rate_kernel(float* sink, int iters) {
  float x[8];
  #pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = -1e-3f * static_cast<float>((threadIdx.x + i) & 63);
  for (int it = 0; it < iters; ++it) {
    #pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = ex2_approx(-x[i]);
  }
  float s = 0.f;
  #pragma unroll
  for (int i = 0; i < 8; ++i) s += x[i];
  if (s < 0.f) sink[blockIdx.x] = s;
}

// 16 KB fp32 tiles of shared memory (zeros) added into `dst` by 1-D bulk
// reduce-adds from one thread per CTA, two in flight: the outflow of
// reduction traffic an SM sustains, which bounds the atomic dQ strategy.
__global__ void __launch_bounds__(128) reduce_rate_kernel(float* dst, int tiles, int rounds) {
  extern __shared__ __align__(128) float zeros[];
  for (int i = threadIdx.x; i < 2 * 4096; i += 128) zeros[i] = 0.f;
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t base = smem_u32(zeros);
    for (int it = 0; it < rounds; ++it) {
      const int tile = static_cast<int>((static_cast<long long>(blockIdx.x) * 7 + it * 13ll) % tiles);
      asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 16384;"
                   ::"l"(dst + static_cast<size_t>(tile) * 4096), "r"(base + (it & 1) * 16384)
                   : "memory");
      bulk_commit_group();
      bulk_wait_read_one_left();
    }
    bulk_wait_all();
  }
}

size_t bwd_workspace_bytes(int B, int H, int N, int d, int deterministic) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t delta = (rows * sizeof(float) + 255) / 256 * 256;
  if (deterministic) return delta;   // dQ is written directly, no accumulator
  const size_t acc = (rows * d * sizeof(float) + 255) / 256 * 256;
  return delta + acc + kBwdSchedBytes;   // + the persistent kernel's work counter
}

}  // namespace fa

using fa::Problem;

namespace fa {
namespace {
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// Short queries of a GQA group share one query-row block (see FwdArgs::pack).
bool pack_groups(int H, int Hkv, int Nq) { return H > Hkv && Nq <= 64; }

// Split count for fa_fwd_splitkv: among the counts that keep at least four
// key tiles per split and give at least two waves of CTAs, the one whose
// last wave is fullest (fewest idle SMs); 1 when there are enough CTAs.
int auto_splits(int B, int H, int Hkv, int Nq, int Nk, int d) {
  const int rows = pack_groups(H, Hkv, Nq) ? (H / Hkv) * Nq : Nq;
  const long long ctas =
      static_cast<long long>((rows + 127) / 128) * (pack_groups(H, Hkv, Nq) ? Hkv : H) * B;
  const int n_kv = (Nk + fwd_key_tile(d) - 1) / fwd_key_tile(d);
  const long long sms = num_sms();
  if (ctas >= 2 * sms) return 1;
  const int max_sp = std::max(1, n_kv / 4);
  int best = 1;
  double best_eff = -1.0;
  for (int sp = 1; sp <= max_sp; ++sp) {
    const long long total = ctas * sp;
    if (total < 2 * sms && sp < max_sp) continue;
    const double waves = static_cast<double>(total) / sms;
    const double eff = waves / std::ceil(waves);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = sp;
    }
    if (total >= 8 * sms) break;
  }
  return best;
}

size_t splitkv_bytes(int B, int H, int Nq, int d, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  const size_t o = (static_cast<size_t>(splits) * rows * d * 4 + 255) / 256 * 256;
  const size_t l = (static_cast<size_t>(splits) * rows * 4 + 255) / 256 * 256;
  return o + l;
}

// Strides of a caller's view: each a positive multiple of 8 elements (16
// bytes, the tensor-map stride unit) below 2^39 elements.
bool valid_strides(const fa_strides* s, int n, Strides* out) {
  if (s == nullptr) return false;
  for (int i = 0; i < n; ++i) {
    const long long v[3] = {s[i].batch, s[i].head, s[i].row};
    for (long long x : v)
      if (x < 8 || x % 8 != 0 || x >= (1ll << 39)) return false;
    out[i] = {s[i].batch, s[i].head, s[i].row};
  }
  return true;
}

// st: element strides of q, k, v, o (nullptr: contiguous).
int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
               fa_stream_t stream, int splits = 1, void* workspace = nullptr,
               size_t workspace_bytes = 0, const BlockMask* mask = nullptr,
               const Strides* strd = nullptr) {
  Problem pr;
  int st = validate(B, H, Hkv, Nq, Nk, d, causal, scale, dtype, &pr);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  if (splits > 1) {
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < splitkv_bytes(B, H, Nq, d, splits))
      return FA_ERR_WORKSPACE;
  }
  if ((st = check_device(&pr.err)) != FA_OK) return st;
  FwdArgs a{q, k, v, o, lse};
  if (strd != nullptr) {
    a.qs = strd[0];
    a.ks = strd[1];
    a.vs = strd[2];
    a.os = strd[3];
  } else {
    a.qs = a.os = contiguous_strides(H, Nq, d);
    a.ks = a.vs = contiguous_strides(Hkv, Nk, d);
  }
  // packing needs the G * Nq rows of a group evenly spaced in q and o
  const bool even = Nq == 1 || (a.qs.h == Nq * a.qs.n && a.os.h == Nq * a.os.n);
  a.pack = pack_groups(H, Hkv, Nq) && mask == nullptr && even ? 1 : 0;
  if (mask != nullptr) a.mask = *mask;
  a.splits = splits;
  if (splits > 1) {
    const size_t rows = static_cast<size_t>(B) * H * Nq;
    a.o_part = static_cast<float*>(workspace);
    a.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          (static_cast<size_t>(splits) * rows * d * 4 + 255) /
                                              256 * 256);
  }
  cudaError_t e = launch_fwd(pr, a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_fwd launch");
  return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Hkv, int N, int d, int causal, float scale, int dtype,
                      fa_stream_t stream) {
  return fa::fwd_common(q, k, v, o, lse, B, H, Hkv, N, N, d, causal, scale, dtype, stream);
}

extern "C" int fa_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                         fa_stream_t stream) {
  return fa::fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, dtype, stream);
}

extern "C" size_t fa_fwd_splitkv_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d,
                                                int num_splits) {
  Problem pr;
  if (num_splits < 0 ||
      fa::validate(B, H, Hkv, Nq, Nk, d, 0, 1.0f, FA_BF16, &pr) != FA_OK)
    return 0;
  const int sp = num_splits == 0 ? fa::auto_splits(B, H, Hkv, Nq, Nk, d) : num_splits;
  return fa::splitkv_bytes(B, H, Nq, d, sp);
}

extern "C" int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                              float scale, int dtype, int num_splits, void* workspace,
                              size_t workspace_bytes, fa_stream_t stream) {
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  Problem pr;
  int st = fa::validate(B, H, Hkv, Nq, Nk, d, causal, scale, dtype, &pr);
  if (st != FA_OK) return st;
  const int sp = num_splits == 0 ? fa::auto_splits(B, H, Hkv, Nq, Nk, d) : num_splits;
  return fa::fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, dtype, stream, sp,
                        workspace, workspace_bytes);
}

namespace fa {
namespace {
// Checks a block mask's arguments and the step-list capacities for the
// shape (pr already validated); fills *m.
int mask_args(const Problem& pr, const unsigned char* block_mask, int mask_heads, BlockMask* m) {
  if (block_mask == nullptr) return FA_ERR_INVALID_ARG;
  if (mask_heads != 1 && mask_heads != pr.H) return FA_ERR_INVALID_ARG;
  m->ptr = block_mask;
  m->heads = mask_heads;
  m->nbr = (pr.Nq + kMaskBlock - 1) / kMaskBlock;
  m->nbc = (pr.Nk + kMaskBlock - 1) / kMaskBlock;
  return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int Hkv, int Nq, int Nk, int d,
                                  int causal, float scale, int dtype,
                                  const unsigned char* block_mask, int mask_heads,
                                  fa_stream_t stream) {
  Problem pr;
  int st = fa::validate(B, H, Hkv, Nq, Nk, d, causal, scale, dtype, &pr);
  if (st != FA_OK) return st;
  fa::BlockMask m;
  if ((st = fa::mask_args(pr, block_mask, mask_heads, &m)) != FA_OK) return st;
  if ((Nk + fa::fwd_key_tile(d) - 1) / fa::fwd_key_tile(d) > fa::kFwdListCap)
    return FA_ERR_INVALID_ARG;
  return fa::fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, dtype, stream, 1,
                        nullptr, 0, &m);
}

extern "C" int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                              float scale, int dtype, const fa_strides* strides,
                              fa_stream_t stream) {
  fa::Strides st[4];
  if (!fa::valid_strides(strides, 4, st)) return FA_ERR_INVALID_ARG;
  return fa::fwd_common(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, dtype, stream, 1,
                        nullptr, 0, nullptr, st);
}

extern "C" size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d) {
  Problem pr;
  if (fa::validate(B, H, Hkv, N, N, d, 0, 1.0f, FA_BF16, &pr) != FA_OK) return 0;
  return fa::bwd_workspace_bytes(B, H, N, d, 0);
}

extern "C" size_t fa_bwd_workspace_size_for(int B, int H, int Hkv, int Nq, int d,
                                            int deterministic) {
  Problem pr;
  if (deterministic != 0 && deterministic != 1) return 0;
  if (fa::validate(B, H, Hkv, Nq, Nq, d, 0, 1.0f, FA_BF16, &pr) != FA_OK) return 0;
  return fa::bwd_workspace_bytes(B, H, Nq, d, deterministic);
}

namespace fa {
namespace {
int bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
               int Nk, int d, int causal, float scale, int dtype, void* workspace,
               size_t workspace_bytes, fa_stream_t stream, int deterministic,
               const BlockMask* mask = nullptr, const Strides* strd = nullptr);
}  // namespace
}  // namespace fa

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int H, int Hkv, int N, int d, int causal, float scale, int dtype,
                      void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return fa::bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, N, d, causal, scale,
                        dtype, workspace, workspace_bytes, stream, 0);
}

extern "C" int fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, int B, int H, int Hkv, int N, int d, int causal,
                                    float scale, int dtype, void* workspace,
                                    size_t workspace_bytes, fa_stream_t stream) {
  return fa::bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, N, N, d, causal, scale,
                        dtype, workspace, workspace_bytes, stream, 1);
}

extern "C" int fa_bwd_qk(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                         int deterministic, void* workspace, size_t workspace_bytes,
                         fa_stream_t stream) {
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  return fa::bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale,
                        dtype, workspace, workspace_bytes, stream, deterministic);
}

extern "C" int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, void* dq, void* dk,
                                  void* dv, int B, int H, int Hkv, int Nq, int Nk, int d,
                                  int causal, float scale, int dtype,
                                  const unsigned char* block_mask, int mask_heads,
                                  int deterministic, void* workspace, size_t workspace_bytes,
                                  fa_stream_t stream) {
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  Problem pr;
  int st = fa::validate(B, H, Hkv, Nq, Nk, d, causal, scale, dtype, &pr);
  if (st != FA_OK) return st;
  fa::BlockMask m;
  if ((st = fa::mask_args(pr, block_mask, mask_heads, &m)) != FA_OK) return st;
  const int bq = fa::bwd_query_tile(d);
  if (static_cast<long long>(H / Hkv) * ((Nq + bq - 1) / bq) > fa::bwd_list_cap(d))
    return FA_ERR_INVALID_ARG;
  if (deterministic && (Nk + fa::kDqKeyTile - 1) / fa::kDqKeyTile > fa::kDqListCap)
    return FA_ERR_INVALID_ARG;
  return fa::bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale,
                        dtype, workspace, workspace_bytes, stream, deterministic, &m);
}

extern "C" int fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                              float scale, int dtype, const fa_strides* strides,
                              int deterministic, void* workspace, size_t workspace_bytes,
                              fa_stream_t stream) {
  if (deterministic != 0 && deterministic != 1) return FA_ERR_INVALID_ARG;
  fa::Strides st[8];
  if (!fa::valid_strides(strides, 8, st)) return FA_ERR_INVALID_ARG;
  return fa::bwd_common(q, k, v, o, lse, dout, dq, dk, dv, B, H, Hkv, Nq, Nk, d, causal, scale,
                        dtype, workspace, workspace_bytes, stream, deterministic, nullptr, st);
}

namespace fa {
namespace {
int bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Nq,
               int Nk, int d, int causal, float scale, int dtype, void* workspace,
               size_t workspace_bytes, fa_stream_t stream, int deterministic,
               const BlockMask* mask, const Strides* strd) {
  Problem pr;
  int st = fa::validate(B, H, Hkv, Nq, Nk, d, causal, scale, dtype, &pr);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!fa::aligned(q, 16) || !fa::aligned(k, 16) || !fa::aligned(v, 16) || !fa::aligned(o, 16) ||
      !fa::aligned(dout, 16) || !fa::aligned(dq, 16) || !fa::aligned(dk, 16) ||
      !fa::aligned(dv, 16) || !fa::aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  // scratch of the path that runs: D, and the fp32 dQ accumulator unless
  // dQ is formed by the query-outer kernel
  const size_t need = fa::bwd_workspace_bytes(B, H, Nq, d, deterministic);
  if (!workspace || workspace_bytes < need || !fa::aligned(workspace, 256))
    return FA_ERR_WORKSPACE;
  if ((st = fa::check_device(&pr.err)) != FA_OK) return st;
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  float* delta = static_cast<float*>(workspace);
  float* acc = deterministic ? nullptr
                            : reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                       (rows * sizeof(float) + 255) / 256 * 256);
  unsigned int* units =
      deterministic ? nullptr
                    : reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(acc) +
                                                      (rows * d * sizeof(float) + 255) / 256 * 256);
  // dQ strategy: atomic adds into the fp32 accumulator unless
  // reproducibility is asked for.
  fa::BwdArgs a{q, k, v, o, lse, dout, dq, dk, dv, delta, acc, deterministic};
  a.units = units;
  if (mask != nullptr) a.mask = *mask;
  if (strd != nullptr) {
    a.qs = strd[0];
    a.ks = strd[1];
    a.vs = strd[2];
    a.os = strd[3];
    a.dos = strd[4];
    a.dqs = strd[5];
    a.dks = strd[6];
    a.dvs = strd[7];
  } else {
    a.qs = a.os = a.dos = a.dqs = contiguous_strides(H, Nq, d);
    a.ks = a.vs = a.dks = a.dvs = contiguous_strides(Hkv, Nk, d);
  }
  cudaError_t e = fa::launch_bwd(pr, a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fa::cuda_fail(e, "fa_bwd launch");
  return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" int fa_get_device_status(fa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fa::cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, fa::g_device_error, sizeof(word));
  if (e != cudaSuccess) return fa::cuda_fail(e, "read device error word");
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(fa::g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return fa::cuda_fail(e, "clear device error word");
    if (word & fa::kErrTimeout) return FA_ERR_TIMEOUT;
    std::snprintf(fa::g_cuda_msg, sizeof(fa::g_cuda_msg),
                  "a kernel found its dynamic shared memory base misaligned (error word %#x)",
                  word);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

extern "C" const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "success";
    case FA_ERR_INVALID_ARG: return "invalid argument (pointer, alignment, size or scale)";
    case FA_ERR_UNSUPPORTED: return "unsupported head dim, dtype or device (needs sm_103)";
    case FA_ERR_CUDA: return fa::g_cuda_msg;
    case FA_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case FA_ERR_WORKSPACE: return "backward workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

extern "C" int fa_timing_enable(int capacity) {
  std::lock_guard<std::mutex> lk(fa::g_timing.mu);
  for (cudaEvent_t e : fa::g_timing.start) cudaEventDestroy(e);
  for (cudaEvent_t e : fa::g_timing.stop) cudaEventDestroy(e);
  fa::g_timing.start.clear();
  fa::g_timing.stop.clear();
  fa::g_timing.kind.clear();
  fa::g_timing.enabled = false;
  if (capacity < 0) return FA_ERR_INVALID_ARG;
  for (int i = 0; i < capacity; ++i) {
    cudaEvent_t a, b;
    cudaError_t e = cudaEventCreate(&a);
    if (e == cudaSuccess) {
      e = cudaEventCreate(&b);
      if (e != cudaSuccess) cudaEventDestroy(a);
    }
    if (e != cudaSuccess) return fa::cuda_fail(e, "cudaEventCreate");
    fa::g_timing.start.push_back(a);
    fa::g_timing.stop.push_back(b);
  }
  fa::g_timing.enabled = capacity > 0;
  return FA_OK;
}

extern "C" int fa_timing_read(double* ms, int* launches) {
  if (!ms || !launches) return FA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(fa::g_timing.mu);
  for (int i = 0; i < FA_NUM_KERNEL_KINDS; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  for (size_t i = 0; i < fa::g_timing.kind.size(); ++i) {
    cudaError_t e = cudaEventSynchronize(fa::g_timing.stop[i]);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, fa::g_timing.start[i], fa::g_timing.stop[i]);
    if (e != cudaSuccess) return fa::cuda_fail(e, "timing event");
    const int k = fa::g_timing.kind[i];
    if (k >= 0 && k < FA_NUM_KERNEL_KINDS) {
      ms[k] += t;
      launches[k] += 1;
    }
  }
  fa::g_timing.kind.clear();
  return FA_OK;
}

extern "C" int fa_selftest_expired_wait(int limit_us, fa_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return FA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int st = fa::check_device(&err);
  if (st != FA_OK) return st;
  fa::expired_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      err, static_cast<uint64_t>(limit_us) * 1000ull);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : fa::cuda_fail(e, "selftest launch");
}

extern "C" int fa_measure_reduce_rate(void* scratch, size_t scratch_bytes, double* bytes_per_s,
                                      fa_stream_t stream) {
  if (!bytes_per_s || !scratch || scratch_bytes < (1u << 20) || !fa::aligned(scratch, 256))
    return FA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int st = fa::check_device(&err);
  if (st != FA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long tiles_ll = static_cast<long long>(scratch_bytes / 16384);
  const int tiles = static_cast<int>(std::min<long long>(tiles_ll, 1 << 30));
  const int blocks = fa::num_sms(), rounds = 400;
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return fa::cuda_fail(e, "cudaEventCreate");
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
    cudaEventDestroy(e0);
    return fa::cuda_fail(e, "cudaEventCreate");
  }
  double best = 0.0;
  for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {
    cudaEventRecord(e0, s);
    fa::reduce_rate_kernel<<<blocks, 128, 2 * 16384, s>>>(static_cast<float*>(scratch), tiles, rounds);
    cudaEventRecord(e1, s);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && rep > 0 && ms > 0.f)   // the first run is a warm-up
      best = std::max(best, 16384.0 * blocks * rounds / (ms * 1e-3));
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return fa::cuda_fail(e, "reduce rate kernel");
  *bytes_per_s = best;
  return FA_OK;
}

extern "C" int fa_measure_ex2_rate(double* exps_per_s, fa_stream_t stream) {
  if (!exps_per_s) return FA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int st = fa::check_device(&err);
  if (st != FA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int blocks = 8 * fa::num_sms(), threads = 256, iters = 4096;
  cudaEvent_t e0, e1;
  cudaError_t e = cudaEventCreate(&e0);
  if (e != cudaSuccess) return fa::cuda_fail(e, "cudaEventCreate");
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
    cudaEventDestroy(e0);
    return fa::cuda_fail(e, "cudaEventCreate");
  }
  double best = 0.0;
  for (int rep = 0; rep < 4 && e == cudaSuccess; ++rep) {
    cudaEventRecord(e0, s);
    fa::ex2_rate_kernel<<<blocks, threads, 0, s>>>(nullptr, iters);
    cudaEventRecord(e1, s);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && rep > 0 && ms > 0.f)   // the first run is a warm-up
      best = std::max(best, 8.0 * blocks * threads * static_cast<double>(iters) / (ms * 1e-3));
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return fa::cuda_fail(e, "ex2 rate kernel");
  *exps_per_s = best;
  return FA_OK;
}
