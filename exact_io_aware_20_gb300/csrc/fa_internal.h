// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Shapes and pointers of one call, after validation.
struct Problem {
  int B, H, Hkv;
  int Nq, Nk;     // query and key lengths (the causal mask is anchored bottom-right)
  int d;
  int causal;
  int bf16;       // 1 = bf16, 0 = f16
  float scale;
  unsigned int* err;   // device error word (bit 0: a bounded wait expired)
};

// Element strides of a 16-bit [batch][heads][rows][d] view whose d elements
// are contiguous (the layout of every q, k, v, o and gradient tensor; the
// contiguous case is {heads * rows * d, rows * d, d}).
struct Strides {
  long long b = 0, h = 0, n = 0;
};
inline Strides contiguous_strides(int heads, int rows, int d) {
  return {static_cast<long long>(heads) * rows * d, static_cast<long long>(rows) * d, d};
}

// Block mask of block-sparse attention: bytes [heads][nbr][nbc], block
// (i, j) covering query rows [128 i, 128 i + 128) and keys [128 j, 128 j +
// 128); nonzero = the block is computed.  heads is 1 (one mask for every
// query head) or H.  ptr == nullptr: dense attention.
constexpr int kMaskBlock = 128;
struct BlockMask {
  const unsigned char* ptr = nullptr;
  int heads = 1;
  int nbr = 0, nbc = 0;   // ceil(Nq / 128), ceil(Nk / 128)
};

// Capacity of the per-CTA step lists (entries) under a block mask: key tiles
// of the forward and of the deterministic dQ kernel, (head, query tile)
// steps of the backward main kernel.  The C-ABI layer rejects shapes whose
// lists could exceed them.
constexpr int kFwdListCap = 8192;
constexpr int kDqListCap = 8192;
constexpr int kDqKeyTile = 64;   // keys per tile of the deterministic dQ kernel
int bwd_list_cap(int d);
int bwd_query_tile(int d);

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int pack = 0;              // 1: the G query heads of a KV group form one row block
  int splits = 1;            // > 1: split the key range, partials in o_part / lse_part
  float* o_part = nullptr;   // [splits][B*H*Nq][d] fp32
  float* lse_part = nullptr; // [splits][B*H*Nq] fp32
  BlockMask mask;            // block-sparse (needs pack == 0, splits == 1)
  Strides qs, ks, vs, os;    // element strides of q, k, v, o (set by the caller)
};

// Key tiles of the forward kernel (for choosing a split count).
int fwd_key_tile(int d);

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  float* delta;    // [B, H, Nq] fp32 scratch
  float* dq_acc;   // [B, H, Nq, d] fp32 scratch (unused when deterministic)
  int deterministic;   // dQ from the query-outer kernel, without atomics
  BlockMask mask = {};  // block-sparse
  unsigned int* units = nullptr;   // work counter of the persistent d = 128 kernel (scratch)
  // element strides of q, k, v, o, dout, dq, dk, dv (set by the caller); the
  // scratch (delta, dq_acc) and lse are always contiguous
  Strides qs = {}, ks = {}, vs = {}, os = {}, dos = {}, dqs = {}, dks = {}, dvs = {};
};

// Encode a 4-D tiled tensor map over a 16-bit [batch][heads][rows][cols]
// view (cols contiguous, element strides st) with a box of box_cols x
// box_rows of one (head, batch) and 128-byte swizzle; TMA coordinates are
// (col, row, head, batch).
cudaError_t make_tmap_4d(CUtensorMap* map, const void* base, int cols, int rows, int heads,
                         int batch, const Strides& st, int box_cols, int box_rows);

// Encode a 3-D tiled tensor map over a contiguous fp32 [planes][rows][cols]
// array with a box of box_cols x box_rows of one plane and no swizzle;
// coordinates (col, row, plane).
cudaError_t make_tmap_f32_3d(CUtensorMap* map, const float* base, int cols, int rows, int planes,
                             int box_cols, int box_rows);

// Diagnostics timing (see fa_timing_enable in fa.h): returns a slot to pass
// to timing_end, or -1 when timing is off or out of event pairs.
int timing_begin(int kind, cudaStream_t stream);
void timing_end(int slot, cudaStream_t stream);

cudaError_t launch_fwd(const Problem& p, const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_blocksparse(const Problem& p, const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd(const Problem& p, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_blocksparse(const Problem& p, const BwdArgs& a, cudaStream_t stream);
// d = 128, dense, dQ by atomic adds: the fused five-product kernel.
cudaError_t launch_bwd_fused(const Problem& p, const BwdArgs& a, cudaStream_t stream);
// d = 256, dense: dK and dV from the cluster-pair kernel, dQ from the
// query-outer kernel (no atomics; needs only D in the scratch).
cudaError_t launch_bwd_pair(const Problem& p, const BwdArgs& a, cudaStream_t stream);
// Deterministic dQ (query-outer, no atomics); needs D in a.delta.
cudaError_t launch_bwd_dq(const Problem& p, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq_blocksparse(const Problem& p, const BwdArgs& a, cudaStream_t stream);

// Bytes of backward scratch for a problem: delta, and unless deterministic
// the fp32 dq accumulator (each rounded up to 256 bytes) and kBwdSchedBytes
// for the work counter of the persistent d = 128 kernel.
constexpr size_t kBwdSchedBytes = 256;
size_t bwd_workspace_bytes(int B, int H, int N, int d, int deterministic);

}  // namespace fa
