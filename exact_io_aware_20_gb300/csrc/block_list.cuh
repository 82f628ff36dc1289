// Block-sparse attention: the work list one CTA keeps under a block mask.
//
// Block-sparse FlashAttention ("FlashAttention: Fast and Memory-Efficient
// Exact Attention with IO-Awareness", abstract and "Key contributions") is
// exact attention restricted to the kept blocks of a given pattern: a tile
// pair whose mask block is zero is skipped outright, so the work, and the
// HBM traffic, fall with the fraction of kept blocks.
//
// Each CTA walks a sequence of steps (key tiles for a query tile, or query
// tiles for a key tile).  Before the warps split up, one warp reads the
// CTA's row or column of the mask and writes the kept steps, in order, to a
// shared-memory list; every role then walks that list instead of the dense
// range.  Mask blocks are 128 x 128; a kernel tile smaller than 128 (64
// keys, or 64 query rows) is a sub-step of its block.
#pragma once

#include <cstdint>

namespace fa {

// One warp (all 32 lanes) compacts the n candidate blocks into `list`:
// candidate e, when kept(e), contributes the codes code(e, s) >= 0 of its SUB
// sub-steps (a negative code is a sub-step outside the CTA's range, such as a
// key tile past the causal limit).  Codes come out in order of e, then s.
// Returns the number of codes (in every lane); codes past `cap` are not
// stored, and the host keeps the count within cap.
template <int SUB, class Kept, class Code>
__device__ __forceinline__ int compact_steps(int n, Kept kept, Code code, uint16_t* list, int cap) {
  const int lane = threadIdx.x & 31;
  int count = 0;
  for (int base = 0; base < n; base += 32) {
    const int e = base + lane;
    const bool keep = e < n && kept(e);
    int mine[SUB];
    int c = 0;
    #pragma unroll
    for (int s = 0; s < SUB; ++s) {
      mine[s] = keep ? code(e, s) : -1;
      c += mine[s] >= 0 ? 1 : 0;
    }
    // inclusive prefix sum of the per-lane counts
    int incl = c;
    #pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int at = count + incl - c;
    #pragma unroll
    for (int s = 0; s < SUB; ++s) {
      if (mine[s] >= 0) {
        if (at < cap) list[at] = static_cast<uint16_t>(mine[s]);
        ++at;
      }
    }
    count += __shfl_sync(0xffffffffu, incl, 31);
  }
  return count;
}

}  // namespace fa
