// Forward kernel of exact attention on sm_103a: O = softmax(scale * Q K^T) V
// and the row logsumexp L, computed tile by tile without writing the score
// matrix to memory.  Instantiated dense in fa_fwd.cu and block-sparse in
// fa_fwd_blocksparse.cu.
//
// Method ("FlashAttention-2: Faster Attention with Better Parallelism and
// Work Partitioning", paper digest):
//  - section 2 Q2, improvement 2: the outer loop runs over query tiles, which
//    are independent, so work units are (batch, head, query tile);
//  - section 2 Q2, tweak 1: the output is kept unnormalised,
//    O~(j) = diag(exp(m(j-1) - m(j))) O~(j-1) + exp(S(j) - m(j)) V(j), and is
//    divided by the row sum l once at the end;
//  - section 2 Q2, tweak 2: only L = m + log(l) is written for the backward;
//  - section 2 Q2, causal masking: key tiles entirely above the diagonal are
//    skipped and the mask is applied only on tiles that cross it;
//  - section 4 "six checks", GQA/MQA: query head h reads key/value head
//    h / (H / Hkv) by index, with no copy.
// Under a block mask (block-sparse attention, "FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", abstract) a unit walks
// only the key tiles of its kept mask blocks: the Q / K producer reads the
// unit's mask row and publishes the kept tiles as a bit set in a unit record
// that the other warps read.
//
// GB300 design (not the pages' A100 design): a work unit is one 128-row
// query tile (of one split of the keys, head, batch); a persistent grid of one
// CTA per SM walks the units (with or without a block mask), TMEM, the
// barriers and the K / V rings living across units; warp-specialised:
//   warp 0      TMA producer: each unit's Q, then K_j through a smem ring;
//   warp 6      TMA producer: V_j through a second ring;
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM score buffers,
//               O += P_j V_j with P_j read from TMEM (tcgen05 "TS" form);
//   warps 2..5  softmax: one query row per thread, read S_j from TMEM, mask,
//               running max / sum, write P_j back into the score buffer as
//               16-bit, rescale O in TMEM when the max moved, epilogue.
// The O rescale is skipped while the running max has grown by at most 2^8
// (log2 units); the final division and L use the same stale maximum, so the
// result is unchanged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#pragma once

#include "block_list.cuh"
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int kBR = 128;             // query rows per tile (= MMA M)
constexpr int kThreads = 224;        // 7 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int BC, int KST, int VST>
struct FwdLayout {
  static constexpr int kNch = D / 64;                 // 64-column (128-byte) chunks
  static constexpr int kQBytes = kBR * D * 2;
  static constexpr int kKVBytes = BC * D * 2;
  // For d <= 128 each V stage is followed by a 64-column chunk of ones, so
  // the P V product, widened to N = d + 16, also sums the rounded weights of
  // every row into 16 extra TMEM columns (the row sum l_r without ALU work).
  static constexpr bool kOnes = D <= 128;
  static constexpr int kOnesCols = kOnes ? 16 : 0;
  // d = 256: a whole 128-key K or V tile is 64 KB, so the rings hold smaller
  // pieces, each with its own barriers: K in 64-column chunks (the pieces
  // S = Q K^T consumes one after another along d) and V in halves of BC / 2
  // keys (the pieces P V consumes along the keys).  KST and VST then count
  // pieces, and a slot is freed as soon as the products reading it are done.
  static constexpr bool kChunked = D > 128 && BC == 128;
  static constexpr int kKSlot = kChunked ? BC * 128 : kKVBytes;
  static constexpr int kVHalf = (BC / 2) * D * 2;
  static constexpr int kVStage = kChunked ? kVHalf : kKVBytes + (kOnes ? BC * 128 : 0);
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + KST * kKSlot;
  static constexpr int kBarOff = kVOff + VST * kVStage;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 1;
  static constexpr int kKFull = 2;
  static constexpr int kKEmpty = kKFull + KST;
  static constexpr int kVFull = kKEmpty + KST;
  static constexpr int kVEmpty = kVFull + VST;
  static constexpr int kSFull = kVEmpty + VST;   // 2
  static constexpr int kPFull = kSFull + 2;      // 2
  static constexpr int kODone = kPFull + 2;
  static constexpr int kDrain = kODone + 1;
  static constexpr int kUnitFull = kDrain + 1;     // 2: unit records (block mask)
  static constexpr int kUnitEmpty = kUnitFull + 2; // 2
  static constexpr int kNumBars = kUnitEmpty + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // Under a block mask: two unit records {kept tiles, bit set of the kept
  // key tiles (one bit per 128-key tile, up to kFwdListCap tiles)}
  static constexpr int kRecOff = kMiscOff + 16;
  static constexpr int kRecBytes = 16 + kFwdListCap / 8;
  static constexpr int kAlloc = kRecOff + 2 * kRecBytes + 1024;   // slack to align the base
  static constexpr int kAllocDense = kRecOff + 1024;              // without the records
  // TMEM columns
  static constexpr uint32_t kS0 = 0, kS1 = BC, kO = 2 * BC;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kO + D + kOnesCols <= kTmemCols, "TMEM budget");
  static_assert(kAllocDense <= 227 * 1024, "shared memory budget");
  static_assert(kRecBytes % 16 == 0, "unit records are 16-byte aligned");
};

struct FwdParams {
  void* o;
  float* lse;
  int H, Hkv, G;
  int B_;             // batch (the persistent kernel derives its units from it)
  int sec_heads;      // persistent causal order: (batch, head) pairs per section
  int Nq, Nk;         // query rows per head (packed rows, see mask_rows) / key length
  int off;            // under the mask query i sees keys k <= i + off
  int mask_rows;      // query index of a row for the mask: row % mask_rows (== Nq unless
                      // the query heads of a KV group are packed into one row block)
  int num_q_tiles;
  int splits;         // > 1: each CTA covers tiles_per_split key tiles and writes a
  int tiles_per_split;  // normalised partial O (fp32) and its L to o_part / lse_part
  float* o_part;
  float* lse_part;
  float scale_log2;   // scale * log2(e)
  BlockMask mask;     // block-sparse: only kept blocks' key tiles (splits == 1, no packing)
  long long o_sb, o_sh, o_sn;   // element strides of o over (batch, head, row) in this
                                // kernel's view (packed rows: row stride and group stride)
  unsigned int* err;
};

template <int D, int BC, bool CAUSAL, bool BF16, int KST, int VST, bool SPARSE>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D, BC, KST, VST>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool packed = p.mask_rows != p.Nq;
  // Work units (split, query tile, head, batch), numbered with the split
  // fastest, then query tiles (under the mask the longest first), heads,
  // batches.  The grid is persistent: CTA c takes unit k * G + c in even
  // rounds k and k * G + G - 1 - c in odd ones (G = grid size), so that over
  // two rounds of longest-first units every CTA gets about the same work.
  const int ux = p.num_q_tiles * p.splits;
  const long long n_units = static_cast<long long>(ux) * p.H * p.B_;
  auto unit_of = [&](int k) -> long long {
    const long long G = gridDim.x;
    const long long u = k * G + ((k & 1) ? G - 1 - blockIdx.x : blockIdx.x);
    return u < n_units ? u : -1;
  };
  // n_kv: key tiles of the unit; lim: the tiles its rows may see (the
  // causal / length limit), of which a block mask keeps n_kv
  struct Unit {
    int split, qt, h, b, n_kv, j_base, lim;
  };
  auto decode = [&](long long u) {
    Unit w;
    const int bx = static_cast<int>(u % ux);
    const long long hb = u / ux;
    w.h = static_cast<int>(hb % p.H);
    w.b = static_cast<int>(hb / p.H);
    w.split = p.splits > 1 ? bx % p.splits : 0;
    const int xt = p.splits > 1 ? bx / p.splits : bx;
    w.qt = CAUSAL ? (p.num_q_tiles - 1 - xt) : xt;
    int n = (p.Nk + BC - 1) / BC;
    if (CAUSAL) {
      // last key any row of this tile may see (bottom-right aligned mask);
      // negative when every row of the tile sees none (only if Nq > Nk)
      const int max_i = packed ? p.mask_rows - 1 : min((w.qt + 1) * kBR, p.Nq) - 1;
      const int last_key = max_i + p.off;
      n = last_key < 0 ? 0 : min(n, last_key / BC + 1);
    }
    // key tiles [j_base, j_base + n) of this split
    w.j_base = w.split * p.tiles_per_split;
    if (p.splits > 1) n = max(0, min(n, w.j_base + p.tiles_per_split) - w.j_base);
    w.n_kv = n;
    w.lim = n;
    return w;
  };
  constexpr bool sparse = SPARSE;
  static_assert(!SPARSE || BC == kMaskBlock, "a key tile is a mask block");
  // Under a block mask a unit walks the kept blocks of its query tile's mask
  // row.  The Q / K producer reads the row and publishes each unit's record
  // (the kept count and a bit set of the kept key tiles) in one of two slots;
  // the other warps take the unit's tiles from the record and release the
  // slot when they are done with it.
  auto mask_row = [&](const Unit& w) -> const unsigned char* {
    const int mh = p.mask.heads == 1 ? 0 : w.h;
    return p.mask.ptr + (static_cast<size_t>(mh) * p.mask.nbr + w.qt) * p.mask.nbc;
  };
  auto rec_n = [&](int k) -> volatile int* {
    return reinterpret_cast<volatile int*>(smem + L::kRecOff + (k & 1) * L::kRecBytes);
  };
  auto rec_bits = [&](int k) -> const volatile uint32_t* {
    return reinterpret_cast<const volatile uint32_t*>(smem + L::kRecOff + (k & 1) * L::kRecBytes + 16);
  };
  // the key tiles of unit w in order: next() once per step j (a whole warp)
  struct TileWalk {
    const volatile uint32_t* bits;
    int base, word;
    uint32_t cur;
    __device__ __forceinline__ int next(int j) {
      if constexpr (!SPARSE) {
        return base + j;
      } else {
        while (cur == 0) cur = bits[++word];
        const int i = __ffs(cur) - 1;
        cur &= cur - 1;
        return word * 32 + i;
      }
    }
  };
  auto walk_of = [&](const Unit& w, int k) {
    TileWalk t;
    t.base = w.j_base;
    t.word = 0;
    t.bits = sparse ? rec_bits(k) : nullptr;
    t.cur = sparse ? t.bits[0] : 0u;
    return t;
  };
  // the merge of split partials (launched as this grid's dependent) may start
  // its launch now; it waits for this grid's completion before reading
  if (p.splits > 1) grid_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 128);
    }
    mbar_init(bar(L::kODone), 1);
    mbar_init(bar(L::kDrain), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kUnitFull + s), 1);
      mbar_init(bar(L::kUnitEmpty + s), 6);   // V producer, MMA, four softmax warps
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  if constexpr (L::kOnes) {
    if (warp >= 2 && warp < 6) {
      // the ones chunks (any layout of all-ones is all-ones), written once
      const uint32_t one2 = BF16 ? 0x3F803F80u : 0x3C003C00u;
      for (int sv = 0; sv < VST; ++sv) {
        uint4* dst = reinterpret_cast<uint4*>(smem + L::kVOff + sv * L::kVStage + L::kKVBytes);
        for (int i = threadIdx.x - 64; i < BC * 128 / 16; i += 128)
          dst[i] = make_uint4(one2, one2, one2, one2);
      }
      fence_proxy_async_smem();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Unit k of this CTA; under a block mask the kept tiles come from its
  // record (a whole warp waits for it; false also when the wait gave up).
  // The Q / K producer makes the records (publish_unit) and does not call this.
  auto unit_at = [&](int k, Unit& w) -> bool {
    const long long u = unit_of(k);
    if (u < 0) return false;
    w = decode(u);
    if (sparse) {
      if (!wait_uniform(bar(L::kUnitFull + (k & 1)), (k >> 1) & 1, abort)) return false;
      w.n_kv = *rec_n(k);
    }
    return true;
  };
  auto release_unit = [&](int k) {
    if (sparse) mbar_arrive_warp(bar(L::kUnitEmpty + (k & 1)));
  };
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS0 = tmem + L::kS0, tS1 = tmem + L::kS1, tO = tmem + L::kO;

  if (warp == 0) {
    // ------------------------------------------------------------ producer: Q, K
    // Each unit's Q tile (once the previous unit's last S product has
    // completed), then its K tiles through the K ring; the V ring has a warp
    // of its own (warp 6), so that neither stream's waits hold up the
    // other's loads (in one thread, in order, a V slot waiting for P V(j)
    // would hold back K(j + 2), which S(j + 2) needs before the MMA warp
    // issues P V(j + 1)).  The whole warp runs the loop, one elected lane
    // issues the copies.
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    __syncwarp();
    int issued = 0, q_issued = 0;   // K pieces, Q tiles
    bool ok = true;
    Unit w;
    for (int k = 0; ok; ++k) {
      const long long u = unit_of(k);
      if (u < 0) break;
      w = decode(u);
      if (sparse) {
        // the unit's record, once the six readers are done with unit k - 2's:
        // the kept tiles of the query tile's mask row within its limit, read
        // eight 32-block chunks at a time (their loads in flight together)
        if (k >= 2 && !wait_uniform(bar(L::kUnitEmpty + (k & 1)), ((k >> 1) - 1) & 1, abort)) break;
        const unsigned char* row = mask_row(w);
        volatile uint32_t* bits =
            reinterpret_cast<volatile uint32_t*>(smem + L::kRecOff + (k & 1) * L::kRecBytes + 16);
        int n = 0;
        for (int base = 0; base < w.lim; base += 256) {
          unsigned char v[8];
          #pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int e = base + 32 * c + lane;
            v[c] = e < w.lim ? row[e] : 0;
          }
          #pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t m = __ballot_sync(0xffffffffu, v[c] != 0);
            if (base + 32 * c < w.lim) {
              if (lane == 0) bits[(base >> 5) + c] = m;
              n += __popc(m);
            }
          }
        }
        if (lane == 0) {
          *rec_n(k) = n;
          mbar_arrive(bar(L::kUnitFull + (k & 1)));   // (releases lane 0's writes)
        }
        __syncwarp();
        w.n_kv = n;
      }
      if (k >= 1 && !wait_uniform(bar(L::kQEmpty), (k - 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kQFull), L::kQBytes);
        #pragma unroll
        for (int c = 0; c < L::kNch; ++c)
          tma_load_4d(sbase + L::kQOff + c * (kBR * 128), &tm_q, bar(L::kQFull), c * 64, w.qt * kBR,
                      w.h, w.b);
      }
      __syncwarp();
      ++q_issued;
      const int kh = w.h / p.G;
      TileWalk tw = walk_of(w, k);
      for (int j = 0; ok && j < w.n_kv; ++j) {
        const int jt = tw.next(j);
        #pragma unroll 1
        for (int c = 0; c < (L::kChunked ? L::kNch : 1); ++c) {
          const int s = issued % KST;
          if (issued >= KST && !wait_uniform(bar(L::kKEmpty + s), ((issued / KST) + 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(L::kKFull + s), L::kKSlot);
            if constexpr (L::kChunked) {
              tma_load_4d(sbase + L::kKOff + s * L::kKSlot, &tm_k, bar(L::kKFull + s), c * 64,
                          jt * BC, kh, w.b);
            } else {
              #pragma unroll
              for (int cc = 0; cc < L::kNch; ++cc)
                tma_load_4d(sbase + L::kKOff + s * L::kKSlot + cc * (BC * 128), &tm_k,
                            bar(L::kKFull + s), cc * 64, jt * BC, kh, w.b);
            }
          }
          __syncwarp();
          ++issued;
        }
      }
    }
    // Never leave the CTA with copies in flight: wait for every load issued
    // (they have completed already on the normal path).
    if (q_issued > 0) drain_wait(bar(L::kQFull), (q_issued - 1) & 1);
    for (int i = max(0, issued - KST); i < issued; ++i)
      drain_wait(bar(L::kKFull + i % KST), (i / KST) & 1);
  } else if (warp == 6) {
    // ------------------------------------------------------------ producer: V
    int issued = 0;
    bool ok = true;
    Unit w;
    for (int k = 0; ok && unit_at(k, w); ++k) {
      const int kh = w.h / p.G;
      TileWalk tw = walk_of(w, k);
      for (int j = 0; ok && j < w.n_kv; ++j) {
        const int jt = tw.next(j);
        #pragma unroll 1
        for (int hv = 0; hv < (L::kChunked ? 2 : 1); ++hv) {
          const int sv = issued % VST;
          if (issued >= VST && !wait_uniform(bar(L::kVEmpty + sv), ((issued / VST) + 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            if constexpr (L::kChunked) {
              mbar_arrive_expect_tx(bar(L::kVFull + sv), L::kVHalf);
              #pragma unroll
              for (int c = 0; c < L::kNch; ++c)
                tma_load_4d(sbase + L::kVOff + sv * L::kVStage + c * ((BC / 2) * 128), &tm_v,
                            bar(L::kVFull + sv), c * 64, jt * BC + hv * (BC / 2), kh, w.b);
            } else {
              mbar_arrive_expect_tx(bar(L::kVFull + sv), L::kKVBytes);
              #pragma unroll
              for (int c = 0; c < L::kNch; ++c)
                tma_load_4d(sbase + L::kVOff + sv * L::kVStage + c * (BC * 128), &tm_v,
                            bar(L::kVFull + sv), c * 64, jt * BC, kh, w.b);
            }
          }
          __syncwarp();
          ++issued;
        }
      }
      if (ok) release_unit(k);
    }
    for (int i = max(0, issued - VST); i < issued; ++i)
      drain_wait(bar(L::kVFull + i % VST), (i / VST) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Warp-wide; each tcgen05 instruction is issued by one elected lane.
    // Descriptors are built once and advanced by constant offsets.  Global
    // step g counts the CTA's key tiles over all its units: it indexes the
    // score buffers and the K / V rings, and the parities of S_FULL, P_FULL
    // and O_DONE.
    constexpr uint32_t kIdS = idesc_f16(kBR, BC, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t kIdO = idesc_f16(kBR, D + L::kOnesCols, BF16 ? 1 : 0, 0, 1);
    const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sbase + L::kVOff, BC * 128, 1024);
    // a V half: 64-column chunks of BC / 2 keys each
    const uint64_t v_desc_half = smem_desc_sw128(sbase + L::kVOff, (BC / 2) * 128, 1024);
    auto issue_s = [&](int g) -> bool {
      const uint32_t d_tmem = (g & 1) ? tS1 : tS0;
      if constexpr (L::kChunked) {
        // one chunk of K (64 columns of d) at a time, each slot freed as soon
        // as its four products are done
        #pragma unroll 1
        for (int c = 0; c < L::kNch; ++c) {
          const int ck = g * L::kNch + c, s = ck % KST;
          if (!wait_uniform(bar(L::kKFull + s), (ck / KST) & 1, abort)) return false;
          tc_fence_after();
          const uint64_t ks = desc_add(k_desc, s * L::kKSlot);
          #pragma unroll
          for (int w = 0; w < 4; ++w)
            mma_ss(d_tmem, desc_add(q_desc, c * (kBR * 128) + w * 32), desc_add(ks, w * 32), kIdS,
                   (c > 0 || w > 0) ? 1u : 0u);
          mma_commit(bar(L::kKEmpty + s));
        }
        mma_commit(bar(L::kSFull + (g & 1)));
        return true;
      }
      const int s = g % KST;
      if (!wait_uniform(bar(L::kKFull + s), (g / KST) & 1, abort)) return false;
      tc_fence_after();
      const uint64_t ks = desc_add(k_desc, s * L::kKSlot);
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(d_tmem, desc_add(q_desc, c * (kBR * 128) + w * 32),
               desc_add(ks, c * (BC * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull + (g & 1)));
      mma_commit(bar(L::kKEmpty + s));
      return true;
    };
    bool ok = true;
    int g = 0;                 // key tiles so far
    Unit w;
    for (int k = 0; ok && unit_at(k, w); ++k) {
      // The tile count and the step index that selects ring slots and score
      // buffers (and so the MMA descriptors) are read from lane 0: the
      // compiler then knows they are the same in every lane and keeps the
      // loop and the descriptor arithmetic on the uniform datapath.  Taken
      // from the unit record as they are, each key tile's products took
      // 5-10% longer to issue (head256 forward 352 -> 376 us).
      const int n = __shfl_sync(0xffffffffu, w.n_kv, 0);
      release_unit(k);   // (only the count is needed here)
      ok = wait_uniform(bar(L::kQFull), k & 1, abort);
      if (ok && n > 0) ok = issue_s(g);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          if (!issue_s(__shfl_sync(0xffffffffu, g + j + 1, 0))) { ok = false; break; }
        } else {
          mma_commit(bar(L::kQEmpty));     // the unit's last S has been issued
        }
        if (!wait_uniform(bar(L::kPFull + ((g + j) & 1)), ((g + j) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        // O += P V (the first of a unit overwrites O: every softmax thread
        // reads the previous unit's O out, and waits for the loads, before
        // it turns to this unit's scores, so P_FULL of this tile implies O
        // is free).  Inline here: as a separate function the issue sequence
        // ran ~10% slower (head256 forward 354 -> 393 us).
        const int gj = __shfl_sync(0xffffffffu, g + j, 0);
        const uint32_t a_tmem = (gj & 1) ? tS1 : tS0;
        if constexpr (L::kChunked) {
          // one half of the keys at a time
          #pragma unroll 1
          for (int hv = 0; hv < 2; ++hv) {
            const int vh = 2 * gj + hv, sv = vh % VST;
            if (!wait_uniform(bar(L::kVFull + sv), (vh / VST) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vs = desc_add(v_desc_half, sv * L::kVStage);
            #pragma unroll
            for (int w2 = 0; w2 < BC / 32; ++w2)
              mma_ts(tO, a_tmem + (hv * (BC / 32) + w2) * 8, desc_add(vs, w2 * 2048), kIdO,
                     (j > 0 || hv > 0 || w2 > 0) ? 1u : 0u);
            mma_commit(bar(L::kVEmpty + sv));
          }
          if (!ok) break;
          mma_commit(bar(L::kODone));
        } else {
          const int sv = gj % VST;
          if (!wait_uniform(bar(L::kVFull + sv), (gj / VST) & 1, abort)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vs = desc_add(v_desc, sv * L::kVStage);
          #pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_ts(tO, a_tmem + kk * 8, desc_add(vs, kk * 2048), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kODone));
          mma_commit(bar(L::kVEmpty + sv));
        }
      }
      if (!ok) break;
      if (n == 0) mma_commit(bar(L::kQEmpty));
      g += n;
    }
    // Every MMA issued above completes before TMEM is released.
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ softmax (warps 2..5)
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int r_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int g = 0;
    Unit w;
    for (int k = 0; ok && unit_at(k, w); ++k) {
      const int n_kv = w.n_kv, qt = w.qt, h = w.h, b = w.b, split = w.split;
      const int row = qt * kBR + r_tile;
      const int qi = row % p.mask_rows;             // query index of this row for the mask
      float m_ref = -INFINITY, l = 0.f, l_r = 0.f;
      // A warp whose 32 rows all lie past the last query row (short or packed
      // queries) only keeps the barrier protocol: its Q rows are zero-filled,
      // so its scores are 0 and the P it leaves in TMEM is 0, and its rows are
      // never stored.
      const bool idle = qt * kBR + quarter * 32 >= p.Nq;
      TileWalk tw = walk_of(w, k);   // (idle warps never read it)
      for (int j = 0; j < n_kv; ++j) {
        const int gj = g + j;
        const uint32_t tS = ((gj & 1) ? tS1 : tS0) + lane_off;
        if (!wait_uniform(bar(L::kSFull + (gj & 1)), (gj >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        if (idle) {
          if (j > 0 && j == n_kv - 1 && !wait_uniform(bar(L::kODone), (gj - 1) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_before();
          mbar_arrive(bar(L::kPFull + (gj & 1)));
          continue;
        }
        uint32_t sr[BC];
        #pragma unroll
        for (int c = 0; c < BC / 32; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_ld_wait();
        reg_fence(sr);
        float* s = reinterpret_cast<float*>(sr);
        const int col0 = tw.next(j) * BC;
        const int min_i = packed ? 0 : qt * kBR;
        const bool need_mask = (CAUSAL && col0 + BC - 1 > min_i + p.off) || (col0 + BC > p.Nk);
        if (need_mask) {
          // columns [0, lim) of the tile are kept (one comparison per score)
          const int lim = min(p.Nk - col0, CAUSAL ? qi + p.off - col0 + 1 : BC);
          #pragma unroll
          for (int i = 0; i < BC; ++i)
            if (i >= lim) s[i] = -INFINITY;
        }
        // Row max as a tree of three-input maxima (independent partial maxima
        // keep the single warp per sub-partition busy instead of waiting on a
        // 127-long dependent chain).
        static_assert(BC % 16 == 0, "row max tree covers 16 columns per step");
        float mpart[8];
        #pragma unroll
        for (int u = 0; u < 8; ++u) mpart[u] = fmaxf(s[2 * u], s[2 * u + 1]);
        #pragma unroll
        for (int i = 16; i < BC; i += 16) {
          #pragma unroll
          for (int u = 0; u < 8; ++u) mpart[u] = fmax3(mpart[u], s[i + 2 * u], s[i + 2 * u + 1]);
        }
        const float mx = fmax3(fmax3(mpart[0], mpart[1], mpart[2]), fmax3(mpart[3], mpart[4], mpart[5]),
                               fmaxf(mpart[6], mpart[7]));
        const float m_new = fmaxf(m_ref, mx * p.scale_log2);
        const bool need = m_new > m_ref + kRescaleThreshold;
        const bool any = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (any) {
          alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
          l_r *= alpha;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        uint32_t pk[BC / 2];
        // Exponent arguments two at a time (packed FMA); four independent
        // partial sums of each kind (exact, and of the rounded weights).
        f2 rs[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        float rs_r[4] = {0.f, 0.f, 0.f, 0.f};
        const f2 cs = {p.scale_log2, p.scale_log2}, cm = {-m_use, -m_use};
        #pragma unroll
        for (int i = 0; i < BC / 2; ++i) {
          const f2 arg = ffma2(f2{s[2 * i], s[2 * i + 1]}, cs, cm);
          const f2 pe = {ex2_approx(arg.x), ex2_approx(arg.y)};
          pk[i] = pack2<BF16>(pe.x, pe.y);
          rs[i & 3] = fadd2(rs[i & 3], pe);
          // l_r sums the rounded weights the P V product uses, so the final
          // division of O normalises exactly those weights; L uses the exact l.
          // With the ones chunk the tensor core forms l_r next to O instead.
          if constexpr (!L::kOnes) rs_r[i & 3] = add_packed<BF16>(rs_r[i & 3], pk[i]);
        }
        const f2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
        l += (rs01.x + rs01.y) + (rs23.x + rs23.y);
        l_r += (rs_r[0] + rs_r[1]) + (rs_r[2] + rs_r[3]);
        #pragma unroll
        for (int c = 0; c < BC / 64; ++c)
          tmem_st32(tS + 32 * c, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32 * c]));
        tmem_st_wait();
        // O_DONE completes once per P V product.  S(g) was issued after
        // P V(g-2), and its S_FULL completes only once every earlier product
        // of the issuing thread has, so here only P V(g-1) can be outstanding
        // and the barrier is at P V(g-1)'s phase or one past it: a parity
        // wait for it is exact even when earlier phases were not waited for.
        // It is needed before a rescale of O, and on the last tile (so that
        // at the epilogue only the last product can be outstanding).  The
        // first tile of a unit has no earlier product on O to wait for.
        if (j > 0 && (any || j == n_kv - 1) &&
            !wait_uniform(bar(L::kODone), (gj - 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (any && j > 0) {
          // O holds P_0..P_{j-1} V, all complete: rescale it.
          tc_fence_after();
          #pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o2[64];
            tmem_ld32(tO + lane_off + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(&o2[0]));
            tmem_ld32(tO + lane_off + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(&o2[32]));
            tmem_ld_wait();
            reg_fence(o2);
            #pragma unroll
            for (int i = 0; i < 64; ++i) o2[i] = __float_as_uint(__uint_as_float(o2[i]) * alpha);
            tmem_st32(tO + lane_off + 64 * c, *reinterpret_cast<const uint32_t(*)[32]>(&o2[0]));
            tmem_st32(tO + lane_off + 64 * c + 32, *reinterpret_cast<const uint32_t(*)[32]>(&o2[32]));
          }
          if constexpr (L::kOnes) {
            uint32_t lr[16];
            tmem_ld16(tO + lane_off + D, lr);
            tmem_ld_wait();
            reg_fence(lr);
            #pragma unroll
            for (int i = 0; i < 16; ++i) lr[i] = __float_as_uint(__uint_as_float(lr[i]) * alpha);
            tmem_st16(tO + lane_off + D, lr);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(bar(L::kPFull + (gj & 1)));
      }
      if (!ok) break;
      release_unit(k);
      // ------------------------------------------------------------ epilogue
      const size_t rows_total = static_cast<size_t>(p.B_) * p.H * p.Nq;
      const size_t row_base = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      const bool in_range = row < p.Nq;
      if (n_kv == 0) {
        // no row of this tile sees any key (of this split's range): O = 0,
        // L = -inf, as the final result or as this split's partial
        if (in_range) {
          const size_t r = row_base + row;
          if (p.splits > 1) {
            const size_t rp = split * rows_total + r;
            float4* prow = reinterpret_cast<float4*>(p.o_part + rp * D);
            #pragma unroll
            for (int i = 0; i < D / 4; ++i) prow[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[rp] = -INFINITY;
          } else {
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + b * p.o_sb +
                                                   h * p.o_sh + row * p.o_sn);
            #pragma unroll
            for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[r] = -INFINITY;
          }
        }
        continue;
      }
      if (!wait_uniform(bar(L::kODone), (g + n_kv - 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      if constexpr (L::kOnes) {
        uint32_t lr[16];
        tmem_ld16(tO + lane_off + D, lr);
        tmem_ld_wait();
        reg_fence(lr);
        l_r = __uint_as_float(lr[0]);
      }
      const float inv_l = l_r > 0.f ? 1.f / l_r : 0.f;
      const float lse = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      if (p.splits > 1) {
        // partial result of this key range, combined by fwd_combine_splits
        const size_t r = split * rows_total + row_base + (in_range ? row : 0);
        float4* orow = reinterpret_cast<float4*>(p.o_part + r * D);
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o1[32];
          tmem_ld32(tO + lane_off + 32 * c, o1);
          tmem_ld_wait();
          reg_fence(o1);
          if (in_range) {
            #pragma unroll
            for (int i = 0; i < 8; ++i)
              orow[c * 8 + i] = make_float4(
                  __uint_as_float(o1[4 * i]) * inv_l, __uint_as_float(o1[4 * i + 1]) * inv_l,
                  __uint_as_float(o1[4 * i + 2]) * inv_l, __uint_as_float(o1[4 * i + 3]) * inv_l);
          }
        }
        if (in_range) p.lse_part[r] = lse;
      } else {
        uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + b * p.o_sb +
                                               h * p.o_sh + (in_range ? row : 0) * p.o_sn);
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o1[32];
          tmem_ld32(tO + lane_off + 32 * c, o1);
          tmem_ld_wait();
          reg_fence(o1);
          uint32_t wv[16];
          #pragma unroll
          for (int i = 0; i < 16; ++i)
            wv[i] = pack2<BF16>(__uint_as_float(o1[2 * i]) * inv_l, __uint_as_float(o1[2 * i + 1]) * inv_l);
          if (in_range) {
            #pragma unroll
            for (int i = 0; i < 4; ++i)
              orow[c * 4 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
          }
        }
        if (in_range) p.lse[row_base + row] = lse;
      }
      g += n_kv;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort == 2) atomicOr(p.err, kErrTimeout);
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// d = 128, two query tiles per CTA (the path for long queries), persistent.
//
// With one tile per CTA the tensor pipe idles while the softmax of tile j
// runs (P V_j needs P_j) and the softmax warps idle while the products run.
// Here a work unit is two query tiles A and B (rows [256 t, 256 t + 128) and
// [256 t + 128, 256 t + 256) of one head) with one softmax warpgroup each;
// every key tile is loaded once for both, and the MMA warp interleaves the
// tiles:  P V_A(j), S_A(j+1), P V_B(j), S_B(j+1), ...
// so while one warpgroup exponentiates, the pipe works for the other.
// TMEM: S_A, S_B, O_A, O_B (128 columns each; P written over S in 16 bits).
// The row sums are formed on the ALU (no room for the ones columns), and O
// is divided by the exact sum of the weights.
//
// Persistent: one CTA per SM walks a list of units ordered by length under
// the mask (see fwd2_unit), taking one unit of every round of gridDim.x
// (forwards and backwards in turn, see fwd2_unit_index).  TMEM,
// barriers and the K/V ring live across units (phase counters continue), the
// next unit's scores start while the previous unit's epilogue drains O, and
// its K/V tiles stream behind the previous unit's without a gap.
// Warps: 0 TMA producer, 1 MMA issuer, 2..5 softmax tile A, 6..9 tile B.
constexpr int kFwd2Threads = 320;

struct Fwd2Layout {
  static constexpr int kTile = 128 * 128 * 2;   // one 128 x 128 16-bit tile (32 KB)
  static constexpr int kQOff = 0;               // Q_A, Q_B
  static constexpr int kKOff = 2 * kTile;       // two stages
  static constexpr int kVOff = 4 * kTile;       // two stages
  static constexpr int kBarOff = 6 * kTile;
  static constexpr int kQFull = 0, kQEmpty = 1, kKFull = 2, kKEmpty = 4, kVFull = 6,
                       kVEmpty = 8, kSFull = 10, kPFull = 12, kODone = 14, kOFree = 16,
                       kDrain = 18, kNumBars = 19;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTS = 0, kTO = 256, kTmemCols = 512;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// Work unit x of the persistent forward: 256-row block, head, batch, and the
// key tiles of its two query tiles (0 if a tile holds no query row, or if
// under the mask none of its rows sees a key).
struct Fwd2Unit {
  int blk, h, b, n_kv[2], n_max;
};

template <bool CAUSAL>
__device__ __forceinline__ Fwd2Unit fwd2_unit(const FwdParams& p, int x) {
  Fwd2Unit w;
  int bh;
  if (CAUSAL) {
    // (batch, head) pairs in sections whose K / V fit in L2 together, the
    // section's heads innermost.  The last section walks its 256-row blocks
    // longest first, the one before shortest first, and so on: unit lengths
    // along the list rise and fall without jumps and end with the shortest,
    // which keeps the round assignment balanced.
    const int hb = p.H * p.B_;
    const int n_sec = (hb + p.sec_heads - 1) / p.sec_heads;
    const int per_sec = p.sec_heads * p.num_q_tiles;
    const int sec = x / per_sec, r = x - sec * per_sec;
    const int width = min(p.sec_heads, hb - sec * p.sec_heads);
    const int k = r / width;
    w.blk = ((n_sec - 1 - sec) & 1) ? k : p.num_q_tiles - 1 - k;
    bh = sec * p.sec_heads + r % width;
  } else {
    // consecutive units are consecutive blocks of one head (shared K / V)
    w.blk = x % p.num_q_tiles;
    bh = x / p.num_q_tiles;
  }
  w.b = bh / p.H;
  w.h = bh - w.b * p.H;
  #pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int first = w.blk * 256 + 128 * u;
    w.n_kv[u] = (p.Nk + 127) / 128;
    if (first >= p.Nq) {
      w.n_kv[u] = 0;
    } else if (CAUSAL) {
      const int last_key = min(first + 128, p.Nq) - 1 + p.off;
      w.n_kv[u] = last_key < 0 ? 0 : min(w.n_kv[u], last_key / 128 + 1);
    }
  }
  w.n_max = max(w.n_kv[0], w.n_kv[1]);
  return w;
}

// The i-th unit of this CTA, or -1 past the end: rounds of gridDim.x units,
// walked forwards in even rounds and backwards in odd ones, so that over two
// rounds of a longest-first list every CTA gets about the same work.
__device__ __forceinline__ int fwd2_unit_index(int i, int n_units) {
  const int base = i * static_cast<int>(gridDim.x);
  const int x = base + ((i & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                                 : static_cast<int>(blockIdx.x));
  return (base < n_units && x < n_units) ? x : -1;
}

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kFwd2Threads, 1)
fwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Fwd2Layout;
  constexpr int D = 128, BC = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = p.num_q_tiles * p.H * p.B_;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 4);      // one arrival per softmax warp
      mbar_init(bar(L::kODone + s), 1);
      mbar_init(bar(L::kOFree + s), 128);
    }
    mbar_init(bar(L::kDrain), 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    __syncwarp();
    int it = 0, kt = 0;                 // units and key tiles loaded so far
    int k_issued = 0, v_issued = 0, q_issued = 0;
    bool ok = true;
    auto load_kv = [&](const Fwd2Unit& w, int j) -> bool {
      const int g = kt + j, s = g & 1;
      const int kh = w.h / p.G;
      if (g >= 2 && !wait_uniform(bar(L::kKEmpty + s), ((g >> 1) + 1) & 1, abort)) return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kKFull + s), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kKOff + s * L::kTile + c * (BC * 128), &tm_k, bar(L::kKFull + s),
                      c * 64, j * BC, kh, w.b);
      }
      __syncwarp();
      ++k_issued;
      if (g >= 2 && !wait_uniform(bar(L::kVEmpty + s), ((g >> 1) + 1) & 1, abort)) return false;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kVFull + s), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kVOff + s * L::kTile + c * (BC * 128), &tm_v, bar(L::kVFull + s),
                      c * 64, j * BC, kh, w.b);
      }
      __syncwarp();
      ++v_issued;
      return true;
    };
    for (int x = fwd2_unit_index(0, n_units); ok && x >= 0; x = fwd2_unit_index(++it, n_units)) {
      const Fwd2Unit w = fwd2_unit<CAUSAL>(p, x);
      // the first key tile streams behind the previous unit's; Q waits until
      // the previous unit's scores have all been issued and have completed
      if (w.n_max > 0 && !load_kv(w, 0)) { ok = false; break; }
      if (it >= 1 && !wait_uniform(bar(L::kQEmpty), (it - 1) & 1, abort)) { ok = false; break; }
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kQFull), 2 * L::kTile);
        #pragma unroll
        for (int u = 0; u < 2; ++u) {
          #pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sbase + L::kQOff + u * L::kTile + c * (128 * 128), &tm_q, bar(L::kQFull),
                        c * 64, w.blk * 256 + 128 * u, w.h, w.b);
        }
      }
      __syncwarp();
      ++q_issued;
      for (int j = 1; j < w.n_max; ++j)
        if (!load_kv(w, j)) { ok = false; break; }
      kt += w.n_max;
    }
    if (q_issued > 0) drain_wait(bar(L::kQFull), (q_issued - 1) & 1);
    for (int g = max(0, k_issued - 2); g < k_issued; ++g)
      drain_wait(bar(L::kKFull + (g & 1)), (g >> 1) & 1);
    for (int g = max(0, v_issued - 2); g < v_issued; ++g)
      drain_wait(bar(L::kVFull + (g & 1)), (g >> 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(128, BC, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t kIdO = idesc_f16(128, D, BF16 ? 1 : 0, 0, 1);
    const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sbase + L::kVOff, BC * 128, 1024);
    auto issue_s = [&](int u, int stage) {
      const uint64_t qs = desc_add(q_desc, u * L::kTile);
      const uint64_t ks = desc_add(k_desc, stage * L::kTile);
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tmem + L::kTS + 128 * u, desc_add(qs, c * (128 * 128) + w * 32),
               desc_add(ks, c * (BC * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull + u));
    };
    int it = 0, kt = 0;
    int cp[2] = {0, 0};                  // P_FULL phases consumed per tile
    int of[2] = {0, 0};                  // units so far with products on each tile
    bool ok = true;
    for (int x = fwd2_unit_index(0, n_units); ok && x >= 0; x = fwd2_unit_index(++it, n_units)) {
      const Fwd2Unit w = fwd2_unit<CAUSAL>(p, x);
      if (!wait_uniform(bar(L::kQFull), it & 1, abort)) { ok = false; break; }
      if (w.n_max > 0) {
        if (!wait_uniform(bar(L::kKFull + (kt & 1)), (kt >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        if (w.n_kv[0] > 0) issue_s(0, kt & 1);
        if (w.n_kv[1] > 0) issue_s(1, kt & 1);
        mma_commit(bar(L::kKEmpty + (kt & 1)));
      }
      // Q is free for the next unit once the last score product of this one
      // completes (the scores of key tile j + 1 are issued in step j)
      if (w.n_max <= 1) mma_commit(bar(L::kQEmpty));
      // the last epilogue that read O_u out is done before P V overwrites it
      // (O_FREE completes once per unit with products on the tile, so it
      // never runs two phases ahead of this wait)
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (w.n_kv[u] > 0 && of[u] > 0 && !wait_uniform(bar(L::kOFree + u), (of[u] - 1) & 1, abort)) {
          ok = false;
          break;
        }
        of[u] += w.n_kv[u] > 0 ? 1 : 0;
      }
      if (!ok) break;
      for (int j = 0; ok && j < w.n_max; ++j) {
        const int g = kt + j, s = g & 1;
        if (!wait_uniform(bar(L::kVFull + s), (g >> 1) & 1, abort)) { ok = false; break; }
        // K(g + 1) (loaded a stage ahead) before the P waits, so that no wait
        // sits between P V and the next scores
        const bool k_ready = j + 1 < w.n_max;
        if (k_ready &&
            !wait_uniform(bar(L::kKFull + ((g + 1) & 1)), ((g + 1) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        #pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (j >= w.n_kv[u]) continue;
          if (!wait_uniform(bar(L::kPFull + u), cp[u] & 1, abort)) { ok = false; break; }
          ++cp[u];
          tc_fence_after();
          const uint64_t vs = desc_add(v_desc, s * L::kTile);
          #pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_ts(tmem + L::kTO + 128 * u, tmem + L::kTS + 128 * u + kk * 8,
                   desc_add(vs, kk * 2048), kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kODone + u));
          if (j + 1 < w.n_kv[u]) {
            issue_s(u, (g + 1) & 1);
          }
        }
        if (!ok) break;
        mma_commit(bar(L::kVEmpty + s));
        if (k_ready) mma_commit(bar(L::kKEmpty + ((g + 1) & 1)));
        if (j + 2 == w.n_max) mma_commit(bar(L::kQEmpty));
      }
      kt += w.n_max;
    }
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int u = (warp - 2) >> 2;                // query tile of this warpgroup
    const int quarter = warp & 3;
    const int r_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + L::kTS + 128 * u + lane_off;
    const uint32_t tO = tmem + L::kTO + 128 * u + lane_off;
    int cs = 0, co = 0;                           // S_FULL / O_DONE phases consumed
    bool ok = true;
    for (int i = 0, x = fwd2_unit_index(0, n_units); ok && x >= 0;
         x = fwd2_unit_index(++i, n_units)) {
      int row0, nk;                               // first row of the tile, its key tiles
      {
        const Fwd2Unit w = fwd2_unit<CAUSAL>(p, x);
        row0 = w.blk * 256 + 128 * u;
        nk = w.n_kv[u];
      }
      const int row = row0 + r_tile;
      float m_ref = -INFINITY, l = 0.f;
      const bool idle = row0 + quarter * 32 >= p.Nq;
      for (int j = 0; j < nk; ++j) {
        if (!wait_uniform(bar(L::kSFull + u), cs & 1, abort)) { ok = false; break; }
        ++cs;
        tc_fence_after();
        if (idle) {
          tc_fence_before();
          mbar_arrive_warp(bar(L::kPFull + u));
          continue;
        }
        const int col0 = j * BC;
        const bool need_mask =
            (CAUSAL && col0 + BC - 1 > row0 + p.off) || (col0 + BC > p.Nk);
        uint32_t sr[BC];
        #pragma unroll
        for (int c = 0; c < BC / 32; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_ld_wait();
        reg_fence(sr);
        float* s = reinterpret_cast<float*>(sr);
        if (need_mask) {
          // columns [0, lim) of the tile are kept: key < Nk and (causal)
          // key <= row + off, one comparison per score
          const int lim = min(p.Nk - col0, CAUSAL ? row + p.off - col0 + 1 : BC);
          #pragma unroll
          for (int i = 0; i < BC; ++i)
            if (i >= lim) s[i] = -INFINITY;
        }
        float mpart[8];
        #pragma unroll
        for (int uu = 0; uu < 8; ++uu) mpart[uu] = fmaxf(s[2 * uu], s[2 * uu + 1]);
        #pragma unroll
        for (int i = 16; i < BC; i += 16) {
          #pragma unroll
          for (int uu = 0; uu < 8; ++uu) mpart[uu] = fmax3(mpart[uu], s[i + 2 * uu], s[i + 2 * uu + 1]);
        }
        const float mx = fmax3(fmax3(mpart[0], mpart[1], mpart[2]), fmax3(mpart[3], mpart[4], mpart[5]),
                               fmaxf(mpart[6], mpart[7]));
        const float m_new = fmaxf(m_ref, mx * p.scale_log2);
        const bool need = m_new > m_ref + kRescaleThreshold;
        const bool any = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (any) {
          alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_new);
          m_ref = m_new;
          l *= alpha;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // weights written over S as 16 bits, 32 columns at a time; the exact
        // sum l serves both L and the final division (rounding to nearest
        // leaves the rounded weights' sum unbiased)
        f2 rs[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        const f2 cs2 = {p.scale_log2, p.scale_log2}, cm = {-m_use, -m_use};
        #pragma unroll
        for (int c = 0; c < BC / 32; ++c) {
          uint32_t pk[16];
          #pragma unroll
          for (int i = 0; i < 16; ++i) {
            const f2 arg = ffma2(f2{s[32 * c + 2 * i], s[32 * c + 2 * i + 1]}, cs2, cm);
            const f2 pe = {ex2_approx(arg.x), ex2_approx(arg.y)};
            pk[i] = pack2<BF16>(pe.x, pe.y);
            rs[i & 3] = fadd2(rs[i & 3], pe);
          }
          tmem_st16(tS + 16 * c, pk);
        }
        const f2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
        l += (rs01.x + rs01.y) + (rs23.x + rs23.y);
        tmem_st_wait();
        // O needs no wait before its rescale: S(j) was issued after P V(j-1)
        // on this tile, and its S_FULL completes only once every earlier
        // product has (tcgen05.commit tracks all of the issuing thread's prior
        // products), so P V(j-1) is done and P V(j) waits for this P_FULL
        if (any && j > 0) {
          tc_fence_after();
          #pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o2[64];
            tmem_ld32(tO + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(&o2[0]));
            tmem_ld32(tO + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(&o2[32]));
            tmem_ld_wait();
            reg_fence(o2);
            #pragma unroll
            for (int i = 0; i < 64; ++i) o2[i] = __float_as_uint(__uint_as_float(o2[i]) * alpha);
            tmem_st32(tO + 64 * c, *reinterpret_cast<const uint32_t(*)[32]>(&o2[0]));
            tmem_st32(tO + 64 * c + 32, *reinterpret_cast<const uint32_t(*)[32]>(&o2[32]));
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive_warp(bar(L::kPFull + u));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      const bool in_range = row < p.Nq;
      const Fwd2Unit w = fwd2_unit<CAUSAL>(p, x);   // recomputed: h and b
      const size_t lrow = (static_cast<size_t>(w.b) * p.H + w.h) * p.Nq + (in_range ? row : 0);
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + w.b * p.o_sb +
                                             w.h * p.o_sh + (in_range ? row : 0) * p.o_sn);
      if (nk == 0) {
        // no row of this tile sees any key: O = 0, L = -inf
        if (in_range) {
          #pragma unroll
          for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[lrow] = -INFINITY;
        }
      } else {
        // O_DONE completes once per P V product of the tile and only the
        // unit's last one is waited for: P V(nk-2) is done (see above), so
        // the barrier is at that product's phase or one past it
        co += nk;
        if (!wait_uniform(bar(L::kODone + u), (co - 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o1[32];
          tmem_ld32(tO + 32 * c, o1);
          tmem_ld_wait();
          reg_fence(o1);
          uint32_t wv[16];
          #pragma unroll
          for (int i = 0; i < 16; ++i)
            wv[i] = pack2<BF16>(__uint_as_float(o1[2 * i]) * inv_l,
                                __uint_as_float(o1[2 * i + 1]) * inv_l);
          if (in_range) {
            #pragma unroll
            for (int i = 0; i < 4; ++i)
              orow[c * 4 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
          }
        }
        if (in_range) p.lse[lrow] = lse;
        // O of this tile has been read out: the next P V may overwrite it
        tc_fence_before();
        mbar_arrive(bar(L::kOFree + u));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort == 2) atomicOr(p.err, kErrTimeout);
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <bool CAUSAL, bool BF16>
cudaError_t launch_fwd2(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  using L = Fwd2Layout;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  if ((e = make_tmap_4d(&tq, a.q, 128, pr.Nq, pr.H, pr.B, a.qs, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tk, a.k, 128, pr.Nk, pr.Hkv, pr.B, a.ks, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, 128, pr.Nk, pr.Hkv, pr.B, a.vs, 64, 128)) != cudaSuccess) return e;
  auto kern = fwd2_kernel<CAUSAL, BF16>;
  static bool attr_set = false;
  static int n_sms = 0;
  if (!attr_set) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    attr_set = true;
  }
  FwdParams p = {};
  p.o = a.o;
  p.lse = a.lse;
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.G = pr.H / pr.Hkv;
  p.B_ = pr.B;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.mask_rows = pr.Nq;
  p.num_q_tiles = (pr.Nq + 255) / 256;
  p.splits = 1;
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  p.o_sb = a.os.b;
  p.o_sh = a.os.h;
  p.o_sn = a.os.n;
  p.err = pr.err;
  // causal order: sections of (batch, head) pairs whose K and V (2 Nk d
  // 16-bit values per KV head) take about 64 MB of L2 together
  {
    const long long kv_head = 4ll * pr.Nk * 128;
    const long long kv_heads = std::max<long long>(1, (64ll << 20) / kv_head);
    p.sec_heads = static_cast<int>(std::min<long long>(kv_heads * p.G, 1ll * pr.H * pr.B));
  }
  const long long n_units = static_cast<long long>(p.num_q_tiles) * pr.H * pr.B;
  if (n_units >= (1ll << 31)) return cudaErrorInvalidValue;   // unit indices are int
  dim3 grid(static_cast<unsigned>(std::min<long long>(n_units, std::max(n_sms, 1))), 1, 1);
  const int slot = timing_begin(FA_KERNEL_FWD, stream);
  kern<<<grid, kFwd2Threads, L::kAlloc, stream>>>(tq, tk, tv, p);
  timing_end(slot, stream);
  return cudaGetLastError();
}

// Merge the per-split partial results of one query row: with L_s the split
// logsumexps, L = ln sum_s exp(L_s) and O = sum_s exp(L_s - L) O_s.  One warp
// per row: lane s holds split s's weight, and the partial rows of up to 8
// splits are loaded before they are summed (a split without keys for the row
// left O_s = 0 and L_s = -inf, weight 0).  Launched as the split kernel's
// programmatic dependent: it waits for the partials here.  A row no split
// has a key for gets O = 0, L = -inf.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
fwd_combine_splits(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                   uint16_t* __restrict__ o, float* __restrict__ lse, size_t rows, int splits,
                   int H, int Nq, Strides os) {
  grid_dependency_wait();
  const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int kPer = D / 32;
  float m = -INFINITY;
  for (int s0 = 0; s0 < splits; s0 += 32)
    if (s0 + lane < splits) m = fmaxf(m, lse_part[(s0 + lane) * rows + row]);
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  // row = (b * H + h) * Nq + i of the output view
  const size_t bh = row / Nq;
  const long long i = static_cast<long long>(row - bh * Nq);
  const long long hh = static_cast<long long>(bh % H), bb = static_cast<long long>(bh / H);
  uint16_t* orow = o + bb * os.b + hh * os.h + i * os.n + lane * kPer;
  if (m == -INFINITY) {
    #pragma unroll
    for (int i = 0; i < kPer; i += 2) *reinterpret_cast<uint32_t*>(orow + i) = 0u;
    if (lane == 0) lse[row] = -INFINITY;
    return;
  }
  float acc[kPer];
  #pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float sum = 0.f;
  for (int s0 = 0; s0 < splits; s0 += 32) {
    const int n = min(32, splits - s0);
    const float ls = lane < n ? lse_part[(s0 + lane) * rows + row] : -INFINITY;
    const float wl = ls == -INFINITY ? 0.f : expf(ls - m);
    sum += wl;
    #pragma unroll 8
    for (int k = 0; k < n; ++k) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      const float* src = o_part + ((s0 + k) * rows + row) * D + lane * kPer;
      float x[kPer];
      if constexpr (kPer == 2) {
        const float2 t = *reinterpret_cast<const float2*>(src);
        x[0] = t.x; x[1] = t.y;
      } else {
        #pragma unroll
        for (int c = 0; c < kPer; c += 4) {
          const float4 t = *reinterpret_cast<const float4*>(src + c);
          x[c] = t.x; x[c + 1] = t.y; x[c + 2] = t.z; x[c + 3] = t.w;
        }
      }
      #pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] = fmaf(w, x[c], acc[c]);
    }
  }
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = 1.f / sum;
  #pragma unroll
  for (int i = 0; i < kPer; i += 2)
    *reinterpret_cast<uint32_t*>(orow + i) = pack2<BF16>(acc[i] * inv, acc[i + 1] * inv);
  if (lane == 0) lse[row] = m + logf(sum);
}

template <int D, int BC, bool CAUSAL, bool BF16, int KST, int VST, bool SPARSE>
cudaError_t launch_variant(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, BC, KST, VST>;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  if ((e = make_tmap_4d(&tk, a.k, D, pr.Nk, pr.Hkv, pr.B, a.ks, 64, BC)) != cudaSuccess) return e;
  // V in halves of BC / 2 keys when the rings hold pieces of tiles
  if ((e = make_tmap_4d(&tv, a.v, D, pr.Nk, pr.Hkv, pr.B, a.vs, 64, L::kChunked ? BC / 2 : BC)) !=
      cudaSuccess)
    return e;
  auto kern = fwd_kernel<D, BC, CAUSAL, BF16, KST, VST, SPARSE>;
  // without a block mask the list is never touched and not allocated
  constexpr int kSmem = SPARSE ? L::kAlloc : L::kAllocDense;   // (records only with a block mask)
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int G = pr.H / pr.Hkv;
  FwdParams p;
  p.o = a.o;
  p.lse = a.lse;
  // Packed: the G heads of a group are G * Nq consecutive rows of q, o and
  // lse, so the group runs as one "head" of G * Nq query rows.
  p.H = a.pack ? pr.Hkv : pr.H;
  p.Hkv = pr.Hkv;
  p.G = a.pack ? 1 : G;
  p.Nq = a.pack ? G * pr.Nq : pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.mask_rows = pr.Nq;
  p.num_q_tiles = (p.Nq + kBR - 1) / kBR;
  p.scale_log2 = pr.scale * 1.4426950408889634f;
  p.err = pr.err;
  p.B_ = pr.B;
  const int n_kv_tiles = (pr.Nk + BC - 1) / BC;
  p.splits = 1;
  p.tiles_per_split = n_kv_tiles;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.mask = a.mask;
  if (a.splits > 1) {
    p.tiles_per_split = (n_kv_tiles + a.splits - 1) / a.splits;
    p.splits = (n_kv_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  }
  // Packed: row r = g * Nq + i of KV group kh is query head kh * G + g, row i;
  // the caller packs only when those rows are evenly spaced (Nq == 1, or
  // head stride == Nq * row stride), so the group is one strided view.
  Strides qv = a.qs, ov = a.os;
  if (a.pack) {
    qv = {a.qs.b, G * a.qs.h, pr.Nq == 1 ? a.qs.h : a.qs.n};
    ov = {a.os.b, G * a.os.h, pr.Nq == 1 ? a.os.h : a.os.n};
  }
  p.o_sb = ov.b;
  p.o_sh = ov.h;
  p.o_sn = ov.n;
  if ((e = make_tmap_4d(&tq, a.q, D, p.Nq, p.H, pr.B, qv, 64, kBR)) != cudaSuccess) return e;
  // persistent: one CTA per SM walking the units
  static int n_sms = 0;
  if (n_sms == 0) {
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
  }
  const long long n_units = static_cast<long long>(p.num_q_tiles) * p.splits * p.H * pr.B;
  if (n_units >= (1ll << 31)) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(std::min<long long>(n_units, std::max(n_sms, 1))), 1, 1);
  const int slot = timing_begin(FA_KERNEL_FWD, stream);
  kern<<<grid, kThreads, kSmem, stream>>>(tq, tk, tv, p);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!SPARSE && p.splits > 1) {
    // the merge is the split kernel's programmatic dependent: its launch and
    // first instructions overlap the split kernel's last CTAs
    const size_t rows = static_cast<size_t>(pr.B) * pr.H * pr.Nq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fwd_combine_splits<D, BF16>, static_cast<const float*>(a.o_part),
                           static_cast<const float*>(a.lse_part), static_cast<uint16_t*>(a.o),
                           a.lse, rows, p.splits, pr.H, pr.Nq, a.os);
  }
  return e;
}

template <int D, int BC, int KST, int VST, bool SPARSE>
cudaError_t dispatch_flags(const Problem& pr, const FwdArgs& a, cudaStream_t s) {
  if (pr.causal) {
    return pr.bf16 ? launch_variant<D, BC, true, true, KST, VST, SPARSE>(pr, a, s)
                   : launch_variant<D, BC, true, false, KST, VST, SPARSE>(pr, a, s);
  }
  return pr.bf16 ? launch_variant<D, BC, false, true, KST, VST, SPARSE>(pr, a, s)
                 : launch_variant<D, BC, false, false, KST, VST, SPARSE>(pr, a, s);
}

// Tile configuration per head dimension: key tile BC, K and V ring stages.
template <bool SPARSE>
cudaError_t launch_fwd_for(const Problem& pr, const FwdArgs& a, cudaStream_t stream) {
  // d = 128, long queries, one pass: two query tiles per CTA
  if (!SPARSE && pr.d == 128 && !a.pack && a.splits <= 1 && pr.Nq > 128) {
    if (pr.causal)
      return pr.bf16 ? launch_fwd2<true, true>(pr, a, stream) : launch_fwd2<true, false>(pr, a, stream);
    return pr.bf16 ? launch_fwd2<false, true>(pr, a, stream) : launch_fwd2<false, false>(pr, a, stream);
  }
  switch (pr.d) {
    case 64: return dispatch_flags<64, 128, 3, 3, SPARSE>(pr, a, stream);
    case 128: return dispatch_flags<128, 128, 2, 2, SPARSE>(pr, a, stream);
    // d = 256: 128-key tiles through rings of pieces (six K chunks and two
    // V halves; five K chunks with a block mask, whose unit records also
    // need shared memory)
    case 256: return dispatch_flags<256, 128, SPARSE ? 5 : 6, 2, SPARSE>(pr, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace fa
