// Backward kernels of exact attention on sm_103a: dQ, dK, dV of sum(O o dO).
// Instantiated dense in fa_bwd.cu and block-sparse in fa_bwd_blocksparse.cu.
//
// Method ("FlashAttention-2: Faster Attention with Better Parallelism and
// Work Partitioning", paper digest):
//  - section 2 Q2, improvement 2 (backward): the outer loop runs over
//    key/value tiles; dK and dV stay on chip for the whole loop, and dQ is
//    accumulated across key/value tiles with atomic adds;
//  - section 4 "logsumexp fusion": the softmax weights are rebuilt from the
//    saved L as P = exp(S - L), so S and P are never stored;
//  - section 4 notation table: D = rowsum(dO o O), computed once up front;
//  - section 3 "FLOPs": five products per tile, S = Q K^T, dP = dO V^T,
//    dV += P^T dO, dK += dS^T Q, dQ += dS K with dS = P o (dP - D);
//  - section 4 "six checks", GQA/MQA: dK and dV sum over the query heads
//    sharing a key/value head; here one CTA loops over all of them, so that
//    sum needs no atomics.
// Under a block mask (block-sparse attention, "FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", abstract) a CTA walks
// only the (head, query tile) steps whose mask block with its key tile is
// kept; a key tile with no step gets dK = dV = 0.
//
// Three kernels: preprocess (D and a zeroed fp32 dQ accumulator), a main
// kernel, and a conversion of the accumulator to the output dtype (with the
// softmax scale applied).  The main kernels here: bwd_kernel (d = 64, and
// d = 256 under a block mask) and bwd128_kernel (d = 128: the key-outer half
// of the reproducible backward, and the block-sparse backward).  The default
// dense d = 128 backward runs the fused kernel of fa_bwd_fused_kernel.cuh,
// which uses the preprocess and conversion kernels of this file; the dense
// d = 256 backward runs the cluster pair of fa_bwd_pair_kernel.cuh (dK, dV)
// and the query-outer dQ kernel of fa_bwd_dq_kernel.cuh.
//
// bwd_kernel, one CTA per (batch, key/value head, 128-key tile[, half of
// d when d = 256]); 10 warps:
//   warp 0      TMA producer: K and V once, then (Q_i, dO_i) tiles;
//   warp 1      MMA issuer (tcgen05, fp32 accumulators in TMEM);
//   warps 2..5  one key row per thread: P^T = exp(S^T - L) with the masks,
//               written to TMEM (16-bit) as the A operand of dV += P^T dO;
//               dS^T = P^T o (dP^T - D) written to shared memory (128-byte
//               swizzle) as the operand of dK += dS^T Q and of dQ;
//               epilogue for dK (times scale) and dV;
//   warps 6..9  read the dQ tile out of TMEM and add it to the fp32
//               accumulator in global memory (red.global.add).
// S^T and dP^T are computed with keys on the TMEM lanes (M = 128) so the
// dK/dV accumulators and the score tiles share one layout.  Two tile shapes:
//   d = 64:  128 query rows per step; dQ = dS K (query rows on lanes).
//   d = 256: 64 query rows per step; dQ^T = K^T dS^T (d on lanes), split
//            over two CTAs by output half of d (S^T and dP^T are computed by
//            both), because dK + dV for all 256 columns would fill TMEM.
// (bwd128_kernel, below, has its own description.)
#pragma once

#include <type_traits>

#include "block_list.cuh"
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int kBC = 128;        // key rows per CTA
constexpr int kBwdThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

// Bit of the device error word: the dynamic shared memory base was not
// 1024-byte aligned and the layout did not fit behind the aligned base.
constexpr unsigned int kErrSmemBase = 2u;

template <int D, int DH, int BR, int QST>
struct BwdLayout {
  static constexpr bool kDqT = (BR == 64);
  static constexpr int kNch = D / 64;
  static constexpr int kKBytes = kBC * D * 2;
  static constexpr int kQBytes = BR * D * 2;
  static constexpr int kDSBytes = kBC * BR * 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKBytes;
  static constexpr int kQOff = kVOff + kKBytes;
  static constexpr int kDOOff = kQOff + QST * kQBytes;
  static constexpr int kDSOff = kDOOff + QST * kQBytes;
  // Two score buffers in TMEM when there is room for them and the Q/dO ring
  // can hold the next tile while the current one is still in use.
  static constexpr int kSBuf = (kDqT && QST >= 2) ? 2 : 1;
  static constexpr int kLDOff = kDSOff + kDSBytes;   // 4 warps x 2 bufs x {-L*log2e, -D} [BR]
  static constexpr int kBarOff = kLDOff + 4 * 2 * 2 * BR * 4;
  static constexpr int kKVFull = 0;
  static constexpr int kQDFull = 1;
  static constexpr int kQDEmpty = kQDFull + QST;
  static constexpr int kSFull = kQDEmpty + QST;     // one per score buffer
  static constexpr int kDPFull = kSFull + 2;
  static constexpr int kPFull = kDPFull + 1;
  static constexpr int kDSFull = kPFull + 1;
  static constexpr int kDSEmpty = kDSFull + 1;
  static constexpr int kDQFull = kDSEmpty + 1;
  static constexpr int kDQEmpty = kDQFull + 1;
  static constexpr int kFinal = kDQEmpty + 1;
  static constexpr int kDrain = kFinal + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // (head, query tile) steps kept under a block mask
  static constexpr int kListCap = D == 256 ? 4096 : 8192;
  static constexpr int kListOff = kMiscOff + 16;
  static constexpr int kBytes = kListOff + kListCap * 2;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kAllocDense = kListOff + 1024;   // without the list
  // TMEM columns
  static constexpr uint32_t kTdV = 0, kTdK = DH, kTS = 2 * DH, kTdP = 2 * DH + kSBuf * BR,
                            kTdQ = 2 * DH + (kSBuf + 1) * BR;
  static constexpr uint32_t kDqCols = kDqT ? BR : D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kTdQ + kDqCols <= kTmemCols, "TMEM budget");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kDqT ? (DH == 128) : (BR == 128 && D == DH), "tile shapes");
};

struct BwdParams {
  const float* lse;
  const float* delta;
  float* dq_acc;
  uint16_t* dk;
  uint16_t* dv;
  int H, Hkv, G;
  int Nq, Nk;         // query / key lengths
  int off;            // Nk - Nq: under the mask query i sees keys k <= i + off
  int n_q_tiles;
  float scale, scale_log2;
  int heavy_first;   // dispatch order, see bwd_kernel
  int with_dq;       // 0: dK and dV only (dQ comes from the query-outer kernel)
  BlockMask mask;    // block-sparse: only the kept blocks' steps
  Strides dks, dvs;  // element strides of dk, dv
  unsigned int* err;
  // persistent fused kernel: work counter (zero at launch), units = key
  // tiles x groups, groups = (batch, kv head) pairs, and how many of the last
  // groups are taken heavy first in the key-tile-fastest order
  unsigned int* units;
  int n_units, n_kv_tiles, n_groups, tail_groups;
  // One key tile in all (keys <= 128, d = 64): every (head, query tile) has a
  // single dQ contribution, so bwd_kernel forms D itself from O and dO and
  // writes dQ (times scale, in the output dtype) directly: one launch for the
  // whole backward, no accumulator
  int direct = 0;
  const uint16_t* o = nullptr;
  const uint16_t* dout = nullptr;
  uint16_t* dq = nullptr;
  Strides os, dos, dqs;
};

template <int D, int DH, int BR, int QST, bool CAUSAL, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
           const BwdParams p) {
  using L = BwdLayout<D, DH, BR, QST>;
  constexpr int kNSplit = D / DH;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  int* list_count = reinterpret_cast<int*>(smem + L::kMiscOff + 8);
  uint16_t* step_list = reinterpret_cast<uint16_t*>(smem + L::kListOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Two dispatch orders (chosen on the host):
  //  - key tiles vary fastest, so the CTAs of one (batch, kv head) group run
  //    together and share its Q / dO tiles in L2;
  //  - heavy first: under the mask the work of a CTA falls with its key tile,
  //    so when single CTAs are long, every group's heaviest tiles go first and
  //    the last wave holds only short CTAs.
  int jt, dh, kh, b;
  if (p.heavy_first) {
    jt = blockIdx.y;
    dh = blockIdx.x % kNSplit;
    kh = (blockIdx.x / kNSplit) % p.Hkv;
    b = blockIdx.x / (kNSplit * p.Hkv);
  } else {
    jt = blockIdx.x / kNSplit;
    dh = blockIdx.x % kNSplit;
    kh = blockIdx.y;
    b = blockIdx.z;
  }
  const int kv0 = jt * kBC;
  // first query tile with a row that sees key kv0 (i + off >= kv0)
  const int i0 = CAUSAL ? max(0, kv0 - p.off) / BR : 0;
  const int n_i = p.n_q_tiles - i0;
  int n_steps = p.G * n_i;
  constexpr bool sparse = SPARSE;
  // Step order: query tiles from the last down to i0, the G heads of the
  // group innermost.  CTAs of a group that run together then work on the
  // same query tiles at the same time, so the dQ accumulator rows they add
  // into (and the Q / dO tiles they load) stay in L2.
  if (sparse && warp == 2) {
    // the kept steps of that order: mask block (query block of tile i, this
    // key tile) nonzero for head g's pattern
    const int cnt = compact_steps<1>(
        p.G * n_i,
        [&](int e) {
          const int i = p.n_q_tiles - 1 - e / p.G, g = e % p.G;
          const int mh = p.mask.heads == 1 ? 0 : kh * p.G + g;
          const int qb = i * BR / kMaskBlock;
          return p.mask.ptr[(static_cast<size_t>(mh) * p.mask.nbr + qb) * p.mask.nbc + jt] != 0;
        },
        [&](int e, int) {
          const int i = p.n_q_tiles - 1 - e / p.G, g = e % p.G;
          return g * p.n_q_tiles + i;
        },
        step_list, L::kListCap);
    if (lane == 0) *list_count = min(cnt, L::kListCap);
  }
  // query head and first query row of step t
  auto step_hq = [&](int t, int& h, int& q0) {
    int g, i;
    if (sparse) {
      const int c = step_list[t];
      g = c / p.n_q_tiles;
      i = c - g * p.n_q_tiles;
    } else {
      g = t % p.G;
      i = p.n_q_tiles - 1 - t / p.G;
    }
    h = kh * p.G + g;
    q0 = i * BR;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVFull), 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(bar(L::kQDFull + s), 1);
      mbar_init(bar(L::kQDEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kSFull + 1), 1);
    mbar_init(bar(L::kDPFull), 1);
    mbar_init(bar(L::kPFull), 128);
    mbar_init(bar(L::kDSFull), 128);
    mbar_init(bar(L::kDSEmpty), 1);
    mbar_init(bar(L::kDQFull), 1);
    mbar_init(bar(L::kDQEmpty), 128);
    mbar_init(bar(L::kFinal), 1);
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
  if (sparse) n_steps = *list_count;
  const uint32_t tmem = *tmem_holder;
  const uint32_t tdV = tmem + L::kTdV, tdK = tmem + L::kTdK, tS0 = tmem + L::kTS,
                 tdP = tmem + L::kTdP, tdQ = tmem + L::kTdQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; one elected lane issues the copies.
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(L::kKVFull), 2 * L::kKBytes);
      #pragma unroll
      for (int c = 0; c < L::kNch; ++c) {
        tma_load_4d(sbase + L::kKOff + c * (kBC * 128), &tm_k, bar(L::kKVFull), c * 64, kv0, kh, b);
        tma_load_4d(sbase + L::kVOff + c * (kBC * 128), &tm_v, bar(L::kKVFull), c * 64, kv0, kh, b);
      }
    }
    __syncwarp();
    int issued = 0;
    for (int t = 0; t < n_steps; ++t) {
      const int st = t % QST;
      if (t >= QST && !wait_uniform(bar(L::kQDEmpty + st), ((t / QST) + 1) & 1, abort)) break;
      int h, q0;
      step_hq(t, h, q0);
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kQDFull + st), 2 * L::kQBytes);
        #pragma unroll
        for (int c = 0; c < L::kNch; ++c) {
          tma_load_4d(sbase + L::kQOff + st * L::kQBytes + c * (BR * 128), &tm_q,
                      bar(L::kQDFull + st), c * 64, q0, h, b);
          tma_load_4d(sbase + L::kDOOff + st * L::kQBytes + c * (BR * 128), &tm_do,
                      bar(L::kQDFull + st), c * 64, q0, h, b);
        }
      }
      __syncwarp();
      ++issued;
    }
    drain_wait(bar(L::kKVFull), 0);
    for (int t = max(0, issued - QST); t < issued; ++t)
      drain_wait(bar(L::kQDFull + t % QST), (t / QST) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Warp-wide; each tcgen05 instruction is issued by one elected lane.
    // Descriptors are built once and advanced by constant offsets.
    {
      constexpr uint32_t kIdS = idesc_f16(kBC, BR, BF16 ? 1 : 0, 0, 0);
      constexpr uint32_t kIdKV = idesc_f16(kBC, DH, BF16 ? 1 : 0, 0, 1);
      constexpr uint32_t kIdQ = L::kDqT ? idesc_f16(DH, BR, BF16 ? 1 : 0, 1, 1)
                                        : idesc_f16(BR, D, BF16 ? 1 : 0, 1, 1);
      const uint32_t dh_chunk = static_cast<uint32_t>(dh * (DH / 64));
      // K-major views (LBO unused): K, V, Q stages, dO stages, dS^T.
      const uint64_t k_kmaj = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
      const uint64_t v_kmaj = smem_desc_sw128(sbase + L::kVOff, 16, 1024);
      const uint64_t q_kmaj = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t do_kmaj = smem_desc_sw128(sbase + L::kDOOff, 16, 1024);
      const uint64_t ds_kmaj = smem_desc_sw128(sbase + L::kDSOff, 16, 1024);
      // MN-major views: LBO = distance between 64-column chunks.
      const uint64_t q_mn = smem_desc_sw128(sbase + L::kQOff, BR * 128, 1024);
      const uint64_t do_mn = smem_desc_sw128(sbase + L::kDOOff, BR * 128, 1024);
      const uint64_t k_mn = smem_desc_sw128(sbase + L::kKOff, kBC * 128, 1024);
      const uint64_t ds_mn = smem_desc_sw128(sbase + L::kDSOff, kBC * 128, 1024);
      auto s_tmem = [&](int t) { return tS0 + (t % L::kSBuf) * BR; };
      // S^T_t = K Q_t^T (waits for the (Q_t, dO_t) tile).
      auto issue_s = [&](int t) -> bool {
        if (!wait_uniform(bar(L::kQDFull + t % QST), (t / QST) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t qs = (t % QST) * L::kQBytes;
        #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = kk >> 2, w = kk & 3;
          mma_ss(s_tmem(t), desc_add(k_kmaj, c * (kBC * 128) + w * 32),
                 desc_add(q_kmaj, qs + c * (BR * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kSFull + t % L::kSBuf));
        return true;
      };
      // dP^T_t = V dO_t^T (the tile is known to be loaded).
      auto issue_dp = [&](int t) {
        const uint32_t qs = (t % QST) * L::kQBytes;
        #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t c = kk >> 2, w = kk & 3;
          mma_ss(tdP, desc_add(v_kmaj, c * (kBC * 128) + w * 32),
                 desc_add(do_kmaj, qs + c * (BR * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kDPFull));
      };
      bool ok = wait_uniform(bar(L::kKVFull), 0, abort);
      if (ok && L::kSBuf == 2 && n_steps > 0) {
        ok = issue_s(0);
        if (ok) issue_dp(0);
      }
      for (int t = 0; ok && t < n_steps; ++t) {
        const int st = t % QST;
        const uint32_t qs = st * L::kQBytes;
        if constexpr (L::kSBuf == 2) {
          // The next scores go to the other buffer now, so the P / dS warps
          // can start on them while this step's products run.
          if (t + 1 < n_steps && !issue_s(t + 1)) break;
        } else {
          if (!issue_s(t)) break;
          issue_dp(t);
        }
        // dV += P^T dO (P^T from TMEM, dO MN-major)
        if (!wait_uniform(bar(L::kPFull), t & 1, abort)) break;
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tdV, s_tmem(t) + kk * 8, desc_add(do_mn, qs + dh_chunk * (BR * 128) + kk * 2048),
                 kIdKV, (t > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q (dS^T K-major in shared memory, Q MN-major)
        if (!wait_uniform(bar(L::kDSFull), t & 1, abort)) break;
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ss(tdK, desc_add(ds_kmaj, (kk >> 2) * (kBC * 128) + (kk & 3) * 32),
                 desc_add(q_mn, qs + dh_chunk * (BR * 128) + kk * 2048), kIdKV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        // dK was the last reader of Q_t and dO_t: the stage can be refilled.
        mma_commit(bar(L::kQDEmpty + st));
        // dQ contribution of this key tile
        if (p.with_dq) {
        if (t > 0 && !wait_uniform(bar(L::kDQEmpty), (t - 1) & 1, abort)) break;
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < kBC / 16; ++kk) {
          if constexpr (L::kDqT) {
            // dQ^T = K^T dS^T: A = K^T (d x keys, MN-major), B = dS^T (keys x q, MN-major)
            mma_ss(tdQ, desc_add(k_mn, dh_chunk * (kBC * 128) + kk * 2048),
                   desc_add(ds_mn, kk * 2048), kIdQ, kk > 0 ? 1u : 0u);
          } else {
            // dQ = dS K: A = dS (q x keys, MN-major), B = K (keys x d, MN-major)
            mma_ss(tdQ, desc_add(ds_mn, kk * 2048), desc_add(k_mn, kk * 2048), kIdQ,
                   kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(L::kDQFull));
        }
        mma_commit(bar(L::kDSEmpty));
        // The P / dS warps are done with dP^T_t (they signalled dS_t), so the
        // next dP^T can overwrite it.
        if constexpr (L::kSBuf == 2) {
          if (t + 1 < n_steps) issue_dp(t + 1);
        }
      }
      mma_commit(bar(L::kFinal));
      mma_commit(bar(L::kDrain));
      drain_wait(bar(L::kDrain), 0);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ P / dS warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;           // key row within the tile
    const int kv = kv0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // Each warp stages -L*log2(e) and -D of a query tile in its own
    // shared-memory slice (two buffers), loading the next tile's values into
    // registers while the current tile is processed; only __syncwarp is
    // needed.
    float* ld_base = reinterpret_cast<float*>(smem + L::kLDOff) + (warp - 2) * 2 * 2 * BR;
    constexpr int kPer = BR / 32;
    float rl[kPer], rd[kPer];
    auto load_ld = [&](int t) {
      int h, q0;
      step_hq(t, h, q0);
      const size_t base = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      #pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int q = q0 + lane + 32 * u;
        rl[u] = q < p.Nq ? -p.lse[base + q] * kLog2e : -INFINITY;
        if (p.direct) {
          // D = rowsum(dO o O) of query row q, in fp32
          float acc = 0.f;
          if (q < p.Nq) {
            const uint4* orow = reinterpret_cast<const uint4*>(p.o + b * p.os.b + h * p.os.h +
                                                               static_cast<long long>(q) * p.os.n);
            const uint4* drow = reinterpret_cast<const uint4*>(p.dout + b * p.dos.b + h * p.dos.h +
                                                               static_cast<long long>(q) * p.dos.n);
            #pragma unroll
            for (int c = 0; c < D / 8; ++c) {
              const uint4 x = orow[c], y = drow[c];
              const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
              #pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 a = unpack2<BF16>(xs[e]), g = unpack2<BF16>(ys[e]);
                acc = fmaf(a.x, g.x, acc);
                acc = fmaf(a.y, g.y, acc);
              }
            }
          }
          rd[u] = -acc;
        } else {
          rd[u] = q < p.Nq ? -p.delta[base + q] : 0.f;
        }
      }
    };
    auto store_ld = [&](int t) {
      float* dst = ld_base + (t & 1) * 2 * BR;
      #pragma unroll
      for (int u = 0; u < kPer; ++u) {
        dst[lane + 32 * u] = rl[u];
        dst[BR + lane + 32 * u] = rd[u];
      }
    };
    if (n_steps > 0) {
      load_ld(0);
      store_ld(0);
    }
    __syncwarp();
    bool ok = true;
    for (int t = 0; t < n_steps; ++t) {
      int h_t, q0;
      step_hq(t, h_t, q0);
      (void)h_t;
      const float* sL = ld_base + (t & 1) * 2 * BR;   // -L * log2(e)
      const float* sD = sL + BR;                       // -D
      if (t + 1 < n_steps) load_ld(t + 1);             // in flight during this step
      const uint32_t tS = tS0 + (t % L::kSBuf) * BR;
      // P^T = exp(S^T * scale - L), masked
      if (!wait_uniform(bar(L::kSFull + t % L::kSBuf), (t / L::kSBuf) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const bool kv_out = kv >= p.Nk;
      const bool diag = CAUSAL && (q0 + p.off < kv0 + kBC);   // tile crosses the diagonal
      const bool masked = __any_sync(0xffffffffu, kv_out || diag);
      const f2 cs = {p.scale_log2, p.scale_log2};
      // 128 query columns (d = 64): the weights stay in registers as the
      // 16-bit pairs written to TMEM (64 registers, not 128 in fp32, which
      // spilled), and dS uses those rounded weights, as dV does
      constexpr bool kPackP = BR > 64;
      float P[kPackP ? 1 : BR];
      uint32_t Pk[kPackP ? BR / 2 : 1];
      #pragma unroll
      for (int c0 = 0; c0 < BR; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(tS + lane_off + c0, sr);
        tmem_ld_wait();
        reg_fence(sr);
        float Pc[32];
        #pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const f2 arg = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs,
                               f2{sL[c0 + c], sL[c0 + c + 1]});
          Pc[c] = ex2_approx(arg.x);
          Pc[c + 1] = ex2_approx(arg.y);
        }
        if (masked) {
          #pragma unroll
          for (int c = 0; c < 32; ++c)
            if (kv_out || (diag && kv > q0 + c0 + c + p.off)) Pc[c] = 0.f;
        }
        uint32_t pk[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(Pc[2 * c], Pc[2 * c + 1]);
        #pragma unroll
        for (int c = 0; c < 32; ++c) {
          if constexpr (kPackP) {
            if ((c & 1) == 0) Pk[(c0 + c) / 2] = pk[c / 2];
          } else {
            P[c0 + c] = Pc[c];
          }
        }
        // P^T (16-bit) goes over the first BR/2 columns of the S^T tile,
        // which this thread has already read.
        tmem_st16(tS + lane_off + c0 / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::kPFull));
      // dS^T = P^T o (dP^T - D), written to shared memory as row r of the
      // dS^T tile with the 128-byte swizzle (16-byte unit u of a row lives
      // at unit u ^ (row % 8)).
      if (!wait_uniform(bar(L::kDPFull), t & 1, abort)) { ok = false; break; }
      if (t > 0 && !wait_uniform(bar(L::kDSEmpty), (t - 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      #pragma unroll
      for (int c0 = 0; c0 < BR; c0 += 32) {
        uint32_t dr[32];
        tmem_ld32(tdP + lane_off + c0, dr);
        tmem_ld_wait();
        reg_fence(dr);
        uint32_t w[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          const f2 diff = fadd2(f2{__uint_as_float(dr[2 * c]), __uint_as_float(dr[2 * c + 1])},
                                f2{sD[c0 + 2 * c], sD[c0 + 2 * c + 1]});
          f2 pv;
          if constexpr (kPackP) {
            const float2 u2 = unpack2<BF16>(Pk[c0 / 2 + c]);
            pv = f2{u2.x, u2.y};
          } else {
            pv = f2{P[c0 + 2 * c], P[c0 + 2 * c + 1]};
          }
          const f2 ds = fmul2(pv, diff);
          w[c] = pack2<BF16>(ds.x, ds.y);
        }
        #pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int u = c0 / 8 + u4, cb = u >> 3, uu = u & 7;
          uint4* dst = reinterpret_cast<uint4*>(smem + L::kDSOff + cb * (kBC * 128) + r * 128 +
                                                ((uu ^ (r & 7)) * 16));
          *dst = make_uint4(w[4 * u4], w[4 * u4 + 1], w[4 * u4 + 2], w[4 * u4 + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kDSFull));
      if (t + 1 < n_steps) {
        store_ld(t + 1);   // the other buffer: last read during step t - 1
        __syncwarp();
      }
    }
    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && wait_uniform(bar(L::kFinal), 0, abort)) {
      tc_fence_after();
      const bool in_range = kv < p.Nk;
      const long long kvr = in_range ? kv : 0;
      uint4* dv_row = reinterpret_cast<uint4*>(p.dv + b * p.dvs.b + kh * p.dvs.h + kvr * p.dvs.n +
                                               dh * DH);
      uint4* dk_row = reinterpret_cast<uint4*>(p.dk + b * p.dks.b + kh * p.dks.h + kvr * p.dks.n +
                                               dh * DH);
      // a key tile no step reached (block mask) has dK = dV = 0; its TMEM
      // accumulators were never written
      const uint32_t live = n_steps > 0 ? 0xffffffffu : 0u;
      #pragma unroll
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t a[32], k2[32];
        tmem_ld32(tdV + lane_off + c0, a);
        tmem_ld32(tdK + lane_off + c0, k2);
        tmem_ld_wait();
        reg_fence(a);
        reg_fence(k2);
        #pragma unroll
        for (int c = 0; c < 32; ++c) {
          a[c] &= live;
          k2[c] &= live;
        }
        uint32_t wv[16], wk[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          wv[c] = pack2<BF16>(__uint_as_float(a[2 * c]), __uint_as_float(a[2 * c + 1]));
          wk[c] = pack2<BF16>(__uint_as_float(k2[2 * c]) * p.scale,
                              __uint_as_float(k2[2 * c + 1]) * p.scale);
        }
        if (in_range) {
          #pragma unroll
          for (int i = 0; i < 4; ++i) {
            dv_row[c0 / 8 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
            dk_row[c0 / 8 + i] = make_uint4(wk[4 * i], wk[4 * i + 1], wk[4 * i + 2], wk[4 * i + 3]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    for (int t = 0; p.with_dq && t < n_steps; ++t) {
      int h, q0;
      step_hq(t, h, q0);
      if (!wait_uniform(bar(L::kDQFull), t & 1, abort)) break;
      tc_fence_after();
      constexpr int kCols = L::kDqCols;
      uint32_t v[kCols];
      #pragma unroll
      for (int c0 = 0; c0 < kCols; c0 += 32)
        tmem_ld32(tdQ + lane_off + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[c0]));
      tmem_ld_wait();
      reg_fence(v);
      tc_fence_before();
      mbar_arrive(bar(L::kDQEmpty));
      const size_t head_row = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      if constexpr (L::kDqT) {
        // lane r = column r of this CTA's half of d; v[c] = dQ[q0 + c][dh*DH + r].
        // Each group of four lanes transposes its 4 x 4 blocks (two butterfly
        // exchanges), so that lane 4i + j holds columns 4i .. 4i + 3 of query
        // row 4m + j, and adds them with one 16-byte red.global.add.v4.f32:
        // an SM sustains about twice the bytes of reductions that way as with
        // one 4-byte add per lane.
        const int i4 = lane >> 2, j4 = lane & 3;
        const bool hi2 = (j4 & 2) != 0, hi1 = (j4 & 1) != 0;
        float* base = p.dq_acc + (head_row + q0) * D + dh * DH + quarter * 32 + 4 * i4;
        const int n_valid = min(BR, p.Nq - q0);
        #pragma unroll
        for (int m = 0; m < BR / 4; ++m) {
          float x0 = __uint_as_float(v[4 * m]), x1 = __uint_as_float(v[4 * m + 1]);
          float x2 = __uint_as_float(v[4 * m + 2]), x3 = __uint_as_float(v[4 * m + 3]);
          // lanes j and j ^ 2 swap the halves of their rows the other needs
          const float s0 = __shfl_xor_sync(0xffffffffu, hi2 ? x0 : x2, 2);
          const float s1 = __shfl_xor_sync(0xffffffffu, hi2 ? x1 : x3, 2);
          if (hi2) { x0 = s0; x1 = s1; } else { x2 = s0; x3 = s1; }
          // lanes j and j ^ 1 swap single values
          const float u0 = __shfl_xor_sync(0xffffffffu, hi1 ? x0 : x1, 1);
          const float u1 = __shfl_xor_sync(0xffffffffu, hi1 ? x2 : x3, 1);
          if (hi1) { x0 = u0; x2 = u1; } else { x1 = u0; x3 = u1; }
          if (4 * m + j4 < n_valid)
            red_add_v4(base + static_cast<size_t>(4 * m + j4) * D, x0, x1, x2, x3);
        }
      } else {
        // lane r = query row q0 + r; v[c] = dQ[q0 + r][c]
        if (p.direct) {
          // the row's one contribution: scale * dQ in the output dtype
          if (q0 + r < p.Nq) {
            uint4* out = reinterpret_cast<uint4*>(p.dq + b * p.dqs.b + h * p.dqs.h +
                                                  static_cast<long long>(q0 + r) * p.dqs.n);
            #pragma unroll
            for (int c = 0; c < kCols / 8; ++c) {
              uint32_t w[4];
              #pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack2<BF16>(__uint_as_float(v[8 * c + 2 * e]) * p.scale,
                                   __uint_as_float(v[8 * c + 2 * e + 1]) * p.scale);
              out[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        } else if (q0 + r < p.Nq) {
          float4* base = reinterpret_cast<float4*>(p.dq_acc + (head_row + q0 + r) * D);
          #pragma unroll
          for (int c = 0; c < kCols / 4; ++c)
            atomicAdd(base + c, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                            __uint_as_float(v[4 * c + 2]),
                                            __uint_as_float(v[4 * c + 3])));
        }
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

// ---------------------------------------------------------------------------
// d = 128: 128 query rows per step.
//
// On sm_103a an M = 128 tcgen05.mma of kind::f16 occupies the tensor pipe
// for 64 cycles whenever N <= 128 (measured: N = 16, 64 and 128 all take 64
// cycles, N = 256 takes 126), so with 64-row steps the products S^T, dP^T and
// dQ^T (N = 64) run at half rate.  With 128-row steps every product has
// N = 128.  TMEM then holds dV (128 columns), dK (128), S^T (128, P^T written
// over it in 16 bits) and dP^T (128).
// Dense (dK and dV only; dQ comes from the query-outer kernel): the P / dS
// warps write dS^T in 16 bits over the dP^T columns they have read, dK reads
// it there (TS form), and the dS^T shared-memory tile becomes a third Q
// stage.  Issue order per step t:
//   dV(t), S(t+1), dK(t), dP(t+1)
// so the exponentials of step t+1 overlap dK(t) and dP(t+1).
// Block-sparse (dQ accumulated here): dS^T goes to shared memory, dQ^T of a
// step is written into the dP^T columns once the dS warps have read dP^T,
// and the next dP^T waits until the dQ warps have read dQ^T out:
//   dV(t), S(t+1), dQ^T(t), dK(t), dP(t+1)
// Warps: 0 TMA producer (K, V once; Q in three or two stages, dO in one),
// 1 MMA issuer, 2..9 P / dS (a key row per thread; warps w and w + 4 share a
// TMEM lane quarter and split the 128 query columns in halves; one arrival
// per warp on P_FULL and DS_FULL), 10..13 dQ (block-sparse only).

constexpr int kB128Threads = 448;

// DS_SMEM: dS^T is written to shared memory (the operand of the dQ^T
// product, which reads it as B); otherwise dS^T (16-bit) goes to TMEM over the
// dP^T columns it was formed from, where dK reads it as the A operand, and
// its shared-memory tile becomes a third Q stage.
template <bool DS_SMEM>
struct B128Layout {
  static constexpr int kTile = 128 * 128 * 2;      // one 128 x 128 16-bit tile
  static constexpr int kQStages = DS_SMEM ? 2 : 3;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTile;
  static constexpr int kQOff = 2 * kTile;          // kQStages stages
  static constexpr int kDOOff = (2 + kQStages) * kTile;   // one stage
  static constexpr int kDSOff = kDOOff + kTile;    // dS^T [keys][q] (DS_SMEM only)
  static constexpr int kLDOff = kDOOff + (DS_SMEM ? 2 : 1) * kTile;  // 8 warps x 2 bufs x {-L*log2e, -D} x 64
  static constexpr int kBarOff = kLDOff + 8 * 2 * 2 * 64 * 4;
  static constexpr int kKVFull = 0, kQFull = 1, kQEmpty = 4, kDOFull = 7, kDOEmpty = 8,
                       kSFull = 9, kDPFull = 10, kPFull = 11, kDSFull = 12, kDSEmpty = 13,
                       kDQFull = 14, kDQEmpty = 15, kFinal = 16, kDrain = 17, kNumBars = 18;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kListCap = 8192;            // (head, query tile) steps under a mask
  static constexpr int kListOff = kMiscOff + 16;
  static constexpr int kBytes = kListOff + kListCap * 2;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kAllocDense = kListOff + 1024;   // without the list
  static constexpr uint32_t kTdV = 0, kTdK = 128, kTS = 256, kTdP = 384, kTmemCols = 512;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

template <bool CAUSAL, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kB128Threads, 1)
bwd128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const BwdParams p) {
  // dense: no dQ product here (the query-outer kernel forms dQ), dS^T in TMEM
  constexpr bool kDsSmem = SPARSE;
  using L = B128Layout<kDsSmem>;
  constexpr int D = 128, BR = 128, QS = L::kQStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  int* list_count = reinterpret_cast<int*>(smem + L::kMiscOff + 8);
  uint16_t* step_list = reinterpret_cast<uint16_t*>(smem + L::kListOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // dispatch orders as in bwd_kernel (one CTA per key tile: no d split)
  int jt, kh, b;
  if (p.heavy_first) {
    jt = blockIdx.y;
    kh = blockIdx.x % p.Hkv;
    b = blockIdx.x / p.Hkv;
  } else {
    jt = blockIdx.x;
    kh = blockIdx.y;
    b = blockIdx.z;
  }
  const int kv0 = jt * kBC;
  const int i0 = CAUSAL ? max(0, kv0 - p.off) / BR : 0;
  const int n_i = p.n_q_tiles - i0;
  int n_steps = p.G * n_i;
  constexpr bool sparse = SPARSE;
  // step order as in bwd_kernel: query tiles descending, heads innermost
  if (sparse && warp == 2) {
    const int cnt = compact_steps<1>(
        p.G * n_i,
        [&](int e) {
          const int i = p.n_q_tiles - 1 - e / p.G, g = e % p.G;
          const int mh = p.mask.heads == 1 ? 0 : kh * p.G + g;
          return p.mask.ptr[(static_cast<size_t>(mh) * p.mask.nbr + i) * p.mask.nbc + jt] != 0;
        },
        [&](int e, int) {
          const int i = p.n_q_tiles - 1 - e / p.G, g = e % p.G;
          return g * p.n_q_tiles + i;
        },
        step_list, L::kListCap);
    if (lane == 0) *list_count = min(cnt, L::kListCap);
  }
  auto step_hq = [&](int t, int& h, int& q0) {
    int g, i;
    if (sparse) {
      const int c = step_list[t];
      g = c / p.n_q_tiles;
      i = c - g * p.n_q_tiles;
    } else {
      g = t % p.G;
      i = p.n_q_tiles - 1 - t / p.G;
    }
    h = kh * p.G + g;
    q0 = i * BR;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVFull), 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(bar(L::kQFull + s), 1);
      mbar_init(bar(L::kQEmpty + s), 1);
    }
    mbar_init(bar(L::kDOFull), 1);
    mbar_init(bar(L::kDOEmpty), 1);
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kDPFull), 1);
    mbar_init(bar(L::kPFull), 8);          // one arrival per P / dS warp
    mbar_init(bar(L::kDSFull), 8);
    mbar_init(bar(L::kDSEmpty), 1);
    mbar_init(bar(L::kDQFull), 1);
    mbar_init(bar(L::kDQEmpty), 128);
    mbar_init(bar(L::kFinal), 1);
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
  if (sparse) n_steps = *list_count;
  const uint32_t tmem = *tmem_holder;
  const uint32_t tdV = tmem + L::kTdV, tdK = tmem + L::kTdK, tS = tmem + L::kTS,
                 tdP = tmem + L::kTdP;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(L::kKVFull), 2 * L::kTile);
      #pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(sbase + L::kKOff + c * (kBC * 128), &tm_k, bar(L::kKVFull), c * 64, kv0, kh, b);
        tma_load_4d(sbase + L::kVOff + c * (kBC * 128), &tm_v, bar(L::kKVFull), c * 64, kv0, kh, b);
      }
    }
    __syncwarp();
    int q_issued = 0, do_issued = 0;
    for (int t = 0; t < n_steps; ++t) {
      const int s = t % QS;
      if (t >= QS && !wait_uniform(bar(L::kQEmpty + s), ((t / QS) + 1) & 1, abort)) break;
      int h, q0;
      step_hq(t, h, q0);
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kQFull + s), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kQOff + s * L::kTile + c * (BR * 128), &tm_q, bar(L::kQFull + s),
                      c * 64, q0, h, b);
      }
      __syncwarp();
      ++q_issued;
      if (t >= 1 && !wait_uniform(bar(L::kDOEmpty), (t - 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kDOFull), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kDOOff + c * (BR * 128), &tm_do, bar(L::kDOFull), c * 64, q0, h, b);
      }
      __syncwarp();
      ++do_issued;
    }
    drain_wait(bar(L::kKVFull), 0);
    for (int t = max(0, q_issued - QS); t < q_issued; ++t)
      drain_wait(bar(L::kQFull + t % QS), (t / QS) & 1);
    if (do_issued > 0) drain_wait(bar(L::kDOFull), (do_issued - 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(kBC, BR, BF16 ? 1 : 0, 0, 0);    // S^T, dP^T
    constexpr uint32_t kIdKV = idesc_f16(kBC, D, BF16 ? 1 : 0, 0, 1);    // dV, dK
    constexpr uint32_t kIdQ = idesc_f16(D, BR, BF16 ? 1 : 0, 1, 1);      // dQ^T
    const uint64_t k_kmaj = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_kmaj = smem_desc_sw128(sbase + L::kVOff, 16, 1024);
    const uint64_t q_kmaj = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t do_kmaj = smem_desc_sw128(sbase + L::kDOOff, 16, 1024);
    const uint64_t ds_kmaj = smem_desc_sw128(sbase + L::kDSOff, 16, 1024);
    const uint64_t q_mn = smem_desc_sw128(sbase + L::kQOff, BR * 128, 1024);
    const uint64_t do_mn = smem_desc_sw128(sbase + L::kDOOff, BR * 128, 1024);
    const uint64_t k_mn = smem_desc_sw128(sbase + L::kKOff, kBC * 128, 1024);
    const uint64_t ds_mn = smem_desc_sw128(sbase + L::kDSOff, kBC * 128, 1024);
    // S^T_t = K Q_t^T into the S columns
    auto issue_s = [&](int t) -> bool {
      if (!wait_uniform(bar(L::kQFull + t % QS), (t / QS) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t qs = (t % QS) * L::kTile;
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tS, desc_add(k_kmaj, c * (kBC * 128) + w * 32),
               desc_add(q_kmaj, qs + c * (BR * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull));
      return true;
    };
    // dP^T_t = V dO_t^T into the dP columns
    auto issue_dp = [&](int t) -> bool {
      if (!wait_uniform(bar(L::kDOFull), t & 1, abort)) return false;
      tc_fence_after();
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tdP, desc_add(v_kmaj, c * (kBC * 128) + w * 32),
               desc_add(do_kmaj, c * (BR * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kDPFull));
      return true;
    };
    bool ok = wait_uniform(bar(L::kKVFull), 0, abort);
    if (ok && n_steps > 0) ok = issue_s(0) && issue_dp(0);
    for (int t = 0; ok && t < n_steps; ++t) {
      const uint32_t qs = (t % QS) * L::kTile;
      // dV += P^T dO: P^T (16-bit) sits in the first 32 columns of each
      // 64-column half of the S columns (one half per P / dS warp).
      if (!wait_uniform(bar(L::kPFull), t & 1, abort)) break;
      tc_fence_after();
      #pragma unroll
      for (int kk = 0; kk < BR / 16; ++kk)
        mma_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(do_mn, kk * 2048), kIdKV,
               (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kDOEmpty));      // dP_t and dV_t were dO_t's readers
      if (t + 1 < n_steps && !issue_s(t + 1)) break;
      if (!wait_uniform(bar(L::kDSFull), t & 1, abort)) break;
      tc_fence_after();
      if constexpr (kDsSmem) {
        if (p.with_dq) {
          // dQ^T = K^T dS^T over the dP columns (their dP^T has been read)
          #pragma unroll
          for (int kk = 0; kk < kBC / 16; ++kk)
            mma_ss(tdP, desc_add(k_mn, kk * 2048), desc_add(ds_mn, kk * 2048), kIdQ,
                   kk > 0 ? 1u : 0u);
          mma_commit(bar(L::kDQFull));
        }
        // dK += dS^T Q
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ss(tdK, desc_add(ds_kmaj, (kk >> 2) * (kBC * 128) + (kk & 3) * 32),
                 desc_add(q_mn, qs + kk * 2048), kIdKV, (t > 0 || kk > 0) ? 1u : 0u);
      } else {
        // dK += dS^T Q, dS^T (16-bit) from TMEM: the first 32 columns of each
        // 64-column half of the dP columns, as P^T in the S columns
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tdK, tdP + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(q_mn, qs + kk * 2048), kIdKV,
                 (t > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar(L::kQEmpty + t % QS));
      if constexpr (kDsSmem) mma_commit(bar(L::kDSEmpty));
      if (t + 1 < n_steps) {
        if (kDsSmem && p.with_dq && !wait_uniform(bar(L::kDQEmpty), t & 1, abort)) break;
        // in TMEM mode dP^T(t + 1) overwrites dS^T(t) after dK(t) has read it
        // (products run in issue order)
        if (!issue_dp(t + 1)) break;
      }
    }
    mma_commit(bar(L::kFinal));
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else if (warp < 10) {
    // ------------------------------------------------------------ P / dS warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;            // query columns [64 half, 64 half + 64)
    const int r = quarter * 32 + lane;           // key row within the tile
    const int kv = kv0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float* ld_base = reinterpret_cast<float*>(smem + L::kLDOff) + (warp - 2) * 2 * 2 * 64;
    float rl[2], rd[2];
    auto load_ld = [&](int t) {
      int h, q0;
      step_hq(t, h, q0);
      const size_t base = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = q0 + 64 * half + lane + 32 * u;
        rl[u] = q < p.Nq ? -p.lse[base + q] * kLog2e : -INFINITY;
        rd[u] = q < p.Nq ? -p.delta[base + q] : 0.f;
      }
    };
    auto store_ld = [&](int t) {
      float* dst = ld_base + (t & 1) * 128;
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        dst[lane + 32 * u] = rl[u];
        dst[64 + lane + 32 * u] = rd[u];
      }
    };
    if (n_steps > 0) {
      load_ld(0);
      store_ld(0);
    }
    __syncwarp();
    bool ok = true;
    for (int t = 0; t < n_steps; ++t) {
      int h_t, q0;
      step_hq(t, h_t, q0);
      (void)h_t;
      const float* sL = ld_base + (t & 1) * 128;   // -L * log2(e) of this half's columns
      const float* sD = sL + 64;                     // -D
      if (t + 1 < n_steps) load_ld(t + 1);
      if (!wait_uniform(bar(L::kSFull), t & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const bool kv_out = kv >= p.Nk;
      const bool diag = CAUSAL && (q0 + p.off < kv0 + kBC);
      const bool masked = __any_sync(0xffffffffu, kv_out || diag);
      const f2 cs = {p.scale_log2, p.scale_log2};
      const int qc0 = q0 + 64 * half;              // first query of this half
      float P[64];
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(tS + lane_off + 64 * half + c0, sr);
        tmem_ld_wait();
        reg_fence(sr);
        // L and D come from shared memory as 16-byte broadcasts (a quarter
        // of the shared-memory wavefronts of scalar loads)
        #pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(sL + c0 + c);
          const f2 a0 = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs,
                              f2{l4.x, l4.y});
          const f2 a1 = ffma2(f2{__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])}, cs,
                              f2{l4.z, l4.w});
          P[c0 + c] = ex2_approx(a0.x);
          P[c0 + c + 1] = ex2_approx(a0.y);
          P[c0 + c + 2] = ex2_approx(a1.x);
          P[c0 + c + 3] = ex2_approx(a1.y);
        }
        if (masked) {
          // queries qc0 + c0 + c with c < z see no key kv (z = 32: the key is
          // past Nk); one comparison per score
          const int z = kv_out ? 32 : (diag ? min(32, kv - p.off - qc0 - c0) : 0);
          #pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < z) P[c0 + c] = 0.f;
        }
        uint32_t pk[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(P[c0 + 2 * c], P[c0 + 2 * c + 1]);
        // P^T over the first 32 columns of this half, already read
        tmem_st16(tS + lane_off + 64 * half + c0 / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bar(L::kPFull));
      // dS^T = P^T o (dP^T - D) into the swizzled dS^T tile (chunk = half)
      if (!wait_uniform(bar(L::kDPFull), t & 1, abort)) { ok = false; break; }
      if (kDsSmem && t > 0 && !wait_uniform(bar(L::kDSEmpty), (t - 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // 16 columns at a time: P (64 values) stays live across the loop
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t dr[16];
        tmem_ld16(tdP + lane_off + 64 * half + c0, dr);
        tmem_ld_wait();
        reg_fence(dr);
        uint32_t w[8];
        #pragma unroll
        for (int c = 0; c < 8; c += 2) {
          const float4 d4 = *reinterpret_cast<const float4*>(sD + c0 + 2 * c);
          const f2 diff0 = fadd2(f2{__uint_as_float(dr[2 * c]), __uint_as_float(dr[2 * c + 1])},
                                 f2{d4.x, d4.y});
          const f2 diff1 = fadd2(f2{__uint_as_float(dr[2 * c + 2]), __uint_as_float(dr[2 * c + 3])},
                                 f2{d4.z, d4.w});
          const f2 ds0 = fmul2(f2{P[c0 + 2 * c], P[c0 + 2 * c + 1]}, diff0);
          const f2 ds1 = fmul2(f2{P[c0 + 2 * c + 2], P[c0 + 2 * c + 3]}, diff1);
          w[c] = pack2<BF16>(ds0.x, ds0.y);
          w[c + 1] = pack2<BF16>(ds1.x, ds1.y);
        }
        if constexpr (kDsSmem) {
          #pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int u = c0 / 8 + u2;
            uint4* dst = reinterpret_cast<uint4*>(smem + L::kDSOff + half * (kBC * 128) +
                                                  r * 128 + ((u ^ (r & 7)) * 16));
            *dst = make_uint4(w[4 * u2], w[4 * u2 + 1], w[4 * u2 + 2], w[4 * u2 + 3]);
          }
        } else {
          // 16 dS^T values packed into 8 TMEM columns, stored over dP^T
          // columns [64 half + c0 / 2, + 8): already read (c0 / 2 + 8 <= c0 + 16)
          tmem_st8(tdP + lane_off + 64 * half + c0 / 2, w);
        }
      }
      if constexpr (kDsSmem) {
        tc_fence_before();
        fence_proxy_async_smem();
      } else {
        tmem_st_wait();
        tc_fence_before();
      }
      mbar_arrive_warp(bar(L::kDSFull));
      if (t + 1 < n_steps) {
        store_ld(t + 1);
        __syncwarp();
      }
    }
    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && wait_uniform(bar(L::kFinal), 0, abort)) {
      tc_fence_after();
      const bool in_range = kv < p.Nk;
      const long long kvr = in_range ? kv : 0;
      uint4* dv_row = reinterpret_cast<uint4*>(p.dv + b * p.dvs.b + kh * p.dvs.h + kvr * p.dvs.n +
                                               64 * half);
      uint4* dk_row = reinterpret_cast<uint4*>(p.dk + b * p.dks.b + kh * p.dks.h + kvr * p.dks.n +
                                               64 * half);
      const uint32_t live = n_steps > 0 ? 0xffffffffu : 0u;
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t a[32], k2[32];
        tmem_ld32(tdV + lane_off + 64 * half + c0, a);
        tmem_ld32(tdK + lane_off + 64 * half + c0, k2);
        tmem_ld_wait();
        reg_fence(a);
        reg_fence(k2);
        uint32_t wv[16], wk[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          wv[c] = pack2<BF16>(__uint_as_float(a[2 * c] & live), __uint_as_float(a[2 * c + 1] & live));
          wk[c] = pack2<BF16>(__uint_as_float(k2[2 * c] & live) * p.scale,
                              __uint_as_float(k2[2 * c + 1] & live) * p.scale);
        }
        if (in_range) {
          #pragma unroll
          for (int i = 0; i < 4; ++i) {
            dv_row[c0 / 8 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
            dk_row[c0 / 8 + i] = make_uint4(wk[4 * i], wk[4 * i + 1], wk[4 * i + 2], wk[4 * i + 3]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    // lane r = column r of d; dQ^T row r holds dQ[q0 + c][r] for the 128 c
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    for (int t = 0; p.with_dq && t < n_steps; ++t) {
      int h, q0;
      step_hq(t, h, q0);
      if (!wait_uniform(bar(L::kDQFull), t & 1, abort)) break;
      tc_fence_after();
      float* base = p.dq_acc + ((static_cast<size_t>(b) * p.H + h) * p.Nq + q0) * D + r;
      const int n_valid = min(BR, p.Nq - q0);
      // two halves of 64 columns (128 values would not fit the register
      // budget); DQEmpty once both are in registers
      #pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t v[64];
        tmem_ld32(tdP + lane_off + 64 * part, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tdP + lane_off + 64 * part + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        reg_fence(v);
        if (part == 1) {
          tc_fence_before();
          mbar_arrive(bar(L::kDQEmpty));
        }
        #pragma unroll
        for (int c = 0; c < 64; ++c)
          if (64 * part + c < n_valid)
            atomicAdd(base + static_cast<size_t>(64 * part + c) * D, __uint_as_float(v[c]));
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

// Element offset of row (b * H + h) * N + i of a strided [B][H][N][d] view.
__device__ __forceinline__ long long view_offset(size_t row, int H, int N, const Strides& s) {
  const size_t bh = row / N;
  const long long i = static_cast<long long>(row - bh * N);
  return static_cast<long long>(bh / H) * s.b + static_cast<long long>(bh % H) * s.h + i * s.n;
}

// D_i = dO_i . O_i (fp32) and a zeroed dQ accumulator row (delta and the
// accumulator are contiguous; o and dout strided), and the persistent
// kernel's work counter set to zero when one is given.  HBM-bound: D / 8 lanes
// per row read 16 bytes of each tensor, a warp covers 256 / D rows per pass
// and makes kPasses passes with every load issued before the first sum, so
// that enough bytes are in flight to keep HBM busy.
constexpr int kPrePasses = 4;
constexpr int kPreWarps = 8;
template <int D>
__host__ __device__ constexpr int pre_rows_per_block() { return kPreWarps * (256 / D) * kPrePasses; }

template <int D, bool BF16>
__global__ void __launch_bounds__(kPreWarps * 32)
bwd_preprocess(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
               float* __restrict__ delta, float* __restrict__ dq_acc, size_t rows, int H, int N,
               Strides os, Strides dos, unsigned int* __restrict__ units) {
  constexpr int kLanes = D / 8;                  // lanes per row
  constexpr int kRowsPerPass = 32 / kLanes;      // rows of one warp per pass
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / kLanes, col = (lane % kLanes) * 8;
  if (units != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *units = 0u;   // work counter
  const size_t row0 = static_cast<size_t>(blockIdx.x) * pre_rows_per_block<D>() +
                      static_cast<size_t>(warp) * kRowsPerPass * kPrePasses + sub;
  uint4 ov[kPrePasses], dv[kPrePasses];
  #pragma unroll
  for (int u = 0; u < kPrePasses; ++u) {
    const size_t row = row0 + static_cast<size_t>(u) * kRowsPerPass;
    ov[u] = dv[u] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      ov[u] = *reinterpret_cast<const uint4*>(o + view_offset(row, H, N, os) + col);
      dv[u] = *reinterpret_cast<const uint4*>(dout + view_offset(row, H, N, dos) + col);
    }
  }
  #pragma unroll
  for (int u = 0; u < kPrePasses; ++u) {
    const size_t row = row0 + static_cast<size_t>(u) * kRowsPerPass;
    float acc = 0.f;
    const uint32_t ow[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
    const uint32_t dw[4] = {dv[u].x, dv[u].y, dv[u].z, dv[u].w};
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = unpack2<BF16>(ow[i]), c = unpack2<BF16>(dw[i]);
      acc = fmaf(a.x, c.x, acc);
      acc = fmaf(a.y, c.y, acc);
    }
    #pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows) {
      if (lane % kLanes == 0) delta[row] = acc;
      if (dq_acc != nullptr) {
        float4* arow = reinterpret_cast<float4*>(dq_acc + row * D + col);
        arow[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        arow[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// dq = scale * dq_acc (contiguous), converted to the output dtype and
// written to the strided dq view; 8 elements per thread.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
bwd_convert_dq(const float* __restrict__ acc, uint16_t* __restrict__ dq, size_t n8, float scale,
               int H, int N, Strides dqs) {
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 c = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    const size_t row = i / (D / 8);
    const int col = static_cast<int>(i - row * (D / 8)) * 8;
    *reinterpret_cast<uint4*>(dq + view_offset(row, H, N, dqs) + col) =
        make_uint4(pack2<BF16>(a.x * scale, a.y * scale), pack2<BF16>(a.z * scale, a.w * scale),
                   pack2<BF16>(c.x * scale, c.y * scale), pack2<BF16>(c.z * scale, c.w * scale));
  }
}

int g_num_sms = 0;

// WIDE: the d = 128 kernel with 128-row steps (bwd128_kernel).
template <int D, int DH, int BR, int QST, bool CAUSAL, bool BF16, bool SPARSE, bool WIDE = false>
cudaError_t launch_variant(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  using L = std::conditional_t<WIDE, B128Layout<SPARSE>, BwdLayout<D, DH, BR, QST>>;
  static_assert(!WIDE || (D == 128 && DH == 128 && BR == 128), "wide kernel shape");
  cudaError_t e;
  const size_t rows = static_cast<size_t>(pr.B) * pr.H * pr.Nq;
  // One key tile (d = 64): the main kernel forms D and writes dQ itself, when
  // every query tile has a step (under the mask the first tile's rows see no
  // key once Nq - Nk >= 128, and no step would write their dQ = 0)
  const bool direct = D == 64 && !WIDE && !SPARSE && pr.Nk <= kBC &&
                      (!CAUSAL || pr.Nq - pr.Nk < BR);
  // 1. preprocess
  int slot = -1;
  if (!direct) {
    slot = timing_begin(FA_KERNEL_BWD_PRE, stream);
    constexpr int kPreRows = pre_rows_per_block<D>();
    bwd_preprocess<D, BF16><<<static_cast<unsigned>((rows + kPreRows - 1) / kPreRows),
                              kPreWarps * 32, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.delta,
        a.deterministic ? nullptr : a.dq_acc, rows, pr.H, pr.Nq, a.os, a.dos, nullptr);
    timing_end(slot, stream);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 2. main kernel
  CUtensorMap tq, tk, tv, tdo;
  if ((e = make_tmap_4d(&tq, a.q, D, pr.Nq, pr.H, pr.B, a.qs, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, D, pr.Nq, pr.H, pr.B, a.dos, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tk, a.k, D, pr.Nk, pr.Hkv, pr.B, a.ks, 64, kBC)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, D, pr.Nk, pr.Hkv, pr.B, a.vs, 64, kBC)) != cudaSuccess) return e;
  auto kern = [] {
    if constexpr (WIDE)
      return bwd128_kernel<CAUSAL, BF16, SPARSE>;
    else
      return bwd_kernel<D, DH, BR, QST, CAUSAL, BF16, SPARSE>;
  }();
  constexpr int kThreadsMain = WIDE ? kB128Threads : kBwdThreads;
  constexpr int kSmem = SPARSE ? L::kAlloc : L::kAllocDense;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
        cudaSuccess)
      return e;
    attr_set = true;
  }
  BwdParams p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq_acc = a.dq_acc;
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.G = pr.H / pr.Hkv;
  p.n_q_tiles = (pr.Nq + BR - 1) / BR;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kLog2e;
  p.err = pr.err;
  p.with_dq = (a.deterministic && !direct) ? 0 : 1;
  p.direct = direct ? 1 : 0;
  p.o = static_cast<const uint16_t*>(a.o);
  p.dout = static_cast<const uint16_t*>(a.dout);
  p.dq = static_cast<uint16_t*>(a.dq);
  p.os = a.os;
  p.dos = a.dos;
  p.dqs = a.dqs;
  // the dense 128-row kernel forms dK and dV only (dS^T lives in TMEM)
  if (WIDE && !SPARSE && p.with_dq) return cudaErrorInvalidValue;
  p.mask = a.mask;
  p.dks = a.dks;
  p.dvs = a.dvs;
  const int n_kv_tiles = (pr.Nk + kBC - 1) / kBC;
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  // Heavy-first order when the longest CTA holds more than a fifth of one
  // SM's share of the work (long causal rows); otherwise L2 locality wins.
  p.heavy_first = 0;
  if (CAUSAL && !SPARSE && n_kv_tiles <= 65535) {
    double total = 0.0;
    for (int j = 0; j < n_kv_tiles; ++j) total += p.n_q_tiles - std::max(0, j * kBC - p.off) / BR;
    total *= static_cast<double>(p.G) * (D / DH) * pr.Hkv * pr.B;
    const double longest = static_cast<double>(p.G) * p.n_q_tiles;
    p.heavy_first = longest > 0.2 * total / g_num_sms ? 1 : 0;
  }
  dim3 grid = p.heavy_first ? dim3((D / DH) * pr.Hkv * pr.B, n_kv_tiles, 1)
                            : dim3(n_kv_tiles * (D / DH), pr.Hkv, pr.B);
  slot = timing_begin(FA_KERNEL_BWD_MAIN, stream);
  kern<<<grid, kThreadsMain, kSmem, stream>>>(tq, tk, tv, tdo, p);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 3. dQ: written by the main kernel (one key tile), the query-outer kernel
  // (deterministic) or the accumulator's conversion
  if (direct) return cudaSuccess;
  if (a.deterministic) return launch_bwd_dq(pr, a, stream);
  const size_t n8 = rows * D / 8;
  const unsigned blocks = static_cast<unsigned>(
      std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(g_num_sms) * 8));
  slot = timing_begin(FA_KERNEL_BWD_CONVERT, stream);
  bwd_convert_dq<D, BF16><<<blocks, 256, 0, stream>>>(a.dq_acc, static_cast<uint16_t*>(a.dq), n8,
                                                      pr.scale, pr.H, pr.Nq, a.dqs);
  timing_end(slot, stream);
  return cudaGetLastError();
}

template <int D, int DH, int BR, int QST, bool SPARSE, bool WIDE = false>
cudaError_t dispatch_flags(const Problem& pr, const BwdArgs& a, cudaStream_t s) {
  if (pr.causal)
    return pr.bf16 ? launch_variant<D, DH, BR, QST, true, true, SPARSE, WIDE>(pr, a, s)
                   : launch_variant<D, DH, BR, QST, true, false, SPARSE, WIDE>(pr, a, s);
  return pr.bf16 ? launch_variant<D, DH, BR, QST, false, true, SPARSE, WIDE>(pr, a, s)
                 : launch_variant<D, DH, BR, QST, false, false, SPARSE, WIDE>(pr, a, s);
}

// Tile configuration per head dimension: output half DH, query rows per step
// BR, Q / dO ring stages.
// d = 128 runs bwd128_kernel (128 query rows per step, two Q stages).
using Cfg64 = BwdLayout<64, 64, 128, 3>;
using Cfg128 = B128Layout<true>;
using Cfg256 = BwdLayout<256, 128, 64, 1>;

template <bool SPARSE>
cudaError_t launch_bwd_for(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  switch (pr.d) {
    case 64: return dispatch_flags<64, 64, 128, 3, SPARSE>(pr, a, stream);
    case 128: return dispatch_flags<128, 128, 128, 2, SPARSE, true>(pr, a, stream);
    case 256: return dispatch_flags<256, 128, 64, 1, SPARSE>(pr, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace fa
