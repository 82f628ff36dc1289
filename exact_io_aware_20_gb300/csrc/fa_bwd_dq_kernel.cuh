// Deterministic dQ kernel of the backward pass (instantiated dense in
// fa_bwd_dq.cu and block-sparse in fa_bwd_dq_blocksparse.cu):
// dQ = scale * sum_j dS_j K_j with
// no atomics.  One CTA owns a 128-row query tile of one head and loops over
// the key tiles in a fixed order, accumulating in TMEM, so the result is the
// same bits on every run.
//
// It recomputes S = Q K^T and dP = dO V^T per key tile (the main backward
// kernel, run in its dK/dV-only mode, computes them too): two extra products
// per tile buy run-to-run reproducibility of dQ.  The pages note that dQ is
// accumulated across key/value blocks with atomic adds and do not discuss
// the resulting non-determinism ("FlashAttention-2: Faster Attention with
// Better Parallelism and Work Partitioning", paper digest, section 7); this
// kernel is the reproducible alternative.
//
// Per key tile j (64 keys): S_j = Q K_j^T and dP_j = dO V_j^T into one of
// two TMEM buffer pairs (M = 128 query rows, N = 64); warps 2..5 (one query
// row per thread) form P = exp(S * scale - L), dS = P o (dP - D) and write
// dS (16-bit) over the S buffer; dQ += dS K_j reads dS from TMEM (A operand)
// and K_j from shared memory (MN-major).  The next tile's S and dP are issued
// before the current dQ product, so the exponentials overlap the tensor work.
//
// Under a block mask (block-sparse attention, "FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", abstract) the CTA
// walks only the key tiles of the kept blocks in its query tile's mask row.
#pragma once

#include "block_list.cuh"
#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

namespace {

constexpr int kDqBR = 128;           // query rows per CTA (MMA M)
constexpr int kDqBC = kDqKeyTile;    // keys per tile (64)
constexpr int kDqThreads = 192;
constexpr float kDqLog2e = 1.4426950408889634f;

template <int D, int KST>
struct DqLayout {
  static constexpr int kNch = D / 64;
  static constexpr int kQBytes = kDqBR * D * 2;
  static constexpr int kKVBytes = kDqBC * D * 2;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kQBytes;
  static constexpr int kKOff = 2 * kQBytes;
  static constexpr int kVOff = kKOff + KST * kKVBytes;
  static constexpr int kBarOff = kVOff + KST * kKVBytes;
  static constexpr int kQDFull = 0;
  static constexpr int kKFull = 1;
  static constexpr int kKEmpty = kKFull + KST;
  static constexpr int kVFull = kKEmpty + KST;
  static constexpr int kVEmpty = kVFull + KST;
  static constexpr int kSFull = kVEmpty + KST;   // 2: S and dP of a tile done
  static constexpr int kDSFull = kSFull + 2;     // 2: dS of a tile in TMEM
  static constexpr int kDQDone = kDSFull + 2;
  static constexpr int kDrain = kDQDone + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kListOff = kMiscOff + 16;   // key tiles kept under a block mask
  static constexpr int kBytes = kListOff + kDqListCap * 2;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kAllocDense = kListOff + 1024;   // without the list
  static constexpr uint32_t kTS = 0, kTdP = 2 * kDqBC, kTdQ = 4 * kDqBC, kTmemCols = 512;
  static_assert(kTdQ + D <= kTmemCols, "TMEM budget");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

struct DqParams {
  const float* lse;
  const float* delta;
  uint16_t* dq;
  int H, Hkv, G;
  int Nq, Nk, off;    // query / key lengths; off = Nk - Nq (bottom-right mask)
  int num_q_tiles;
  float scale, scale_log2;
  BlockMask mask;
  Strides dqs;        // element strides of dq
  unsigned int* err;
};

template <int D, int KST, bool CAUSAL, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kDqThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const DqParams p) {
  using L = DqLayout<D, KST>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  int* list_count = reinterpret_cast<int*>(smem + L::kMiscOff + 8);
  uint16_t* tile_list = reinterpret_cast<uint16_t*>(smem + L::kListOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = CAUSAL ? (p.num_q_tiles - 1 - static_cast<int>(blockIdx.x))
                        : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int kh = h / p.G;
  int n_kv = (p.Nk + kDqBC - 1) / kDqBC;
  if (CAUSAL) {
    const int last_key = min((qt + 1) * kDqBR, p.Nq) - 1 + p.off;
    n_kv = last_key < 0 ? 0 : min(n_kv, last_key / kDqBC + 1);
  }
  constexpr bool sparse = SPARSE;
  if (sparse && warp == 2) {
    constexpr int kSub = kMaskBlock / kDqBC;
    const int mh = p.mask.heads == 1 ? 0 : h;
    const unsigned char* mrow =
        p.mask.ptr + (static_cast<size_t>(mh) * p.mask.nbr + qt) * p.mask.nbc;
    const int lim = n_kv;
    const int cnt = compact_steps<kSub>(
        p.mask.nbc, [&](int e) { return mrow[e] != 0; },
        [&](int e, int sub) { const int j = e * kSub + sub; return j < lim ? j : -1; },
        tile_list, kDqListCap);
    if (lane == 0) *list_count = min(cnt, kDqListCap);
  }
  auto key_tile = [&](int j) -> int { return sparse ? static_cast<int>(tile_list[j]) : j; };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQDFull), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kDSFull + s), 128);
    }
    mbar_init(bar(L::kDQDone), 1);
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
  if (sparse) n_kv = *list_count;
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem + L::kTS, tdP = tmem + L::kTdP, tdQ = tmem + L::kTdQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(L::kQDFull), 2 * L::kQBytes);
      #pragma unroll
      for (int c = 0; c < L::kNch; ++c) {
        tma_load_4d(sbase + L::kQOff + c * (kDqBR * 128), &tm_q, bar(L::kQDFull), c * 64,
                    qt * kDqBR, h, b);
        tma_load_4d(sbase + L::kDOOff + c * (kDqBR * 128), &tm_do, bar(L::kQDFull), c * 64,
                    qt * kDqBR, h, b);
      }
    }
    __syncwarp();
    int k_issued = 0, v_issued = 0;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j % KST;
      if (j >= KST && !wait_uniform(bar(L::kKEmpty + s), ((j / KST) + 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kKFull + s), L::kKVBytes);
        #pragma unroll
        for (int c = 0; c < L::kNch; ++c)
          tma_load_4d(sbase + L::kKOff + s * L::kKVBytes + c * (kDqBC * 128), &tm_k,
                      bar(L::kKFull + s), c * 64, key_tile(j) * kDqBC, kh, b);
      }
      __syncwarp();
      ++k_issued;
      if (j >= KST && !wait_uniform(bar(L::kVEmpty + s), ((j / KST) + 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kVFull + s), L::kKVBytes);
        #pragma unroll
        for (int c = 0; c < L::kNch; ++c)
          tma_load_4d(sbase + L::kVOff + s * L::kKVBytes + c * (kDqBC * 128), &tm_v,
                      bar(L::kVFull + s), c * 64, key_tile(j) * kDqBC, kh, b);
      }
      __syncwarp();
      ++v_issued;
    }
    drain_wait(bar(L::kQDFull), 0);
    for (int j = max(0, k_issued - KST); j < k_issued; ++j)
      drain_wait(bar(L::kKFull + j % KST), (j / KST) & 1);
    for (int j = max(0, v_issued - KST); j < v_issued; ++j)
      drain_wait(bar(L::kVFull + j % KST), (j / KST) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(kDqBR, kDqBC, BF16 ? 1 : 0, 0, 0);
    constexpr uint32_t kIdQ = idesc_f16(kDqBR, D, BF16 ? 1 : 0, 0, 1);
    const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t do_desc = smem_desc_sw128(sbase + L::kDOOff, 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sbase + L::kVOff, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(sbase + L::kKOff, kDqBC * 128, 1024);
    // S_j = Q K_j^T and dP_j = dO V_j^T into buffer pair j & 1.
    auto issue_sdp = [&](int j) -> bool {
      const int s = j % KST;
      if (!wait_uniform(bar(L::kKFull + s), (j / KST) & 1, abort)) return false;
      if (!wait_uniform(bar(L::kVFull + s), (j / KST) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t buf = (j & 1) * kDqBC;
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tS + buf, desc_add(q_desc, c * (kDqBR * 128) + w * 32),
               desc_add(k_desc, s * L::kKVBytes + c * (kDqBC * 128) + w * 32), kIdS,
               kk > 0 ? 1u : 0u);
      }
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tdP + buf, desc_add(do_desc, c * (kDqBR * 128) + w * 32),
               desc_add(v_desc, s * L::kKVBytes + c * (kDqBC * 128) + w * 32), kIdS,
               kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull + (j & 1)));
      mma_commit(bar(L::kVEmpty + s));   // V_j is not read again
      return true;
    };
    bool ok = wait_uniform(bar(L::kQDFull), 0, abort);
    // With two or more K stages the next tile's S and dP go to the other
    // buffer pair before this tile's dQ product.  With one stage K_{j+1}
    // can only arrive after dQ_j (K_j's last reader) has run, so the tiles
    // are processed one after the other.
    if (ok && KST >= 2 && n_kv > 0) ok = issue_sdp(0);
    for (int j = 0; ok && j < n_kv; ++j) {
      if constexpr (KST >= 2) {
        if (j + 1 < n_kv && !issue_sdp(j + 1)) break;
      } else {
        if (!issue_sdp(j)) break;
      }
      if (!wait_uniform(bar(L::kDSFull + (j & 1)), (j >> 1) & 1, abort)) break;
      tc_fence_after();
      const int s = j % KST;
      const uint32_t a_tmem = tS + (j & 1) * kDqBC;
      #pragma unroll
      for (int kk = 0; kk < kDqBC / 16; ++kk)
        mma_ts(tdQ, a_tmem + kk * 8, desc_add(k_mn, s * L::kKVBytes + kk * 2048), kIdQ,
               (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kKEmpty + s));   // K_j's last reader
    }
    mma_commit(bar(L::kDQDone));
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ dS warps
    const int quarter = warp & 3;
    const int row = qt * kDqBR + quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const size_t row_idx = (static_cast<size_t>(b) * p.H + h) * p.Nq + (row < p.Nq ? row : 0);
    const long long dq_off =
        b * p.dqs.b + h * p.dqs.h + static_cast<long long>(row < p.Nq ? row : 0) * p.dqs.n;
    // -L*log2(e) and -D of this thread's row (padding rows: P = 0)
    const float nL = row < p.Nq ? -p.lse[row_idx] * kDqLog2e : -INFINITY;
    const float nD = row < p.Nq ? -p.delta[row_idx] : 0.f;
    const f2 cs = {p.scale_log2, p.scale_log2}, cl = {nL, nL}, cd = {nD, nD};
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!wait_uniform(bar(L::kSFull + (j & 1)), (j >> 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t buf = (j & 1) * kDqBC;
      uint32_t sr[kDqBC], dr[kDqBC];
      #pragma unroll
      for (int c = 0; c < kDqBC / 32; ++c) {
        tmem_ld32(tS + buf + lane_off + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_ld32(tdP + buf + lane_off + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&dr[32 * c]));
      }
      tmem_ld_wait();
      reg_fence(sr);
      reg_fence(dr);
      const int col0 = key_tile(j) * kDqBC;
      const bool masked =
          (CAUSAL && col0 + kDqBC - 1 > qt * kDqBR + p.off) || (col0 + kDqBC > p.Nk);
      uint32_t w[kDqBC / 2];
      #pragma unroll
      for (int c = 0; c < kDqBC; c += 2) {
        const f2 arg = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs, cl);
        f2 pe = {ex2_approx(arg.x), ex2_approx(arg.y)};
        if (masked) {
          if (col0 + c >= p.Nk || (CAUSAL && col0 + c > row + p.off)) pe.x = 0.f;
          if (col0 + c + 1 >= p.Nk || (CAUSAL && col0 + c + 1 > row + p.off)) pe.y = 0.f;
        }
        const f2 ds = fmul2(pe, fadd2(f2{__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])}, cd));
        w[c / 2] = pack2<BF16>(ds.x, ds.y);
      }
      // dS (16-bit) over the first 32 columns of the S buffer, already read
      tmem_st32(tS + buf + lane_off, w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::kDSFull + (j & 1)));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && n_kv == 0) {
      // no row of this tile sees any key: dQ = 0
      if (row < p.Nq) {
        uint4* out = reinterpret_cast<uint4*>(p.dq + dq_off);
        #pragma unroll
        for (int i = 0; i < D / 8; ++i) out[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else if (ok && wait_uniform(bar(L::kDQDone), 0, abort)) {
      tc_fence_after();
      uint4* out = reinterpret_cast<uint4*>(p.dq + dq_off);
      #pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tdQ + lane_off + c0, v);
        tmem_ld_wait();
        reg_fence(v);
        uint32_t o[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * p.scale,
                             __uint_as_float(v[2 * i + 1]) * p.scale);
        if (row < p.Nq) {
          #pragma unroll
          for (int i = 0; i < 4; ++i)
            out[c0 / 8 + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
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

template <int D, int KST, bool CAUSAL, bool BF16, bool SPARSE>
cudaError_t launch_dq_variant(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  using L = DqLayout<D, KST>;
  CUtensorMap tq, tk, tv, tdo;
  cudaError_t e;
  if ((e = make_tmap_4d(&tq, a.q, D, pr.Nq, pr.H, pr.B, a.qs, 64, kDqBR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, D, pr.Nq, pr.H, pr.B, a.dos, 64, kDqBR)) != cudaSuccess)
    return e;
  if ((e = make_tmap_4d(&tk, a.k, D, pr.Nk, pr.Hkv, pr.B, a.ks, 64, kDqBC)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, D, pr.Nk, pr.Hkv, pr.B, a.vs, 64, kDqBC)) != cudaSuccess) return e;
  auto kern = bwd_dq_kernel<D, KST, CAUSAL, BF16, SPARSE>;
  constexpr int kSmem = SPARSE ? L::kAlloc : L::kAllocDense;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
        cudaSuccess)
      return e;
    attr_set = true;
  }
  DqParams p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<uint16_t*>(a.dq);
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.G = pr.H / pr.Hkv;
  p.num_q_tiles = (pr.Nq + kDqBR - 1) / kDqBR;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kDqLog2e;
  p.mask = a.mask;
  p.dqs = a.dqs;
  p.err = pr.err;
  dim3 grid(p.num_q_tiles, pr.H, pr.B);
  const int slot = timing_begin(FA_KERNEL_BWD_DQ, stream);
  kern<<<grid, kDqThreads, kSmem, stream>>>(tq, tk, tv, tdo, p);
  timing_end(slot, stream);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// d = 128: 128-key tiles, so every product is an N = 128 tcgen05.mma (full
// rate; with 64-key tiles S and dP ran at half rate).
// TMEM: S (two buffers, 128 columns each; dS written over S in 16 bits),
// dP (128), dQ (128).  Warps: 0 TMA producer (Q, dO once; K, V rings),
// 1 MMA issuer, 2..9 dS warps (a query row per thread; warps w and w + 4
// share a TMEM lane quarter and split the 128 key columns in halves).
// Issue order per key tile j: S(j+1), [dP(j) read: DP_READ] dP(j+1),
// [dS(j) written: DS_FULL, two barriers alternating] dQ += dS(j) K_j.
// dS stays in TMEM and is the A operand of the dQ product (TS form).
constexpr int kDq128Threads = 320;

// KST: K stages.  K_j is read until dQ_j, the last product of the tile, so
// with two stages the load of K_{j+2} would start only when dQ_j is done;
// the dense kernel has room for a third.
template <int KST>
struct Dq128Layout {
  static constexpr int kTile = 128 * 128 * 2;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTile;
  static constexpr int kKOff = 2 * kTile;             // KST stages
  static constexpr int kVOff = (2 + KST) * kTile;     // two stages
  static constexpr int kBarOff = (4 + KST) * kTile;
  static constexpr int kQDFull = 0, kKFull = 1, kKEmpty = kKFull + KST, kVFull = kKEmpty + KST,
                       kVEmpty = kVFull + 2, kSFull = kVEmpty + 2, kDPFull = kSFull + 2,
                       kDSFull = kDPFull + 1, kDPRead = kDSFull + 2, kDQDone = kDPRead + 1,
                       kDrain = kDQDone + 1, kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kListOff = kMiscOff + 16;
  static constexpr int kBytes = kListOff + kDqListCap * 2;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr int kAllocDense = kListOff + 1024;
  static constexpr uint32_t kTS = 0, kTdP = 256, kTdQ = 384, kTmemCols = 512;
  static_assert(kAllocDense <= 227 * 1024, "shared memory budget");
};

template <bool CAUSAL, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kDq128Threads, 1)
bwd_dq128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const DqParams p) {
  constexpr int KST = SPARSE ? 2 : 3;
  using L = Dq128Layout<KST>;
  static_assert(!SPARSE || L::kAlloc <= 227 * 1024, "shared memory budget");
  constexpr int D = 128, BR = 128, BC = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  int* list_count = reinterpret_cast<int*>(smem + L::kMiscOff + 8);
  uint16_t* tile_list = reinterpret_cast<uint16_t*>(smem + L::kListOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = CAUSAL ? (p.num_q_tiles - 1 - static_cast<int>(blockIdx.x))
                        : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int kh = h / p.G;
  int n_kv = (p.Nk + BC - 1) / BC;
  if (CAUSAL) {
    const int last_key = min((qt + 1) * BR, p.Nq) - 1 + p.off;
    n_kv = last_key < 0 ? 0 : min(n_kv, last_key / BC + 1);
  }
  constexpr bool sparse = SPARSE;
  if (sparse && warp == 2) {
    const int mh = p.mask.heads == 1 ? 0 : h;
    const unsigned char* mrow =
        p.mask.ptr + (static_cast<size_t>(mh) * p.mask.nbr + qt) * p.mask.nbc;
    const int lim = n_kv;
    const int cnt = compact_steps<1>(
        p.mask.nbc, [&](int e) { return mrow[e] != 0; },
        [&](int e, int) { return e < lim ? e : -1; }, tile_list, kDqListCap);
    if (lane == 0) *list_count = min(cnt, kDqListCap);
  }
  auto key_tile = [&](int j) -> int { return sparse ? static_cast<int>(tile_list[j]) : j; };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQDFull), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
      mbar_init(bar(L::kSFull + s), 1);
    }
    mbar_init(bar(L::kDPFull), 1);
    // one arrival per dS warp.  DS_FULL alternates between two barriers: a
    // warp may arrive for tile j + 1 (its dP_{j+1} is issued once every warp
    // has read dP_j) before a slower one has arrived for tile j
    mbar_init(bar(L::kDSFull), 8);
    mbar_init(bar(L::kDSFull + 1), 8);
    mbar_init(bar(L::kDPRead), 8);
    mbar_init(bar(L::kDQDone), 1);
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
  if (sparse) n_kv = *list_count;
  const uint32_t tmem = *tmem_holder;
  const uint32_t tdP = tmem + L::kTdP, tdQ = tmem + L::kTdQ;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(L::kQDFull), 2 * L::kTile);
      #pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_4d(sbase + L::kQOff + c * (BR * 128), &tm_q, bar(L::kQDFull), c * 64, qt * BR, h, b);
        tma_load_4d(sbase + L::kDOOff + c * (BR * 128), &tm_do, bar(L::kQDFull), c * 64, qt * BR,
                    h, b);
      }
    }
    __syncwarp();
    int k_issued = 0, v_issued = 0;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1, sk = j % KST;
      if (j >= KST && !wait_uniform(bar(L::kKEmpty + sk), ((j / KST) + 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kKFull + sk), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kKOff + sk * L::kTile + c * (BC * 128), &tm_k, bar(L::kKFull + sk),
                      c * 64, key_tile(j) * BC, kh, b);
      }
      __syncwarp();
      ++k_issued;
      if (j >= 2 && !wait_uniform(bar(L::kVEmpty + s), ((j >> 1) + 1) & 1, abort)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(bar(L::kVFull + s), L::kTile);
        #pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sbase + L::kVOff + s * L::kTile + c * (BC * 128), &tm_v, bar(L::kVFull + s),
                      c * 64, key_tile(j) * BC, kh, b);
      }
      __syncwarp();
      ++v_issued;
    }
    drain_wait(bar(L::kQDFull), 0);
    for (int j = max(0, k_issued - KST); j < k_issued; ++j)
      drain_wait(bar(L::kKFull + j % KST), (j / KST) & 1);
    for (int j = max(0, v_issued - 2); j < v_issued; ++j)
      drain_wait(bar(L::kVFull + (j & 1)), (j >> 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(BR, BC, BF16 ? 1 : 0, 0, 0);   // S, dP
    constexpr uint32_t kIdQ = idesc_f16(BR, D, BF16 ? 1 : 0, 0, 1);    // dQ (B = K MN-major)
    const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t do_desc = smem_desc_sw128(sbase + L::kDOOff, 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sbase + L::kVOff, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(sbase + L::kKOff, BC * 128, 1024);
    auto issue_s = [&](int j) -> bool {
      const int s = j & 1, sk = j % KST;
      if (!wait_uniform(bar(L::kKFull + sk), (j / KST) & 1, abort)) return false;
      tc_fence_after();
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tmem + L::kTS + 128 * s, desc_add(q_desc, c * (BR * 128) + w * 32),
               desc_add(k_desc, sk * L::kTile + c * (BC * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull + s));
      return true;
    };
    auto issue_dp = [&](int j) -> bool {
      const int s = j & 1;
      if (!wait_uniform(bar(L::kVFull + s), (j >> 1) & 1, abort)) return false;
      tc_fence_after();
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tdP, desc_add(do_desc, c * (BR * 128) + w * 32),
               desc_add(v_desc, s * L::kTile + c * (BC * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kDPFull));
      mma_commit(bar(L::kVEmpty + s));   // V_j is not read again
      return true;
    };
    bool ok = wait_uniform(bar(L::kQDFull), 0, abort);
    if (ok && n_kv > 0) ok = issue_s(0) && issue_dp(0);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j & 1;
      // the other S buffer: its dS (tile j - 1) was read by dQ_{j-1}, issued earlier
      if (j + 1 < n_kv && !issue_s(j + 1)) break;
      // dP_{j+1} as soon as the dS warps hold dP_j in registers, so it runs
      // while they form dS_j
      if (j + 1 < n_kv) {
        if (!wait_uniform(bar(L::kDPRead), j & 1, abort)) break;
        tc_fence_after();
        if (!issue_dp(j + 1)) break;
      }
      if (!wait_uniform(bar(L::kDSFull + (j & 1)), (j >> 1) & 1, abort)) break;
      tc_fence_after();
      // dQ += dS_j K_j: dS (16-bit) in the first 32 columns of each 64-column
      // half of S buffer s (one half per dS warp)
      const int sk = j % KST;
      #pragma unroll
      for (int kk = 0; kk < BC / 16; ++kk)
        mma_ts(tdQ, tmem + L::kTS + 128 * s + (kk >> 2) * 64 + (kk & 3) * 8,
               desc_add(k_mn, sk * L::kTile + kk * 2048), kIdQ, (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kKEmpty + sk));   // S_j and dQ_j were K_j's readers
    }
    mma_commit(bar(L::kDQDone));
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ dS warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;          // key columns [64 half, 64 half + 64)
    const int row = qt * BR + quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const size_t row_idx = (static_cast<size_t>(b) * p.H + h) * p.Nq + (row < p.Nq ? row : 0);
    const long long dq_off =
        b * p.dqs.b + h * p.dqs.h + static_cast<long long>(row < p.Nq ? row : 0) * p.dqs.n;
    const float nL = row < p.Nq ? -p.lse[row_idx] * kDqLog2e : -INFINITY;
    const float nD = row < p.Nq ? -p.delta[row_idx] : 0.f;
    const f2 cs = {p.scale_log2, p.scale_log2}, cl = {nL, nL}, cd = {nD, nD};
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int s = j & 1;
      const uint32_t tSb = tmem + L::kTS + 128 * s + lane_off + 64 * half;
      if (!wait_uniform(bar(L::kSFull + s), (j >> 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const int col0 = key_tile(j) * BC + 64 * half;
      const bool masked = (CAUSAL && col0 + 63 > qt * BR + p.off) || (col0 + 64 > p.Nk);
      float P[64];
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(tSb + c0, sr);
        tmem_ld_wait();
        reg_fence(sr);
        #pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const f2 arg = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs, cl);
          P[c0 + c] = ex2_approx(arg.x);
          P[c0 + c + 1] = ex2_approx(arg.y);
        }
        if (masked) {
          // columns [0, lim) of this chunk are kept (one comparison per score)
          const int lim = min(p.Nk - col0 - c0, CAUSAL ? row + p.off - col0 - c0 + 1 : 32);
          #pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= lim) P[c0 + c] = 0.f;
        }
      }
      if (!wait_uniform(bar(L::kDPFull), j & 1, abort)) { ok = false; break; }
      tc_fence_after();
      // all 64 dP values of this half into registers, then release the dP
      // columns for dP_{j+1}
      uint32_t dr[64];
      tmem_ld32(tdP + lane_off + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld32(tdP + lane_off + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_ld_wait();
      reg_fence(dr);
      tc_fence_before();
      mbar_arrive_warp(bar(L::kDPRead));
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t w[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          const f2 ds = fmul2(f2{P[c0 + 2 * c], P[c0 + 2 * c + 1]},
                              fadd2(f2{__uint_as_float(dr[c0 + 2 * c]),
                                       __uint_as_float(dr[c0 + 2 * c + 1])}, cd));
          w[c] = pack2<BF16>(ds.x, ds.y);
        }
        // dS (16-bit) over the first 32 columns of this half, already read
        tmem_st16(tSb + c0 / 2, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bar(L::kDSFull + (j & 1)));
    }
    // ------------------------------------------------------------ epilogue
    uint4* out = reinterpret_cast<uint4*>(p.dq + dq_off + 64 * half);
    if (ok && n_kv == 0) {
      if (row < p.Nq) {
        #pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else if (ok && wait_uniform(bar(L::kDQDone), 0, abort)) {
      tc_fence_after();
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tdQ + lane_off + 64 * half + c0, v);
        tmem_ld_wait();
        reg_fence(v);
        uint32_t o[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * p.scale, __uint_as_float(v[2 * i + 1]) * p.scale);
        if (row < p.Nq) {
          #pragma unroll
          for (int i = 0; i < 4; ++i)
            out[c0 / 8 + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
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

template <bool CAUSAL, bool BF16, bool SPARSE>
cudaError_t launch_dq128(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  using L = Dq128Layout<SPARSE ? 2 : 3>;
  CUtensorMap tq, tk, tv, tdo;
  cudaError_t e;
  if ((e = make_tmap_4d(&tq, a.q, 128, pr.Nq, pr.H, pr.B, a.qs, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, 128, pr.Nq, pr.H, pr.B, a.dos, 64, 128)) != cudaSuccess)
    return e;
  if ((e = make_tmap_4d(&tk, a.k, 128, pr.Nk, pr.Hkv, pr.B, a.ks, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, 128, pr.Nk, pr.Hkv, pr.B, a.vs, 64, 128)) != cudaSuccess) return e;
  auto kern = bwd_dq128_kernel<CAUSAL, BF16, SPARSE>;
  constexpr int kSmem = SPARSE ? L::kAlloc : L::kAllocDense;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
        cudaSuccess)
      return e;
    attr_set = true;
  }
  DqParams p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<uint16_t*>(a.dq);
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.G = pr.H / pr.Hkv;
  p.num_q_tiles = (pr.Nq + 127) / 128;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kDqLog2e;
  p.mask = a.mask;
  p.dqs = a.dqs;
  p.err = pr.err;
  dim3 grid(p.num_q_tiles, pr.H, pr.B);
  const int slot = timing_begin(FA_KERNEL_BWD_DQ, stream);
  kern<<<grid, kDq128Threads, kSmem, stream>>>(tq, tk, tv, tdo, p);
  timing_end(slot, stream);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// d = 256, dense: 128-key tiles, so S and dP are N = 128 products and dQ an
// N = 256 one (full rate; with 64-key tiles S and dP ran at half rate).
// Shared memory: Q and dO (64 KB each, for the whole CTA), one K tile (64 KB,
// read by S_j as four 64-column chunks of d and by dQ_j as two halves of d)
// and a ring of two 64-column chunks of V.  TMEM: S (128 columns), dP (128;
// dS written over it in 16 bits), dQ (256).
// Issue order per key tile j:  dQ(j-1), dP(j), S(j)
// dQ(j-1) is K_{j-1}'s last reader; its two halves release the K tile's two
// halves, so K_j loads while dP(j) runs.  dS(j) goes over the dP columns
// (the warps hold dP(j) in registers by then), so dP(j+1), issued after
// dQ(j), is the first product to overwrite it.
// Warps: 0 producer of Q, dO and K; 10 producer of V; 1 MMA issuer; 2..9 dS
// (a query row per thread; warps w and w + 4 share a TMEM lane quarter and
// split the 128 key columns in halves).
constexpr int kDq256Threads = 352;

struct Dq256Layout {
  static constexpr int kChunk = 128 * 64 * 2;     // [128 rows][64 cols] 16-bit, 128-byte swizzle
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = 4 * kChunk;
  static constexpr int kKOff = 8 * kChunk;
  static constexpr int kVOff = 12 * kChunk;       // two slots
  static constexpr int kBarOff = 14 * kChunk;
  static constexpr int kQDFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 7, kSFull = 9,
                       kDPFull = 10, kDSFull = 11, kDQDone = 13, kDrain = 14, kNumBars = 15;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTS = 0, kTdP = 128, kTdQ = 256, kTmemCols = 512;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kDq256Threads, 1)
bwd_dq256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const DqParams p) {
  using L = Dq256Layout;
  constexpr int BR = 128, BC = 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = CAUSAL ? (p.num_q_tiles - 1 - static_cast<int>(blockIdx.x))
                        : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int kh = h / p.G;
  int n_kv = (p.Nk + BC - 1) / BC;
  if (CAUSAL) {
    const int last_key = min((qt + 1) * BR, p.Nq) - 1 + p.off;
    n_kv = last_key < 0 ? 0 : min(n_kv, last_key / BC + 1);
  }
  // The CTAs of a head start their walk over the key tiles at different
  // tiles (query tile qt at tile qt mod n_kv): walking in step, every CTA
  // asked for each tile first, so every tile's loads waited for DRAM; now a
  // tile is mostly in L2 by the time the next CTA reaches it.  (dQ sums the
  // tiles in this fixed order, the same on every run.)
  auto key_tile = [&](int j) { return n_kv > 0 ? (j + qt) % n_kv : 0; };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQDFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
      mbar_init(bar(L::kDSFull + s), 8);     // one arrival per dS warp, alternating by tile
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kDPFull), 1);
    mbar_init(bar(L::kDQDone), 1);
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
  const uint32_t tS = tmem + L::kTS, tdP = tmem + L::kTdP, tdQ = tmem + L::kTdQ;

  if (warp == 0) {
    // ------------------------------------------------------------ Q, dO, K
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(L::kQDFull), 8 * L::kChunk);
      #pragma unroll
      for (int c = 0; c < 4; ++c) {
        tma_load_4d(sbase + L::kQOff + c * L::kChunk, &tm_q, bar(L::kQDFull), c * 64, qt * BR, h, b);
        tma_load_4d(sbase + L::kDOOff + c * L::kChunk, &tm_do, bar(L::kQDFull), c * 64, qt * BR, h, b);
      }
    }
    __syncwarp();
    int issued[2] = {0, 0};
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      #pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        // half hh of K_j (chunks 2 hh, 2 hh + 1) once dQ(j - 1) has read K_{j-1}'s
        if (j >= 1 && !wait_uniform(bar(L::kKEmpty + hh), (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(L::kKFull + hh), 2 * L::kChunk);
          #pragma unroll
          for (int c = 2 * hh; c < 2 * hh + 2; ++c)
            tma_load_4d(sbase + L::kKOff + c * L::kChunk, &tm_k, bar(L::kKFull + hh), c * 64,
                        key_tile(j) * BC, kh, b);
        }
        __syncwarp();
        ++issued[hh];
      }
    }
    drain_wait(bar(L::kQDFull), 0);
    for (int hh = 0; hh < 2; ++hh)
      if (issued[hh] > 0) drain_wait(bar(L::kKFull + hh), (issued[hh] - 1) & 1);
  } else if (warp == 10) {
    // ------------------------------------------------------------ V
    if (elect_one()) tma_prefetch_desc(&tm_v);
    __syncwarp();
    int i = 0;   // chunks issued
    for (int j = 0; j < n_kv; ++j) {
      bool ok = true;
      #pragma unroll 1
      for (int c = 0; c < 4; ++c, ++i) {
        const int s = i & 1;
        if (i >= 2 && !wait_uniform(bar(L::kVEmpty + s), ((i >> 1) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(L::kVFull + s), L::kChunk);
          tma_load_4d(sbase + L::kVOff + s * L::kChunk, &tm_v, bar(L::kVFull + s), c * 64,
                      key_tile(j) * BC, kh, b);
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    for (int k = max(0, i - 2); k < i; ++k) drain_wait(bar(L::kVFull + (k & 1)), (k >> 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(BR, BC, BF16 ? 1 : 0, 0, 0);   // S, dP
    constexpr uint32_t kIdQ = idesc_f16(BR, 128, BF16 ? 1 : 0, 0, 1);  // dQ halves (B = K MN-major)
    const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t do_desc = smem_desc_sw128(sbase + L::kDOOff, 16, 1024);
    const uint64_t k_desc = smem_desc_sw128(sbase + L::kKOff, 16, 1024);
    const uint64_t v_desc = smem_desc_sw128(sbase + L::kVOff, 16, 1024);
    const uint64_t k_mn = smem_desc_sw128(sbase + L::kKOff, L::kChunk, 1024);
    int vi = 0;   // V chunks read
    // dQ += dS_j K_j: dS (16-bit) in the first 32 columns of each 64-column
    // half of the dP columns (one half per dS warp); each half of d releases
    // its half of the K tile
    auto issue_dq = [&](int j) -> bool {
      if (!wait_uniform(bar(L::kDSFull + (j & 1)), (j >> 1) & 1, abort)) return false;
      tc_fence_after();
      #pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        #pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk)
          mma_ts(tdQ + 128 * hh, tdP + (kk >> 2) * 64 + (kk & 3) * 8,
                 desc_add(k_mn, hh * 2 * L::kChunk + kk * 2048), kIdQ, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kKEmpty + hh));
      }
      return true;
    };
    // dP_j = dO V_j^T, V in chunks of d through the ring
    auto issue_dp = [&](int j) -> bool {
      #pragma unroll 1
      for (int c = 0; c < 4; ++c, ++vi) {
        const int s = vi & 1;
        if (!wait_uniform(bar(L::kVFull + s), (vi >> 1) & 1, abort)) return false;
        tc_fence_after();
        #pragma unroll
        for (int w = 0; w < 4; ++w)
          mma_ss(tdP, desc_add(do_desc, c * L::kChunk + w * 32),
                 desc_add(v_desc, s * L::kChunk + w * 32), kIdS, (c | w) ? 1u : 0u);
        mma_commit(bar(L::kVEmpty + s));
      }
      mma_commit(bar(L::kDPFull));
      return true;
    };
    // S_j = Q K_j^T, K_j's two halves as they land
    auto issue_s = [&](int j) -> bool {
      #pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        if (!wait_uniform(bar(L::kKFull + hh), j & 1, abort)) return false;
        tc_fence_after();
        #pragma unroll
        for (int kk = 8 * hh; kk < 8 * hh + 8; ++kk) {
          const uint32_t c = kk >> 2, w = kk & 3;
          mma_ss(tS, desc_add(q_desc, c * L::kChunk + w * 32), desc_add(k_desc, c * L::kChunk + w * 32),
                 kIdS, kk > 0 ? 1u : 0u);
        }
      }
      mma_commit(bar(L::kSFull));
      return true;
    };
    bool ok = wait_uniform(bar(L::kQDFull), 0, abort);
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j >= 1 && !issue_dq(j - 1)) ok = false;
      else if (!issue_dp(j)) ok = false;
      else if (!issue_s(j)) ok = false;
    }
    if (ok && n_kv > 0) issue_dq(n_kv - 1);
    mma_commit(bar(L::kDQDone));
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ dS warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;          // key columns [64 half, 64 half + 64)
    const int row = qt * BR + quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const size_t row_idx = (static_cast<size_t>(b) * p.H + h) * p.Nq + (row < p.Nq ? row : 0);
    const long long dq_off =
        b * p.dqs.b + h * p.dqs.h + static_cast<long long>(row < p.Nq ? row : 0) * p.dqs.n;
    const float nL = row < p.Nq ? -p.lse[row_idx] * kDqLog2e : -INFINITY;
    const float nD = row < p.Nq ? -p.delta[row_idx] : 0.f;
    const f2 cs = {p.scale_log2, p.scale_log2}, cl = {nL, nL}, cd = {nD, nD};
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!wait_uniform(bar(L::kSFull), j & 1, abort)) { ok = false; break; }
      tc_fence_after();
      const int col0 = key_tile(j) * BC + 64 * half;
      const bool masked = (CAUSAL && col0 + 63 > qt * BR + p.off) || (col0 + 64 > p.Nk);
      float P[64];
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t sr[32];
        tmem_ld32(tS + lane_off + 64 * half + c0, sr);
        tmem_ld_wait();
        reg_fence(sr);
        #pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const f2 arg = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs, cl);
          P[c0 + c] = ex2_approx(arg.x);
          P[c0 + c + 1] = ex2_approx(arg.y);
        }
        if (masked) {
          // columns [0, lim) of this chunk are kept (one comparison per score)
          const int lim = min(p.Nk - col0 - c0, CAUSAL ? row + p.off - col0 - c0 + 1 : 32);
          #pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c >= lim) P[c0 + c] = 0.f;
        }
      }
      if (!wait_uniform(bar(L::kDPFull), j & 1, abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t dr[64];
      tmem_ld32(tdP + lane_off + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld32(tdP + lane_off + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_ld_wait();
      reg_fence(dr);
      #pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t w[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          const f2 ds = fmul2(f2{P[c0 + 2 * c], P[c0 + 2 * c + 1]},
                              fadd2(f2{__uint_as_float(dr[c0 + 2 * c]),
                                       __uint_as_float(dr[c0 + 2 * c + 1])}, cd));
          w[c] = pack2<BF16>(ds.x, ds.y);
        }
        // dS (16-bit) over the first 32 columns of this half of dP, read above
        tmem_st16(tdP + lane_off + 64 * half + c0 / 2, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(bar(L::kDSFull + (j & 1)));
    }
    // ------------------------------------------------------------ epilogue
    uint4* out = reinterpret_cast<uint4*>(p.dq + dq_off + 128 * half);
    if (ok && n_kv == 0) {
      if (row < p.Nq) {
        #pragma unroll
        for (int i = 0; i < 16; ++i) out[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else if (ok && wait_uniform(bar(L::kDQDone), 0, abort)) {
      tc_fence_after();
      #pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tdQ + lane_off + 128 * half + c0, v);
        tmem_ld_wait();
        reg_fence(v);
        uint32_t o[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * p.scale, __uint_as_float(v[2 * i + 1]) * p.scale);
        if (row < p.Nq) {
          #pragma unroll
          for (int i = 0; i < 4; ++i)
            out[c0 / 8 + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
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
  // launched as the dK / dV pair kernel's programmatic dependent (it needs
  // none of that kernel's results, only D): this grid ends only after that
  // one has, so whatever follows on the stream sees dK and dV as well
  grid_dependency_wait();
}

template <bool CAUSAL, bool BF16>
cudaError_t launch_dq256(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  using L = Dq256Layout;
  CUtensorMap tq, tk, tv, tdo;
  cudaError_t e;
  if ((e = make_tmap_4d(&tq, a.q, 256, pr.Nq, pr.H, pr.B, a.qs, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, 256, pr.Nq, pr.H, pr.B, a.dos, 64, 128)) != cudaSuccess)
    return e;
  if ((e = make_tmap_4d(&tk, a.k, 256, pr.Nk, pr.Hkv, pr.B, a.ks, 64, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, 256, pr.Nk, pr.Hkv, pr.B, a.vs, 64, 128)) != cudaSuccess) return e;
  auto kern = bwd_dq256_kernel<CAUSAL, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc)) !=
        cudaSuccess)
      return e;
    attr_set = true;
  }
  DqParams p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<uint16_t*>(a.dq);
  p.H = pr.H;
  p.Hkv = pr.Hkv;
  p.Nq = pr.Nq;
  p.Nk = pr.Nk;
  p.off = pr.Nk - pr.Nq;
  p.G = pr.H / pr.Hkv;
  p.num_q_tiles = (pr.Nq + 127) / 128;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kDqLog2e;
  p.mask = BlockMask{};
  p.dqs = a.dqs;
  p.err = pr.err;
  // Always right behind the dK / dV pair kernel, which issues
  // grid_launch_dependents at its start: this grid's CTAs take the SMs that
  // kernel's last, partly filled wave leaves idle.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_q_tiles, pr.H, pr.B);
  cfg.blockDim = dim3(kDq256Threads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int slot = timing_begin(FA_KERNEL_BWD_DQ, stream);
  e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, p);
  timing_end(slot, stream);
  return e;
}

template <int D, int KST, bool SPARSE>
cudaError_t dispatch_dq(const Problem& pr, const BwdArgs& a, cudaStream_t s) {
  if (pr.causal)
    return pr.bf16 ? launch_dq_variant<D, KST, true, true, SPARSE>(pr, a, s)
                   : launch_dq_variant<D, KST, true, false, SPARSE>(pr, a, s);
  return pr.bf16 ? launch_dq_variant<D, KST, false, true, SPARSE>(pr, a, s)
                 : launch_dq_variant<D, KST, false, false, SPARSE>(pr, a, s);
}

// K / V ring stages per head dimension.
template <bool SPARSE>
cudaError_t launch_bwd_dq_for(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (pr.d == 128) {
    if (pr.causal)
      return pr.bf16 ? launch_dq128<true, true, SPARSE>(pr, a, stream)
                     : launch_dq128<true, false, SPARSE>(pr, a, stream);
    return pr.bf16 ? launch_dq128<false, true, SPARSE>(pr, a, stream)
                   : launch_dq128<false, false, SPARSE>(pr, a, stream);
  }
  if constexpr (!SPARSE) {
    if (pr.d == 256) {
      if (pr.causal)
        return pr.bf16 ? launch_dq256<true, true>(pr, a, stream) : launch_dq256<true, false>(pr, a, stream);
      return pr.bf16 ? launch_dq256<false, true>(pr, a, stream) : launch_dq256<false, false>(pr, a, stream);
    }
  }
  switch (pr.d) {
    case 64: return dispatch_dq<64, 4, SPARSE>(pr, a, stream);
    case 256: return dispatch_dq<256, 1, SPARSE>(pr, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace fa
