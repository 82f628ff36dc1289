// Fused backward at d = 128: all five products of a (key tile, query tile)
// step in one kernel, dQ accumulated across key tiles with atomic adds.
//
// Method ("FlashAttention-2: Faster Attention with Better Parallelism and
// Work Partitioning", paper digest):
//  - section 2 Q2, improvement 2 (backward): the outer loop runs over
//    key/value tiles, dK and dV stay on chip, and dQ is accumulated across
//    key/value tiles with atomic adds;
//  - section 3 "FLOPs": five products per tile, S = Q K^T, dP = dO V^T,
//    dV += P^T dO, dK += dS^T Q, dQ += dS K, with dS = P o (dP - D);
//  - section 4 "logsumexp fusion": P = exp(S - L) from the saved L;
//  - section 4 "six checks", GQA/MQA: one unit walks every query head of its
//    key/value head, so the dK and dV sums over the group stay in TMEM.
//
// Persistent: one CTA per SM takes units (batch, key/value head, 128-key
// tile) from a work counter until none are left, so that one unit's tail
// (its last products, the dK / dV write-out) overlaps the next unit's start
// (its K / V load, first scores and softmax weights).  Units are numbered in
// one of two orders chosen on the host: key tiles fastest (the units of a
// (batch, kv head) group run together and share its Q and dO in L2), with
// the last few groups taken longest key tile first so the launch does not
// end on one long unit; or heavy first (longest key tiles of every group
// first) when single units are long.
//
// Warps (14): 0 TMA producer (the unit counter; K, V once per unit; Q in two
// stages, dO in one); 1 MMA issuer; 2..9 P / dS (a key row per thread; warps
// w and w + 4 share a TMEM lane quarter and split the 128 query columns in
// halves); 10..13 dQ, and the dK / dV write-out of each unit.
// TMEM: dV (128 columns) | dK (128) | S^T (128, P^T over it in 16 bits) |
// dP^T (128, dQ^T over it once the dS warps have read dP^T).
// Issue order per step t:  dV(t), S^T(t+1), dQ^T(t), dK(t), dP^T(t+1)
// dQ^T(t) and dK(t) read dS^T from shared memory.  dP^T(t + 1) overwrites
// dQ^T(t), so it waits until the dQ warps have read dQ^T(t) out of TMEM.
// Between units: S^T(0) and dP^T(0) of the next unit once its K and V have
// landed (loaded after the last products that read the previous K and V);
// dV(0) once the dK / dV columns have been read out.
//
// Adding dQ to the fp32 accumulator is 64 KB of reductions per step.  As
// red.global instructions (one 128-byte line per warp instruction) they
// cost ~2,000 cycles of the SM's load/store path per step (a clock-stamp
// trace), which is as long as the step's products.  Here the dQ warps write
// the dQ tile (fp32) in quarters of 32 query rows to shared-memory staging
// buffers, and one thread hands each to the tensor memory accelerator as a
// bulk reduce-add into the accumulator (cp.reduce.async.bulk.tensor), so the
// additions leave the SM as whole 16 KB tiles (~21 bytes per clock per SM,
// measured).  The dP columns are released as soon as the last quarter is in
// registers.  dK and dV leave through the same staging buffers as 16-bit
// tiles by TMA stores.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

namespace {

constexpr int kFusedThreads = 448;

struct FusedLayout {
  static constexpr int kTile = 128 * 128 * 2;        // one 128 x 128 16-bit tile
  static constexpr int kQStages = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTile;
  static constexpr int kQOff = 2 * kTile;            // kQStages stages
  static constexpr int kDOOff = (2 + kQStages) * kTile;
  static constexpr int kDSOff = kDOOff + kTile;      // dS^T [keys][q], 128-byte swizzle
  static constexpr int kStgOff = kDSOff + kTile;     // dQ staging [64 q][128 d] fp32; dK / dV out
  static constexpr int kLDOff = kStgOff + kTile;     // [2 halves][2 bufs][-L*log2e | -D][64]
  static constexpr int kBarOff = kLDOff + 2 * 2 * 2 * 64 * 4;
  static constexpr int kKVFull = 0, kKVEmpty = 1, kQFull = 2, kQEmpty = kQFull + kQStages,
                       kDOFull = kQEmpty + kQStages, kDOEmpty = kDOFull + 1,
                       kSFull = kDOEmpty + 1, kDPFull = kSFull + 1, kPFull = kDPFull + 1,
                       kDSFull = kPFull + 1, kDSEmpty = kDSFull + 1, kDQFull = kDSEmpty + 1,
                       kDQEmpty = kDQFull + 1, kFinal = kDQEmpty + 1, kAccEmpty = kFinal + 1,
                       kUnitFull = kAccEmpty + 1, kUnitEmpty = kUnitFull + 2,
                       kDrain = kUnitEmpty + 2, kNumBars = kDrain + 1;
  // TMEM base, abort flag, two unit records {key tile, kv head, batch, steps}
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kUnitOff = kMiscOff + 16;
  static constexpr int kBytes = kUnitOff + 2 * 16;
  // The whole opt-in maximum: the layout needs a 1024-byte-aligned base
  // (128-byte swizzle atoms) and leaves less than 1024 bytes of slack, so the
  // kernel checks the base it gets.
  static constexpr int kAlloc = 227 * 1024;
  static constexpr uint32_t kTdV = 0, kTdK = 128, kTS = 256, kTdP = 384, kTmemCols = 512;
  static_assert(kBytes <= kAlloc, "shared memory budget");
  static_assert(kUnitOff % 16 == 0, "unit records are 16-byte aligned");
};

// Named barrier of the four dQ warps (id 0 is __syncthreads).
constexpr int kDqBarrier = 1;
// Warps that read each unit record (MMA, P / dS, dQ).
constexpr int kUnitReaders = 13;

// Unit u of the launch's order -> (key tile, kv head, batch).
__device__ __forceinline__ void fused_unit(const BwdParams& p, int u, int& jt, int& kh, int& b) {
  int grp;
  if (p.heavy_first) {
    jt = u / p.n_groups;
    grp = u % p.n_groups;
  } else {
    const int body = (p.n_groups - p.tail_groups) * p.n_kv_tiles;
    if (u < body) {
      jt = u % p.n_kv_tiles;
      grp = u / p.n_kv_tiles;
    } else {
      const int v = u - body;
      jt = v / p.tail_groups;
      grp = p.n_groups - p.tail_groups + v % p.tail_groups;
    }
  }
  kh = grp % p.Hkv;
  b = grp / p.Hkv;
}

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kFusedThreads, 1)
bwd128_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dqacc,
                   const __grid_constant__ CUtensorMap tm_dk,
                   const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using L = FusedLayout;
  constexpr int D = 128, BR = 128, QS = L::kQStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  if (sbase + L::kBytes > raw + L::kAlloc) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemBase);
    return;
  }
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* unit_rec = reinterpret_cast<volatile int*>(smem + L::kUnitOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Steps of a unit: query tiles from the last down to the first its key
  // tile sees, all G heads of the group for each (heads innermost).  Every
  // unit has at least G steps: under the mask key k < Nk is seen by query
  // k - (Nk - Nq) < Nq.
  auto steps_of = [&](int jt) {
    return p.G * max(0, p.n_q_tiles - (CAUSAL ? max(0, jt * kBC - p.off) / BR : 0));
  };
  auto step_hq = [&](int kh, int t, int& h, int& q0) {
    const int g = t % p.G;
    h = kh * p.G + g;
    q0 = (p.n_q_tiles - 1 - t / p.G) * BR;
  };
  // The k-th unit record of this CTA {key tile, kv head, batch, steps; no
  // steps: no more units}, read by a whole warp once the producer has
  // published it; false once the wait gave up.
  auto read_unit = [&](int k, int (&rec)[4]) -> bool {
    if (!wait_uniform(bar(L::kUnitFull + (k & 1)), (k >> 1) & 1, abort)) return false;
    #pragma unroll
    for (int i = 0; i < 4; ++i) rec[i] = unit_rec[4 * (k & 1) + i];
    mbar_arrive_warp(bar(L::kUnitEmpty + (k & 1)));
    return true;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVFull), 1);
    mbar_init(bar(L::kKVEmpty), 1);
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
    mbar_init(bar(L::kDQEmpty), 4);        // one arrival per dQ warp
    mbar_init(bar(L::kFinal), 1);
    mbar_init(bar(L::kAccEmpty), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kUnitFull + s), 1);
      mbar_init(bar(L::kUnitEmpty + s), kUnitReaders);
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
  const uint32_t tdV = tmem + L::kTdV, tdK = tmem + L::kTdK, tS = tmem + L::kTS,
                 tdP = tmem + L::kTdP;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_dqacc);
      tma_prefetch_desc(&tm_dk);
      tma_prefetch_desc(&tm_dv);
    }
    __syncwarp();
    // the first unit is the CTA's index, later ones come from the counter
    int u = blockIdx.x;
    int k = 0, g = 0;                  // units and steps of this CTA so far
    int q_issued = 0, do_issued = 0, kv_issued = 0;
    bool ok = true;
    while (ok) {
      int jt = 0, kh = 0, b = 0, n = 0;
      if (u < p.n_units) {
        fused_unit(p, u, jt, kh, b);
        n = steps_of(jt);
      }
      // publish the record (n = 0: no more units)
      if (k >= 2 && !wait_uniform(bar(L::kUnitEmpty + (k & 1)), ((k >> 1) - 1) & 1, abort)) break;
      if (elect_one()) {
        unit_rec[4 * (k & 1) + 0] = jt;
        unit_rec[4 * (k & 1) + 1] = kh;
        unit_rec[4 * (k & 1) + 2] = b;
        unit_rec[4 * (k & 1) + 3] = n;
        mbar_arrive(bar(L::kUnitFull + (k & 1)));
      }
      __syncwarp();
      if (n == 0) break;
      const int kv0 = jt * kBC;
      for (int t = 0; t < n; ++t) {
        const int gs = g + t, s = gs % QS;
        if (gs >= QS && !wait_uniform(bar(L::kQEmpty + s), ((gs / QS) + 1) & 1, abort)) {
          ok = false;
          break;
        }
        int h, q0;
        step_hq(kh, t, h, q0);
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(L::kQFull + s), L::kTile);
          #pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sbase + L::kQOff + s * L::kTile + c * (BR * 128), &tm_q, bar(L::kQFull + s),
                        c * 64, q0, h, b);
        }
        __syncwarp();
        ++q_issued;
        if (gs >= 1 && !wait_uniform(bar(L::kDOEmpty), (gs - 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(L::kDOFull), L::kTile);
          #pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sbase + L::kDOOff + c * (BR * 128), &tm_do, bar(L::kDOFull), c * 64, q0, h, b);
        }
        __syncwarp();
        ++do_issued;
        if (t == 0) {
          // K and V of this unit once the previous unit's last products
          // that read them have completed (its first Q and dO are already
          // on their way)
          if (k >= 1 && !wait_uniform(bar(L::kKVEmpty), (k - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(L::kKVFull), 2 * L::kTile);
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
              tma_load_4d(sbase + L::kKOff + c * (kBC * 128), &tm_k, bar(L::kKVFull), c * 64, kv0, kh, b);
              tma_load_4d(sbase + L::kVOff + c * (kBC * 128), &tm_v, bar(L::kKVFull), c * 64, kv0, kh, b);
            }
          }
          __syncwarp();
          ++kv_issued;
        }
      }
      if (!ok) break;
      // the next unit, taken once this one's loads are all issued; its K and
      // V are fetched into L2 meanwhile
      unsigned int nu = 0;
      if (lane == 0) nu = atomicAdd(p.units, 1u);
      u = static_cast<int>(__shfl_sync(0xffffffffu, nu, 0) + gridDim.x);
      if (u < p.n_units && elect_one()) {
        int njt, nkh, nb;
        fused_unit(p, u, njt, nkh, nb);
        #pragma unroll
        for (int c = 0; c < 2; ++c) {
          tma_prefetch_l2_4d(&tm_k, c * 64, njt * kBC, nkh, nb);
          tma_prefetch_l2_4d(&tm_v, c * 64, njt * kBC, nkh, nb);
        }
      }
      __syncwarp();
      g += n;
      ++k;
    }
    // nothing may land in shared memory after the CTA has exited
    if (kv_issued > 0) drain_wait(bar(L::kKVFull), (kv_issued - 1) & 1);
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
    // S^T of global step gs = K Q^T into the S columns
    auto issue_s = [&](int gs) -> bool {
      if (!wait_uniform(bar(L::kQFull + gs % QS), (gs / QS) & 1, abort)) return false;
      tc_fence_after();
      const uint32_t qs = (gs % QS) * L::kTile;
      #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t c = kk >> 2, w = kk & 3;
        mma_ss(tS, desc_add(k_kmaj, c * (kBC * 128) + w * 32),
               desc_add(q_kmaj, qs + c * (BR * 128) + w * 32), kIdS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull));
      return true;
    };
    // dP^T of global step gs = V dO^T into the dP columns
    auto issue_dp = [&](int gs) -> bool {
      if (!wait_uniform(bar(L::kDOFull), gs & 1, abort)) return false;
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
    bool ok = true;
    for (int k = 0, g = 0; ok; ++k) {
      int rec[4];
      if (!read_unit(k, rec)) break;
      const int n = rec[3];
      if (n == 0) break;
      // first scores of the unit once its K and V have landed; dP^T(0) once
      // the previous step's dQ^T has left the dP columns
      if (!wait_uniform(bar(L::kKVFull), k & 1, abort) || !issue_s(g)) break;
      if (g >= 1 && !wait_uniform(bar(L::kDQEmpty), (g - 1) & 1, abort)) break;
      if (!issue_dp(g)) break;
      for (int t = 0; t < n; ++t) {
        const int gs = g + t;
        const uint32_t qs = (gs % QS) * L::kTile;
        // dV += P^T dO: P^T (16-bit) in the first 32 columns of each 64-column
        // half of the S columns (one half per P / dS warp); the first step
        // of a unit overwrites dV, so the previous unit's must be out
        if (!wait_uniform(bar(L::kPFull), gs & 1, abort)) { ok = false; break; }
        if (t == 0 && k >= 1 && !wait_uniform(bar(L::kAccEmpty), (k - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(do_mn, kk * 2048), kIdKV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kDOEmpty));      // dP^T and dV were dO's readers
        if (t + 1 < n && !issue_s(gs + 1)) { ok = false; break; }
        if (!wait_uniform(bar(L::kDSFull), gs & 1, abort)) { ok = false; break; }
        tc_fence_after();
        // dQ^T = K^T dS^T into the dP columns (their dP^T has been read)
        #pragma unroll
        for (int kk = 0; kk < kBC / 16; ++kk)
          mma_ss(tdP, desc_add(k_mn, kk * 2048), desc_add(ds_mn, kk * 2048), kIdQ, kk > 0 ? 1u : 0u);
        mma_commit(bar(L::kDQFull));
        if (t + 1 == n) mma_commit(bar(L::kKVEmpty));   // the unit's last reads of K and V
        // dK += dS^T Q
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ss(tdK, desc_add(ds_kmaj, (kk >> 2) * (kBC * 128) + (kk & 3) * 32),
                 desc_add(q_mn, qs + kk * 2048), kIdKV, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kQEmpty + gs % QS));
        mma_commit(bar(L::kDSEmpty));
        if (t + 1 == n) {
          mma_commit(bar(L::kFinal));     // dK and dV of the unit complete
        } else {
          if (!wait_uniform(bar(L::kDQEmpty), gs & 1, abort)) { ok = false; break; }
          if (!issue_dp(gs + 1)) { ok = false; break; }
        }
      }
      g += n;
    }
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else if (warp < 10) {
    // ------------------------------------------------------------ P / dS warps
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;            // query columns [64 half, 64 half + 64)
    const int r = quarter * 32 + lane;           // key row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // -L*log2(e) and -D of this half's 64 query columns, double-buffered by
    // step; the four warps of a half write the same values to one copy
    float* ld_base = reinterpret_cast<float*>(smem + L::kLDOff) + half * (2 * 2 * 64);
    // The loads are issued a step ahead and their values first touched when
    // they are stored: arithmetic on them right after the load would stall
    // the warp for the global-memory latency at a point where the next
    // scores are already waiting.
    float rl[2], rd[2];
    bool rv[2];
    auto load_ld = [&](int kh, int b, int t) {
      int h, q0;
      step_hq(kh, t, h, q0);
      const size_t base = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = q0 + 64 * half + lane + 32 * u;
        rv[u] = q < p.Nq;
        const size_t i = base + (rv[u] ? q : 0);
        rl[u] = __ldg(p.lse + i);
        rd[u] = __ldg(p.delta + i);
      }
    };
    auto store_ld = [&](int gs) {
      float* dst = ld_base + (gs & 1) * 128;
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        dst[lane + 32 * u] = rv[u] ? -rl[u] * kLog2e : -INFINITY;
        dst[64 + lane + 32 * u] = rv[u] ? -rd[u] : 0.f;
      }
    };
    bool ok = true;
    for (int k = 0, g = 0; ok; ++k) {
      int rec[4];
      if (!read_unit(k, rec)) break;
      const int kh = rec[1], b = rec[2], n = rec[3];
      if (n == 0) break;
      const int kv0 = rec[0] * kBC;
      const int kv = kv0 + r;
      // L and D of the unit's first step (the wait for its first scores,
      // behind the K / V load, covers the load latency)
      load_ld(kh, b, 0);
      store_ld(g);
      __syncwarp();
      for (int t = 0; t < n; ++t) {
        const int gs = g + t;
        int h_t, q0;
        step_hq(kh, t, h_t, q0);
        (void)h_t;
        const float* sL = ld_base + (gs & 1) * 128;  // -L * log2(e) of this half's columns
        const float* sD = sL + 64;                     // -D
        if (t + 1 < n) load_ld(kh, b, t + 1);
        if (!wait_uniform(bar(L::kSFull), gs & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const bool kv_out = kv >= p.Nk;
        const bool diag = CAUSAL && (q0 + p.off < kv0 + kBC);
        const bool masked = __any_sync(0xffffffffu, kv_out || diag);
        const f2 cs = {p.scale_log2, p.scale_log2};
        const int qc0 = q0 + 64 * half;              // first query of this half
        float P[64];
        // 32 columns at a time, the second chunk's TMEM load in flight while
        // the first is exponentiated
        auto p_chunk = [&](const uint32_t (&sr)[32], int c0) {
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
            // queries qc0 + c0 + c with c < z see no key kv (z = 32: the key
            // is past Nk); one comparison per score
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
        };
        {
          const uint32_t src = tS + lane_off + 64 * half;
          uint32_t sa[32], sb[32];
          tmem_ld32(src, sa);
          tmem_ld_wait();
          reg_fence(sa);
          tmem_ld32(src + 32, sb);
          p_chunk(sa, 0);
          tmem_ld_wait();
          reg_fence(sb);
          p_chunk(sb, 32);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(L::kPFull));
        // dS^T = P^T o (dP^T - D) into the swizzled dS^T tile (chunk = half)
        if (!wait_uniform(bar(L::kDPFull), gs & 1, abort)) { ok = false; break; }
        if (gs > 0 && !wait_uniform(bar(L::kDSEmpty), (gs - 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        // 16 columns at a time, the TMEM load of the next chunk in flight
        // while the current one is computed (P, 64 values, stays live)
        auto ds_chunk = [&](const uint32_t (&dr)[16], int c0) {
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
          #pragma unroll
          for (int u2 = 0; u2 < 2; ++u2) {
            const int u = c0 / 8 + u2;
            uint4* dst = reinterpret_cast<uint4*>(smem + L::kDSOff + half * (kBC * 128) + r * 128 +
                                                  ((u ^ (r & 7)) * 16));
            *dst = make_uint4(w[4 * u2], w[4 * u2 + 1], w[4 * u2 + 2], w[4 * u2 + 3]);
          }
        };
        {
          const uint32_t src = tdP + lane_off + 64 * half;
          uint32_t da[16], db[16];
          tmem_ld16(src, da);
          tmem_ld_wait();
          reg_fence(da);
          tmem_ld16(src + 16, db);
          ds_chunk(da, 0);
          tmem_ld_wait();
          reg_fence(db);
          tmem_ld16(src + 32, da);
          ds_chunk(db, 16);
          tmem_ld_wait();
          reg_fence(da);
          tmem_ld16(src + 48, db);
          ds_chunk(da, 32);
          tmem_ld_wait();
          reg_fence(db);
          ds_chunk(db, 48);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        mbar_arrive_warp(bar(L::kDSFull));
        if (t + 1 < n) {
          store_ld(gs + 1);
          __syncwarp();
        }
      }
      g += n;
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    // lane = column r of d: row r of dQ^T holds dQ[q0 + c][r] for the 128 c.
    // The tile leaves in four quarters of 32 query rows through two 16 KB
    // staging buffers, so that the tensor memory accelerator always has a
    // reduce in flight while the next quarter is staged.  One thread (the
    // elected lane of warp 10) issues the reduces, in the order A, B, A, B,
    // and before a buffer is written again waits until at most the other
    // buffer's reduce is still reading (bulk groups complete in order).
    // After a unit's last step the same warps write its dV and dK: key row r
    // of each goes through both buffers (a 128-byte-swizzled 16-bit tile, in
    // two 64-column boxes) and leaves by two TMA stores.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t buf[2] = {sbase + L::kStgOff, sbase + L::kStgOff + 16384};
    const bool issuer = warp == 10 && elect_one();
    uint32_t v[64];
    auto stage = [&](int which, int half) {     // v[32 half .. + 32) -> buffer `which`
      #pragma unroll
      for (int c = 0; c < 32; ++c)
        st_shared_f32(buf[which] + (c * D + r) * 4, __uint_as_float(v[32 * half + c]));
    };
    auto wait_free = [&](int pending) {         // at most `pending` bulk groups still reading
      if (issuer) {
        if (pending == 0) bulk_wait_read_all();
        else bulk_wait_read_one_left();
      }
      named_bar_sync(kDqBarrier, 128);
    };
    auto issue = [&](int which, int row, int plane) {
      fence_proxy_async_smem();
      named_bar_sync(kDqBarrier, 128);
      if (issuer) {
        tma_reduce_add_3d(&tm_dqacc, buf[which], 0, row, plane);
        bulk_commit_group();
      }
    };
    // key row r of the dV or dK columns (times mul) into the staging tile as
    // 16-bit values: columns 32 j .. 32 j + 31 are 16-byte chunks
    // 4 (j & 1) .. + 3 of box j / 2
    auto stage_kv = [&](uint32_t cols, float mul) {
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a[32];
        tmem_ld32(cols + lane_off + 32 * j, a);
        tmem_ld_wait();
        reg_fence(a);
        uint32_t w[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack2<BF16>(__uint_as_float(a[2 * c]) * mul, __uint_as_float(a[2 * c + 1]) * mul);
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int u = 4 * (j & 1) + i;
          uint4* dst = reinterpret_cast<uint4*>(smem + L::kStgOff + (j >> 1) * (kBC * 128) +
                                                r * 128 + ((u ^ (r & 7)) * 16));
          *dst = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    };
    auto store_kv = [&](const CUtensorMap* map, int kv0, int kh, int b) {
      fence_proxy_async_smem();
      named_bar_sync(kDqBarrier, 128);
      if (issuer) {
        tma_store_4d(map, buf[0], 0, kv0, kh, b);
        tma_store_4d(map, buf[1], 64, kv0, kh, b);
        bulk_commit_group();
      }
    };
    for (int k = 0, g = 0;; ++k) {
      // the four warps leave together or not at all (they meet at named
      // barriers below, which do not time out)
      int rec[4];
      if (!named_bar_and(kDqBarrier, 128, read_unit(k, rec))) break;
      const int kv0 = rec[0] * kBC, kh = rec[1], b = rec[2], n = rec[3];
      if (n == 0) break;
      bool ok = true;
      for (int t = 0; t < n; ++t) {
        const int gs = g + t;
        int h, q0;
        step_hq(kh, t, h, q0);
        const int plane = b * p.H + h;
        if (!named_bar_and(kDqBarrier, 128, wait_uniform(bar(L::kDQFull), gs & 1, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld32(tdP + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tdP + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        reg_fence(v);
        wait_free(1);          // buffer A: the previous step's third quarter has been read
        stage(0, 0);
        wait_free(0);          // buffer B: its fourth quarter too
        stage(1, 1);
        tmem_ld32(tdP + lane_off + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tdP + lane_off + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        reg_fence(v);
        tc_fence_before();
        mbar_arrive_warp(bar(L::kDQEmpty));     // the dP columns are free for the next dP^T
        issue(0, q0, plane);
        issue(1, q0 + 32, plane);
        wait_free(1);
        stage(0, 0);
        issue(0, q0 + 64, plane);
        wait_free(1);
        stage(1, 1);
        issue(1, q0 + 96, plane);
      }
      if (!ok) break;
      // dV and dK of the unit, each through both staging buffers
      if (!named_bar_and(kDqBarrier, 128, wait_uniform(bar(L::kFinal), k & 1, abort))) break;
      tc_fence_after();
      wait_free(0);
      stage_kv(tdV, 1.f);
      store_kv(&tm_dv, kv0, kh, b);
      wait_free(0);
      stage_kv(tdK, p.scale);
      tc_fence_before();
      mbar_arrive_warp(bar(L::kAccEmpty));      // dV and dK are out of TMEM
      store_kv(&tm_dk, kv0, kh, b);
      wait_free(0);            // the next step stages into both buffers
      g += n;
    }
    if (issuer) bulk_wait_all();
    __syncwarp();
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

}  // namespace
}  // namespace fa
