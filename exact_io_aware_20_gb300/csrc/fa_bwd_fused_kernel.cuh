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
//  - section 4 "six checks", GQA/MQA: one CTA walks every query head of its
//    key/value head, so the dK and dV sums over the group stay in TMEM.
//
// One CTA per (batch, key/value head, 128-key tile).  Warps (14): 0 TMA
// producer (K, V once; Q in two stages, dO in one); 1 MMA issuer; 2..9
// P / dS (a key row per thread; warps w and w + 4 share a TMEM lane quarter
// and split the 128 query columns in halves); 10..13 dQ.
// TMEM: dV (128 columns) | dK (128) | S^T (128, P^T over it in 16 bits) |
// dP^T (128, dQ^T over it once the dS warps have read dP^T).
// Issue order per step t:  dV(t), S^T(t+1), dQ^T(t), dK(t), dP^T(t+1)
// dQ^T(t) and dK(t) read dS^T from shared memory.  dP^T(t + 1) overwrites
// dQ^T(t), so it waits until the dQ warps have read dQ^T(t) out of TMEM.
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
// registers.
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
  static constexpr int kStgOff = kDSOff + kTile;     // dQ staging [64 q][128 d] fp32
  static constexpr int kLDOff = kStgOff + kTile;     // [2 halves][2 bufs][-L*log2e | -D][64]
  static constexpr int kBarOff = kLDOff + 2 * 2 * 2 * 64 * 4;
  static constexpr int kKVFull = 0, kQFull = 1, kQEmpty = kQFull + kQStages,
                       kDOFull = kQEmpty + kQStages, kDOEmpty = kDOFull + 1,
                       kSFull = kDOEmpty + 1, kDPFull = kSFull + 1, kPFull = kDPFull + 1,
                       kDSFull = kPFull + 1, kDSEmpty = kDSFull + 1, kDQFull = kDSEmpty + 1,
                       kDQEmpty = kDQFull + 1, kFinal = kDQEmpty + 1, kDrain = kFinal + 1,
                       kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  // The whole opt-in maximum: the layout needs a 1024-byte-aligned base
  // (128-byte swizzle atoms) and leaves less than 1024 bytes of slack, so the
  // kernel checks the base it gets.
  static constexpr int kAlloc = 227 * 1024;
  static constexpr uint32_t kTdV = 0, kTdK = 128, kTS = 256, kTdP = 384, kTmemCols = 512;
  static_assert(kBytes <= kAlloc, "shared memory budget");
};

// Named barrier of the four dQ warps (id 0 is __syncthreads).
constexpr int kDqBarrier = 1;

// Bit of the device error word: the dynamic shared memory base was not
// 1024-byte aligned and the layout did not fit behind the aligned base.
constexpr unsigned int kErrSmemBase = 2u;

template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kFusedThreads, 1)
bwd128_fused_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dqacc, const BwdParams p) {
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
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  // Steps: query tiles from the last down to the first the key tile sees,
  // all G heads of the group for each (heads innermost).
  const int n_steps = p.G * max(0, p.n_q_tiles - (CAUSAL ? max(0, kv0 - p.off) / BR : 0));
  auto step_hq = [&](int t, int& h, int& q0) {
    const int g = t % p.G;
    h = kh * p.G + g;
    q0 = (p.n_q_tiles - 1 - t / p.G) * BR;
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
    mbar_init(bar(L::kDQEmpty), 4);        // one arrival per dQ warp
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
      // dV += P^T dO: P^T (16-bit) in the first 32 columns of each 64-column
      // half of the S columns (one half per P / dS warp)
      if (!wait_uniform(bar(L::kPFull), t & 1, abort)) break;
      tc_fence_after();
      #pragma unroll
      for (int kk = 0; kk < BR / 16; ++kk)
        mma_ts(tdV, tS + (kk >> 2) * 64 + (kk & 3) * 8, desc_add(do_mn, kk * 2048), kIdKV,
               (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kDOEmpty));      // dP^T_t and dV_t were dO_t's readers
      if (t + 1 < n_steps && !issue_s(t + 1)) break;
      if (!wait_uniform(bar(L::kDSFull), t & 1, abort)) break;
      tc_fence_after();
      // dQ^T = K^T dS^T into the dP columns (their dP^T has been read)
      #pragma unroll
      for (int kk = 0; kk < kBC / 16; ++kk)
        mma_ss(tdP, desc_add(k_mn, kk * 2048), desc_add(ds_mn, kk * 2048), kIdQ, kk > 0 ? 1u : 0u);
      mma_commit(bar(L::kDQFull));
      // dK += dS^T Q
      #pragma unroll
      for (int kk = 0; kk < BR / 16; ++kk)
        mma_ss(tdK, desc_add(ds_kmaj, (kk >> 2) * (kBC * 128) + (kk & 3) * 32),
               desc_add(q_mn, qs + kk * 2048), kIdKV, (t > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar(L::kQEmpty + t % QS));
      mma_commit(bar(L::kDSEmpty));
      if (t + 1 < n_steps) {
        if (!wait_uniform(bar(L::kDQEmpty), t & 1, abort)) break;
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
    // -L*log2(e) and -D of this half's 64 query columns, double-buffered by
    // step; the four warps of a half write the same values to one copy
    float* ld_base = reinterpret_cast<float*>(smem + L::kLDOff) + half * (2 * 2 * 64);
    // The loads are issued a step ahead and their values first touched when
    // they are stored: arithmetic on them right after the load would stall
    // the warp for the global-memory latency at a point where the next
    // scores are already waiting.
    float rl[2], rd[2];
    bool rv[2];
    auto load_ld = [&](int t) {
      int h, q0;
      step_hq(t, h, q0);
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
    auto store_ld = [&](int t) {
      float* dst = ld_base + (t & 1) * 128;
      #pragma unroll
      for (int u = 0; u < 2; ++u) {
        dst[lane + 32 * u] = rv[u] ? -rl[u] * kLog2e : -INFINITY;
        dst[64 + lane + 32 * u] = rv[u] ? -rd[u] : 0.f;
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
      if (!wait_uniform(bar(L::kDPFull), t & 1, abort)) { ok = false; break; }
      if (t > 0 && !wait_uniform(bar(L::kDSEmpty), (t - 1) & 1, abort)) { ok = false; break; }
      tc_fence_after();
      // 16 columns at a time, the TMEM load of the next chunk in flight while
      // the current one is computed (P, 64 values, stays live throughout)
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
    // lane = column r of d: row r of dQ^T holds dQ[q0 + c][r] for the 128 c.
    // The tile leaves in four quarters of 32 query rows through two 16 KB
    // staging buffers, so that the tensor memory accelerator always has a
    // reduce in flight while the next quarter is staged.  One thread (the
    // elected lane of warp 10) issues the reduces, in the order A, B, A, B,
    // and before a buffer is written again waits until at most the other
    // buffer's reduce is still reading (bulk groups complete in order).
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
    auto wait_free = [&](int pending) {         // at most `pending` reduces still reading
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
    for (int t = 0; t < n_steps; ++t) {
      int h, q0;
      step_hq(t, h, q0);
      const int plane = b * p.H + h;
      // the four warps leave together or not at all (they meet at named
      // barriers below, which do not time out)
      if (!named_bar_and(kDqBarrier, 128, wait_uniform(bar(L::kDQFull), t & 1, abort))) break;
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
      mbar_arrive_warp(bar(L::kDQEmpty));     // the dP columns are free for dP^T(t+1)
      issue(0, q0, plane);
      issue(1, q0 + 32, plane);
      wait_free(1);
      stage(0, 0);
      issue(0, q0 + 64, plane);
      wait_free(1);
      stage(1, 1);
      issue(1, q0 + 96, plane);
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
