// Backward pass at d = 256, dense: dK and dV of a 128-key tile formed by a
// pair of CTAs (a thread-block cluster of two), each holding one of the two
// accumulators in TMEM; dQ comes from the query-outer kernel of
// fa_bwd_dq_kernel.cuh (no atomics).
//
// Method ("FlashAttention-2: Faster Attention with Better Parallelism and
// Work Partitioning", paper digest):
//  - section 2 Q2, improvement 2 (backward): the outer loop runs over
//    key/value tiles and dK, dV stay on chip for the whole loop;
//  - section 3 "FLOPs": the products S = Q K^T, dP = dO V^T, dV += P^T dO,
//    dK += dS^T Q with dS = P o (dP - D) (dQ += dS K is the dQ kernel's);
//  - section 4 "logsumexp fusion": P = exp(S - L) from the saved L;
//  - section 4 "six checks", GQA/MQA: a unit walks every query head of its
//    key/value head, so the dK and dV sums over the group stay in TMEM.
//
// At d = 256 the dK and dV accumulators of 128 keys fill all 512 TMEM
// columns of one SM.  The pair splits each step's products (128 query rows)
// so that no product is formed twice:
//   rank 0: S^T = K Q^T, P^T = exp(S^T * scale - L) (masked), dV += P^T dO;
//   rank 1: dP^T = V dO^T, dS^T = P^T o (dP^T - D), dK += dS^T Q;
// rank 0 sends P^T (16-bit, 32 KB a step) to rank 1's shared memory through
// distributed shared memory, and nothing goes back but a release of the
// buffer.  The exchange runs warp to warp: softmax warp w of rank 0 writes
// the rows (its 32 keys, its 64 queries) that dS warp w of rank 1 reads into
// its own copy of the buffer, and one lane sends them as a single 4 KB bulk
// copy that completes on that warp's own barrier in rank 1 (16-byte stores
// into the other CTA's shared memory, ~17 B/clk per SM, held the warps for
// the whole ~1,900 cycles of a step's 32 KB; the bulk copy moves them no
// faster, but the warps write ~80 B/clk locally and go on to the next step);
// the receiver takes its rows into registers as soon as they have arrived
// and releases them at once.  Every
// product is an M = 128, N >= 128 tcgen05.mma (full rate), and the two CTAs
// carry the same tensor work per step.
// Each CTA holds its stationary tile (K or V, 64 KB) and a ring of
// 64-column chunks through which both of its streamed operands pass in the
// order they are read: the score operand (Q or dO) of step t, then the
// accumulator operand (dO or Q) of step t - 1, and so on; rank 1 also holds
// PBUF buffers of received P^T and rank 0 its own copy of them, from which
// the bulk copies read.  With one buffer the ring has eight slots (128 KB,
// two products ahead): rank 0 writes step t + 1's rows once rank 1 has read
// step t's, which it does first thing, and the two extra slots measured 5%
// faster than a second buffer.
// TMEM: accumulator (256 columns, two 128-column halves of d) | two score
// buffers (128 columns; the 16-bit P^T or dS^T is written over the first 32
// columns of each 64-column half and read there as the A operand).
// Issue order (both CTAs): score(t), acc(t-1), score(t+1), acc(t), ...
// Warps (10): 0 TMA producer; 1 MMA issuer; 2..9 softmax (rank 0) or dS
// (rank 1), a key row per thread, warps w and w + 4 sharing a TMEM lane
// quarter and splitting the 128 query columns in halves.
// dS uses the 16-bit P^T that rank 1 receives (the weights dV multiplies
// with), not the fp32 values.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

namespace {

constexpr int kPairThreads = 320;

// PBUF: buffers of received P^T on rank 1 (1 or 2), each also held by rank
// 0 as the source of its bulk copies; the rest of each CTA's shared memory
// is ring.
template <int PBUF>
struct PairLayout {
  static constexpr int kChunk = 128 * 64 * 2;      // [128 rows][64 cols] 16-bit, 128-byte swizzle
  static constexpr int kRing1 = 10 - 2 * PBUF;     // ring slots of rank 1
  static constexpr int kRing0 = kRing1;            // ring slots of rank 0
  static constexpr int kStatOff = 0;               // K (rank 0) or V (rank 1), 4 chunks of d
  static constexpr int kRingOff = 4 * kChunk;      // the operand ring
  static constexpr int kPOff = kRingOff + kRing1 * kChunk;  // P^T, PBUF x 2 query halves (rank 1
                                                            // receives, rank 0 stages)
  static constexpr int kLDOff = kRingOff + 10 * kChunk;     // [2 halves][3 steps][64]: -L*log2e or -D
  static constexpr int kBarOff = kLDOff + 2 * 3 * 64 * 4;
  // IN_FULL / OUT_FREE: [softmax / dS warp (warp - 2)][P^T buffer, stride 2]
  static constexpr int kStatFull = 0, kRingFull = 1, kRingEmpty = kRingFull + kRing0,
                       kSFull = kRingEmpty + kRing0, kPFull = kSFull + 2, kInFull = kPFull + 2,
                       kOutFree = kInFull + 16, kFinal = kOutFree + 16, kDrain = kFinal + 1,
                       kNumBars = kDrain + 1;
  static constexpr uint32_t kRowsBytes = 32 * 128;   // one warp's rows of one query half
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;   // TMEM base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  // The whole opt-in maximum; the kernel checks that the layout fits behind
  // the 1024-byte-aligned base it gets.
  static constexpr int kAlloc = 227 * 1024;
  static constexpr uint32_t kTAcc = 0, kTScore = 256, kTmemCols = 512;
  static_assert(kBytes + 1008 <= kAlloc, "shared memory budget (any 16-byte-aligned base)");
  static_assert(kRing0 % 2 == 0 && kRing1 % 2 == 0, "operand chunks come in aligned pairs");
  static_assert(kPOff + PBUF * 2 * kChunk <= kLDOff, "rank 1 layout");
  static_assert(kRingOff + kRing0 * kChunk <= kPOff, "rank 0 keeps its own copy of the P^T buffers");
  static_assert(PBUF == 1 || PBUF == 2, "P^T buffers");
};

template <bool CAUSAL, bool BF16, int PBUF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
bwd256_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = PairLayout<PBUF>;
  constexpr int BR = 128;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  // (the same outcome in both CTAs of the cluster: same kernel, same base)
  if (sbase + L::kBytes > raw + L::kAlloc) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemBase);
    return;
  }
  uint8_t* smem = smem_raw + (sbase - raw);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * i; };
  // the dQ kernel that follows (launched as this grid's programmatic
  // dependent; it reads none of this kernel's results) may start filling
  // the SMs this grid's last wave leaves idle
  grid_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  // unit = (key tile, kv head, batch), in the host's order
  const int u = static_cast<int>(blockIdx.x >> 1);
  int jt, grp;
  if (p.heavy_first) {
    jt = u / p.n_groups;
    grp = u % p.n_groups;
  } else {
    jt = u % p.n_kv_tiles;
    grp = u / p.n_kv_tiles;
  }
  const int kh = grp % p.Hkv, b = grp / p.Hkv;
  const int kv0 = jt * kBC;
  // steps: the query tiles from the last down to the first that sees key
  // kv0, the G heads of the group innermost, each unit starting jt tiles into
  // that cycle so that the units of a group do not all ask for the same Q and
  // dO tiles at once (1% faster at head256; the order is fixed, so dK and dV
  // are the same bits on every run)
  const int i0 = CAUSAL ? max(0, kv0 - p.off) / BR : 0;
  const int n_i = max(0, p.n_q_tiles - i0);
  const int n = p.G * n_i;
  auto step_hq = [&](int t, int& h, int& q0) {
    h = kh * p.G + t % p.G;
    q0 = (p.n_q_tiles - 1 - (t / p.G + jt) % max(1, n_i)) * BR;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kStatFull), 1);
    for (int c = 0; c < L::kRing0; ++c) {
      mbar_init(bar(L::kRingFull + c), 1);
      mbar_init(bar(L::kRingEmpty + c), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kSFull + s), 1);
      mbar_init(bar(L::kPFull + s), 8);      // one arrival per softmax / dS warp
    }
    for (int c = 0; c < 16; ++c) {
      mbar_init(bar(L::kInFull + c), 1);     // rank 1: the receiver's expect_tx + the bytes
      mbar_init(bar(L::kOutFree + c), 32);   // rank 0: the 32 readers of the rows
    }
    mbar_init(bar(L::kFinal), 1);
    mbar_init(bar(L::kDrain), 1);
    // rank 1 expects the rows of steps 0 and 1 before the cluster meets, so
    // no rows can land ahead of their expect_tx (later steps' are expected
    // before the buffer is released)
    if (rank == 1) {
      for (int c = 0; c < 16; ++c)
        if ((c & 1) < min(n, PBUF)) mbar_arrive_expect_tx(bar(L::kInFull + c), L::kRowsBytes);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before anything arrives on them
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tAcc = tmem + L::kTAcc, tScore = tmem + L::kTScore;
  const int ring = rank == 0 ? L::kRing0 : L::kRing1;   // ring slots of this CTA

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The ring takes the 64-column chunks of both streamed operands in the
    // order the MMA warp reads them: the score operand of step t (Q or dO),
    // then the accumulator operand of step t - 1 (dO or Q), and so on.
    const CUtensorMap* tm_stat = rank == 0 ? &tm_k : &tm_v;
    const CUtensorMap* tm_a = rank == 0 ? &tm_q : &tm_do;   // score operand
    const CUtensorMap* tm_b = rank == 0 ? &tm_do : &tm_q;   // accumulator operand
    if (elect_one()) {
      tma_prefetch_desc(tm_stat);
      tma_prefetch_desc(tm_a);
      tma_prefetch_desc(tm_b);
      mbar_arrive_expect_tx(bar(L::kStatFull), 4 * L::kChunk);
      #pragma unroll
      for (int c = 0; c < 4; ++c)
        tma_load_4d(sbase + L::kStatOff + c * L::kChunk, tm_stat, bar(L::kStatFull), c * 64, kv0,
                    kh, b);
    }
    __syncwarp();
    int slot = 0, lap = 0, ci = 0;   // next ring slot, times round the ring, chunks issued
    // the four chunks of d of step t's tile of `map`
    auto load_tile = [&](const CUtensorMap* map, int t) -> bool {
      int h, q0;
      step_hq(t, h, q0);
      #pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        if (lap > 0 && !wait_uniform(bar(L::kRingEmpty + slot), (lap - 1) & 1, abort)) return false;
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(L::kRingFull + slot), L::kChunk);
          tma_load_4d(sbase + L::kRingOff + slot * L::kChunk, map, bar(L::kRingFull + slot), c * 64,
                      q0, h, b);
        }
        __syncwarp();
        ++ci;
        if (++slot == ring) {
          slot = 0;
          ++lap;
        }
      }
      return true;
    };
    bool ok = true;
    for (int t = 0; ok && t < n; ++t) {
      ok = load_tile(tm_a, t);
      if (ok && t >= 1) ok = load_tile(tm_b, t - 1);
    }
    if (ok && n > 0) load_tile(tm_b, n - 1);
    // nothing may land in shared memory after the CTA has exited
    drain_wait(bar(L::kStatFull), 0);
    for (int i = max(0, ci - ring); i < ci; ++i)
      drain_wait(bar(L::kRingFull + i % ring), (i / ring) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdS = idesc_f16(kBC, BR, BF16 ? 1 : 0, 0, 0);    // S^T, dP^T
    constexpr uint32_t kIdA = idesc_f16(kBC, 128, BF16 ? 1 : 0, 0, 1);   // dV, dK halves
    const uint64_t stat_k = smem_desc_sw128(sbase + L::kStatOff, 16, 1024);
    const uint64_t ring_k = smem_desc_sw128(sbase + L::kRingOff, 16, 1024);
    // an accumulator operand pair of chunks as B with N = 128 columns of d
    const uint64_t ring_mn = smem_desc_sw128(sbase + L::kRingOff, L::kChunk, 1024);
    int slot = 0, lap = 0;   // next ring slot to read, times round the ring
    auto advance = [&](int k) {
      slot += k;
      if (slot == ring) {
        slot = 0;
        ++lap;
      }
    };
    // score(t) = stationary x (its score operand)^T into buffer t & 1; each
    // ring slot is released as soon as its four products have completed
    auto issue_score = [&](int t) -> bool {
      const uint32_t d = tScore + (t & 1) * 128;
      #pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        if (!wait_uniform(bar(L::kRingFull + slot), lap & 1, abort)) return false;
        tc_fence_after();
        #pragma unroll
        for (int w = 0; w < 4; ++w)
          mma_ss(d, desc_add(stat_k, c * L::kChunk + w * 32),
                 desc_add(ring_k, slot * L::kChunk + w * 32), kIdS, (c | w) ? 1u : 0u);
        mma_commit(bar(L::kRingEmpty + slot));
        advance(1);
      }
      mma_commit(bar(L::kSFull + (t & 1)));
      return true;
    };
    // acc += (16-bit P^T or dS^T of step t, from TMEM) x (dO or Q of step t),
    // one 128-column half of d (two ring chunks, an aligned pair) at a time
    auto issue_acc = [&](int t) -> bool {
      if (!wait_uniform(bar(L::kPFull + (t & 1)), (t >> 1) & 1, abort)) return false;
      const uint32_t a = tScore + (t & 1) * 128;
      #pragma unroll 1
      for (int dh = 0; dh < 2; ++dh) {
        // (an even slot: both chunks of the pair are in the same lap)
        if (!wait_uniform(bar(L::kRingFull + slot), lap & 1, abort) ||
            !wait_uniform(bar(L::kRingFull + slot + 1), lap & 1, abort))
          return false;
        tc_fence_after();
        #pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tAcc + 128 * dh, a + (kk >> 2) * 64 + (kk & 3) * 8,
                 desc_add(ring_mn, slot * L::kChunk + kk * 2048), kIdA, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::kRingEmpty + slot));
        mma_commit(bar(L::kRingEmpty + slot + 1));
        advance(2);
      }
      return true;
    };
    bool ok = wait_uniform(bar(L::kStatFull), 0, abort);
    for (int t = 0; ok && t < n; ++t) {
      if (!issue_score(t)) ok = false;
      else if (t >= 1 && !issue_acc(t - 1)) ok = false;
    }
    if (ok && n > 0) issue_acc(n - 1);
    mma_commit(bar(L::kFinal));
    mma_commit(bar(L::kDrain));
    drain_wait(bar(L::kDrain), 0);
  } else {
    // ------------------------------------------------------------ softmax (rank 0) / dS (rank 1)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;            // query columns [64 half, 64 half + 64)
    const int r = quarter * 32 + lane;           // key row within the tile
    const int kv = kv0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // Step t's P^T goes to buffer t & 1 of rank 1: this warp's rows, row r
    // of this query half (an address in rank 1's shared memory) ...
    const uint32_t p_row0 = (rank == 0 ? mapa_shared(sbase + L::kPOff, peer) : sbase + L::kPOff) +
                            half * L::kChunk + r * 128;
    auto p_row = [&](int pb) { return p_row0 + pb * (2 * L::kChunk); };
    // ... and on rank 0 the same row of its own copy of that buffer, where
    // the row is written before the warp's rows go out as one bulk copy
    auto p_stage = [&](int pb) {
      return sbase + L::kPOff + pb * (2 * L::kChunk) + half * L::kChunk + r * 128;
    };
    // ... and the warp's channel for that buffer: rank 1's IN_FULL (where
    // the sender's bytes land) and rank 0's OUT_FREE (where the reader
    // releases the rows)
    const int ch = 2 * (warp - 2);
    const uint32_t in_full0 =
        rank == 0 ? mapa_shared(bar(L::kInFull + ch), peer) : bar(L::kInFull + ch);
    const uint32_t out_free0 =
        rank == 0 ? bar(L::kOutFree + ch) : mapa_shared(bar(L::kOutFree + ch), peer);
    auto in_full = [&](int pb) { return in_full0 + 8u * pb; };
    auto out_free = [&](int pb) { return out_free0 + 8u * pb; };
    // -L*log2(e) (rank 0) or -D (rank 1) of this half's 64 query columns, one
    // buffer per step in three: a warp writes step t + 1's values at the end
    // of step t, when every warp is past step t - 2 (score(t) was issued
    // after the P_FULL of step t - 2); the four warps of a half write the
    // same values
    float* ld_base = reinterpret_cast<float*>(smem + L::kLDOff) + half * (3 * 64);
    const float* ld_src = rank == 0 ? p.lse : p.delta;
    float lv[2];
    bool lvv[2];
    auto load_ld = [&](int t) {
      int h, q0;
      step_hq(t, h, q0);
      const size_t base = (static_cast<size_t>(b) * p.H + h) * p.Nq;
      #pragma unroll
      for (int v = 0; v < 2; ++v) {
        const int q = q0 + 64 * half + lane + 32 * v;
        lvv[v] = q < p.Nq;
        lv[v] = __ldg(ld_src + base + (lvv[v] ? q : 0));
      }
    };
    auto store_ld = [&](int t) {
      float* dst = ld_base + (t % 3) * 64;
      #pragma unroll
      for (int v = 0; v < 2; ++v)
        dst[lane + 32 * v] = rank == 0 ? (lvv[v] ? -lv[v] * kLog2e : -INFINITY)
                                       : (lvv[v] ? -lv[v] : 0.f);
    };
    if (n > 0) {
      load_ld(0);
      store_ld(0);
    }
    __syncwarp();
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const float* sv = ld_base + (t % 3) * 64;
      // (rank 1 issues the next step's loads after its release arrive below,
      // which would otherwise wait for them)
      if (rank == 0 && t + 1 < n) load_ld(t + 1);
      const uint32_t src = tScore + (t & 1) * 128 + lane_off + 64 * half;
      uint32_t pk[32];   // 16-bit pairs of P^T, query columns 2 j and 2 j + 1 of this half
      if (rank == 0) {
        if (!wait_uniform(bar(L::kSFull + (t & 1)), (t >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        int h, q0;
        step_hq(t, h, q0);
        const bool kv_out = kv >= p.Nk;
        const bool diag = CAUSAL && (q0 + p.off < kv0 + kBC);
        const bool masked = __any_sync(0xffffffffu, kv_out || diag);
        const f2 cs = {p.scale_log2, p.scale_log2};
        const int qc0 = q0 + 64 * half;
        auto p_chunk = [&](const uint32_t (&sr)[32], int c0) {
          float P[32];
          #pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(sv + c0 + c);
            const f2 a0 = ffma2(f2{__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])}, cs,
                                f2{l4.x, l4.y});
            const f2 a1 = ffma2(f2{__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])}, cs,
                                f2{l4.z, l4.w});
            P[c] = ex2_approx(a0.x);
            P[c + 1] = ex2_approx(a0.y);
            P[c + 2] = ex2_approx(a1.x);
            P[c + 3] = ex2_approx(a1.y);
          }
          if (masked) {
            // queries qc0 + c0 + c with c < z see no key kv (z = 32: the key
            // is past Nk)
            const int z = kv_out ? 32 : (diag ? min(32, kv - p.off - qc0 - c0) : 0);
            #pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < z) P[c] = 0.f;
          }
          #pragma unroll
          for (int c = 0; c < 16; ++c) pk[c0 / 2 + c] = pack2<BF16>(P[2 * c], P[2 * c + 1]);
          // P^T over the first 32 columns of this half, already read
          tmem_st16(src + c0 / 2, &pk[c0 / 2]);
        };
        {
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
        // P^T is in TMEM: this CTA's dV may start before the rows below have
        // left (their stores take longer than the exponentials)
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(L::kPFull + (t & 1)));
        // row r of this half of P^T to rank 1's buffer t % PBUF, once rank 1
        // has read step t - PBUF's from it
        // rank 1 has read step t - PBUF's rows, so the bulk copy that took
        // them there has also finished reading this CTA's copy of buffer pb
        const int pb = t % PBUF, use = t / PBUF;
        if (t >= PBUF && !wait_uniform<true>(out_free(pb), (use - 1) & 1, abort)) {
          ok = false;
          break;
        }
        #pragma unroll
        for (int v = 0; v < 8; ++v)
          st_shared_v4(p_stage(pb) + ((v ^ (r & 7)) * 16), pk[4 * v], pk[4 * v + 1],
                       pk[4 * v + 2], pk[4 * v + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        // the warp's 32 rows are one 4 KB block in both CTAs
        if (lane == 0) bulk_copy_to_cluster(p_row(pb), p_stage(pb), L::kRowsBytes, in_full(pb));
        __syncwarp();
      } else {
        // row r of this half of P^T, sent by rank 0: into registers and the
        // rows released before this step's dP^T is waited for
        const int pb = t % PBUF, use = t / PBUF;
        if (!wait_uniform<true>(in_full(pb), use & 1, abort)) { ok = false; break; }
        #pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 w4 = ld_shared_v4(p_row(pb) + ((v ^ (r & 7)) * 16));
          pk[4 * v] = w4.x;
          pk[4 * v + 1] = w4.y;
          pk[4 * v + 2] = w4.z;
          pk[4 * v + 3] = w4.w;
        }
        // step t + PBUF's rows are expected before these are released, so
        // they cannot land ahead of their expect_tx
        if (t + PBUF < n) {
          __syncwarp();
          if (elect_one()) mbar_arrive_expect_tx(in_full(pb), L::kRowsBytes);
          __syncwarp();
        }
        mbar_arrive_remote(out_free(pb));
        if (t + 1 < n) load_ld(t + 1);
        if (!wait_uniform(bar(L::kSFull + (t & 1)), (t >> 1) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        uint32_t da[32], db[32];
        tmem_ld32(src, da);
        tmem_ld32(src + 32, db);
        tmem_ld_wait();
        reg_fence(da);
        reg_fence(db);
        // dS^T = P^T o (dP^T - D) over the first 32 columns of this half
        uint32_t w[32];
        #pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float2 pa = unpack2<BF16>(pk[c]);
          const float2 pb = unpack2<BF16>(pk[16 + c]);
          const f2 da2 = fadd2(f2{__uint_as_float(da[2 * c]), __uint_as_float(da[2 * c + 1])},
                               f2{sv[2 * c], sv[2 * c + 1]});
          const f2 db2 = fadd2(f2{__uint_as_float(db[2 * c]), __uint_as_float(db[2 * c + 1])},
                               f2{sv[32 + 2 * c], sv[32 + 2 * c + 1]});
          const f2 dsa = fmul2(f2{pa.x, pa.y}, da2);
          const f2 dsb = fmul2(f2{pb.x, pb.y}, db2);
          w[c] = pack2<BF16>(dsa.x, dsa.y);
          w[16 + c] = pack2<BF16>(dsb.x, dsb.y);
        }
        tmem_st16(src, &w[0]);
        tmem_st16(src + 16, &w[16]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(L::kPFull + (t & 1)));
      }
      if (t + 1 < n) {
        store_ld(t + 1);
        __syncwarp();
      }
    }
    // ------------------------------------------------------------ dV (rank 0), dK (rank 1)
    if (ok && wait_uniform(bar(L::kFinal), 0, abort)) {
      tc_fence_after();
      const bool in_range = kv < p.Nk;
      const long long kvr = in_range ? kv : 0;
      uint16_t* row = rank == 0 ? p.dv + b * p.dvs.b + kh * p.dvs.h + kvr * p.dvs.n
                                : p.dk + b * p.dks.b + kh * p.dks.h + kvr * p.dks.n;
      uint4* out = reinterpret_cast<uint4*>(row + 128 * half);
      const float mul = rank == 0 ? 1.f : p.scale;
      // a unit with no step never wrote its accumulator
      const uint32_t live = n > 0 ? 0xffffffffu : 0u;
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t a[32];
        tmem_ld32(tAcc + lane_off + 128 * half + 32 * j, a);
        tmem_ld_wait();
        reg_fence(a);
        uint32_t o[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c)
          o[c] = pack2<BF16>(__uint_as_float(a[2 * c] & live) * mul,
                             __uint_as_float(a[2 * c + 1] & live) * mul);
        if (in_range) {
          #pragma unroll
          for (int i = 0; i < 4; ++i)
            out[4 * j + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still write to its shared memory
  cluster_sync();
  tc_fence_after();
  if (threadIdx.x == 0 && *abort == 2) atomicOr(p.err, kErrTimeout);
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace

}  // namespace fa
