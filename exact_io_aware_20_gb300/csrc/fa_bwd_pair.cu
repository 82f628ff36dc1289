// Backward pass at d = 256, dense: D, then dK and dV from the cluster-pair
// kernel of fa_bwd_pair_kernel.cuh, then dQ from the query-outer kernel (no
// atomics, so every output is the same bits on every run).
#include "fa_bwd_pair_kernel.cuh"

namespace fa {

namespace {

// buffers of received P^T on rank 1 (one: two more ring slots, 5% faster)
constexpr int kPairPBuf = 1;

template <bool CAUSAL, bool BF16>
cudaError_t launch_pair(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  constexpr int D = 256, BR = 128;
  cudaError_t e;
  const size_t rows = static_cast<size_t>(pr.B) * pr.H * pr.Nq;
  // 1. D = rowsum(dO o O) (no accumulator to zero)
  int slot = timing_begin(FA_KERNEL_BWD_PRE, stream);
  constexpr int kPreRows = pre_rows_per_block<D>();
  bwd_preprocess<D, BF16><<<static_cast<unsigned>((rows + kPreRows - 1) / kPreRows),
                            kPreWarps * 32, 0, stream>>>(
      static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.delta, nullptr,
      rows, pr.H, pr.Nq, a.os, a.dos, nullptr);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 2. dK, dV: one cluster of two CTAs per (key tile, kv head, batch)
  CUtensorMap tq, tk, tv, tdo;
  if ((e = make_tmap_4d(&tq, a.q, D, pr.Nq, pr.H, pr.B, a.qs, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, D, pr.Nq, pr.H, pr.B, a.dos, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tk, a.k, D, pr.Nk, pr.Hkv, pr.B, a.ks, 64, kBC)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, D, pr.Nk, pr.Hkv, pr.B, a.vs, 64, kBC)) != cudaSuccess) return e;
  using L = PairLayout<kPairPBuf>;
  auto kern = bwd256_pair_kernel<CAUSAL, BF16, kPairPBuf>;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  L::kAlloc)) != cudaSuccess)
      return e;
    attr_set = true;
  }
  BwdParams p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq_acc = nullptr;
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
  p.with_dq = 0;
  p.mask = BlockMask{};
  p.dks = a.dks;
  p.dvs = a.dvs;
  p.units = nullptr;
  p.tail_groups = 0;
  const int n_kv_tiles = (pr.Nk + kBC - 1) / kBC;
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  p.n_groups = pr.Hkv * pr.B;
  p.n_kv_tiles = n_kv_tiles;
  const long long n_units = static_cast<long long>(n_kv_tiles) * p.n_groups;
  if (n_units > (1ll << 30)) return cudaErrorInvalidValue;
  p.n_units = static_cast<int>(n_units);
  // Unit order: key tiles fastest (the units of a group run together and
  // share its Q and dO in L2), or, under the mask, the longest key tiles of
  // every group first when one unit holds more than a fifth of a pair's
  // share of the work.
  p.heavy_first = 0;
  if (CAUSAL) {
    double total = 0.0;
    for (int j = 0; j < n_kv_tiles; ++j) total += p.n_q_tiles - std::max(0, j * kBC - p.off) / BR;
    total *= static_cast<double>(p.G) * p.n_groups;
    const double longest = static_cast<double>(p.G) * p.n_q_tiles;
    p.heavy_first = longest > 0.2 * total / std::max(1, g_num_sms / 2) ? 1 : 0;
  }
  slot = timing_begin(FA_KERNEL_BWD_MAIN, stream);
  kern<<<static_cast<unsigned>(2 * n_units), kPairThreads, L::kAlloc, stream>>>(tq, tk, tv, tdo, p);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 3. dQ (query-outer, written in the output dtype)
  return launch_bwd_dq(pr, a, stream);
}

}  // namespace

cudaError_t launch_bwd_pair(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (pr.d != 256 || a.mask.ptr != nullptr) return cudaErrorInvalidValue;
  if (pr.causal)
    return pr.bf16 ? launch_pair<true, true>(pr, a, stream) : launch_pair<true, false>(pr, a, stream);
  return pr.bf16 ? launch_pair<false, true>(pr, a, stream) : launch_pair<false, false>(pr, a, stream);
}

}  // namespace fa
