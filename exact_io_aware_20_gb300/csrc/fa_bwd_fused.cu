// Backward pass at d = 128, dense, dQ by atomic adds: the fused kernel in
// fa_bwd_fused_kernel.cuh.
#include "fa_bwd_fused_kernel.cuh"

namespace fa {

namespace {

template <bool CAUSAL, bool BF16>
cudaError_t launch_fused(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  constexpr int D = 128, BR = 128;
  cudaError_t e;
  const size_t rows = static_cast<size_t>(pr.B) * pr.H * pr.Nq;
  // 1. D and the zeroed fp32 dQ accumulator
  int slot = timing_begin(FA_KERNEL_BWD_PRE, stream);
  constexpr int kPreRows = pre_rows_per_block<D>();
  bwd_preprocess<D, BF16><<<static_cast<unsigned>((rows + kPreRows - 1) / kPreRows),
                            kPreWarps * 32, 0, stream>>>(
      static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.delta, a.dq_acc,
      rows, pr.H, pr.Nq, a.os, a.dos, a.units);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 2. the fused kernel
  CUtensorMap tq, tk, tv, tdo;
  if ((e = make_tmap_4d(&tq, a.q, D, pr.Nq, pr.H, pr.B, a.qs, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdo, a.dout, D, pr.Nq, pr.H, pr.B, a.dos, 64, BR)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tk, a.k, D, pr.Nk, pr.Hkv, pr.B, a.ks, 64, kBC)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tv, a.v, D, pr.Nk, pr.Hkv, pr.B, a.vs, 64, kBC)) != cudaSuccess) return e;
  CUtensorMap tacc;   // the fp32 dQ accumulator [B * H][Nq][128], boxes of 32 rows
  if ((e = make_tmap_f32_3d(&tacc, a.dq_acc, D, pr.Nq, pr.B * pr.H, D, 32)) != cudaSuccess)
    return e;
  CUtensorMap tdk, tdv;   // outputs, stored as the K / V tiles are loaded
  if ((e = make_tmap_4d(&tdk, a.dk, D, pr.Nk, pr.Hkv, pr.B, a.dks, 64, kBC)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&tdv, a.dv, D, pr.Nk, pr.Hkv, pr.B, a.dvs, 64, kBC)) != cudaSuccess) return e;
  auto kern = bwd128_fused_kernel<CAUSAL, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  FusedLayout::kAlloc)) != cudaSuccess)
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
  p.with_dq = 1;
  p.mask = BlockMask{};
  p.dks = a.dks;
  p.dvs = a.dvs;
  const int n_kv_tiles = (pr.Nk + kBC - 1) / kBC;
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  // Unit order.  Heavy first (the longest key tiles of every group first)
  // when one unit holds more than a fifth of an SM's share of the work;
  // otherwise key tiles fastest, so the units of a group run together and
  // share its Q and dO in L2, with the last groups (about two units per CTA)
  // taken longest key tile first under the mask so the launch does not end
  // on one long unit.
  p.n_groups = pr.Hkv * pr.B;
  p.n_kv_tiles = n_kv_tiles;
  const long long n_units = static_cast<long long>(n_kv_tiles) * p.n_groups;
  if (n_units > (1ll << 30)) return cudaErrorInvalidValue;
  p.n_units = static_cast<int>(n_units);
  p.units = a.units;
  const int n_ctas = static_cast<int>(std::min<long long>(n_units, g_num_sms));
  p.heavy_first = 0;
  p.tail_groups = 0;
  if (CAUSAL) {
    double total = 0.0;
    for (int j = 0; j < n_kv_tiles; ++j) total += p.n_q_tiles - std::max(0, j * kBC - p.off) / BR;
    total *= static_cast<double>(p.G) * p.n_groups;
    const double longest = static_cast<double>(p.G) * p.n_q_tiles;
    p.heavy_first = longest > 0.2 * total / g_num_sms ? 1 : 0;
    if (!p.heavy_first)
      p.tail_groups = std::min(p.n_groups, (2 * n_ctas + n_kv_tiles - 1) / n_kv_tiles);
  }
  slot = timing_begin(FA_KERNEL_BWD_MAIN, stream);
  kern<<<n_ctas, kFusedThreads, FusedLayout::kAlloc, stream>>>(tq, tk, tv, tdo, tacc, tdk, tdv, p);
  timing_end(slot, stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // 3. dq = scale * accumulator, in the output dtype
  const size_t n8 = rows * D / 8;
  const unsigned blocks = static_cast<unsigned>(
      std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(g_num_sms) * 8));
  slot = timing_begin(FA_KERNEL_BWD_CONVERT, stream);
  bwd_convert_dq<D, BF16><<<blocks, 256, 0, stream>>>(a.dq_acc, static_cast<uint16_t*>(a.dq), n8,
                                                      pr.scale, pr.H, pr.Nq, a.dqs);
  timing_end(slot, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_fused(const Problem& pr, const BwdArgs& a, cudaStream_t stream) {
  if (pr.d != 128 || a.mask.ptr != nullptr || a.deterministic || a.units == nullptr)
    return cudaErrorInvalidValue;
  if (pr.causal)
    return pr.bf16 ? launch_fused<true, true>(pr, a, stream) : launch_fused<true, false>(pr, a, stream);
  return pr.bf16 ? launch_fused<false, true>(pr, a, stream) : launch_fused<false, false>(pr, a, stream);
}

}  // namespace fa
