/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library libfa_gb300.so.
 *
 * The operation ("FlashAttention-2: Faster Attention with Better Parallelism
 * and Work Partitioning", paper digest, section 3 "Target operation"):
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 *
 * for every batch b and query head h, with fp16 or bf16 inputs and fp32
 * accumulation.  Query head h reads key/value head h / (H / Hkv), so
 * Hkv == H is multi-head, 1 < Hkv < H grouped-query and Hkv == 1 multi-query
 * attention (same digest, section 4 "six checks", GQA/MQA).  The causal mask
 * keeps key k for query i when k <= i.  The forward pass also writes the row
 * logsumexp L = m + log(l) (natural log, of the scaled scores; same digest,
 * section 2 Q2, tweak 2), which the backward pass uses to rebuild the softmax
 * weights as P = exp(S - L) (section 4).  The backward pass returns the
 * gradients of sum(O o dO) (dQ, dK, dV) using D = rowsum(dO o O) (section 4
 * notation table).
 *
 * Layout (all tensors contiguous, head dimension innermost):
 *   q, o, dout, dq : [B][H][N][d]        16-bit, the `dtype` of the call
 *   k, v, dk, dv   : [B][Hkv][N][d]      16-bit
 *   lse            : [B][H][N]           fp32
 * Supported: d in {64, 128, 256}; any N >= 1 (a length that is not a multiple
 * of the tile size is handled inside the kernels); H % Hkv == 0.
 *
 * Ownership: the caller allocates every buffer (device memory) and keeps it
 * alive until the work on `stream` has finished.  The library makes no
 * allocation when called; the backward pass takes its scratch from the
 * caller's `workspace` (fa_bwd_noalloc excepted: it uses a fixed array the
 * library holds on every device that loads it).  The library caches, per
 * device, the address of its device-side error word: after cudaDeviceReset
 * the library must not be used again in the same process.
 *
 * Semantics: every call only enqueues work on `stream` (NULL is the legacy
 * default stream) and returns; nothing is synchronised.  Outputs are
 * overwritten, never accumulated into.
 *
 * Errors: each call returns an fa_status; nothing is thrown.  Argument errors
 * are found on the host before anything is enqueued.  Kernels never trap:
 * every wait on the device is bounded, and an expired wait is recorded in a
 * device-side error word that fa_get_device_status() reports and clears.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *fa_stream_t;

enum fa_dtype { FA_F16 = 0, FA_BF16 = 1 };

enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size, H % Hkv != 0, scale <= 0 */
  FA_ERR_UNSUPPORTED = 2, /* head dim, dtype or device (not sm_103) not supported */
  FA_ERR_CUDA = 3,        /* a CUDA call failed; fa_strerror(FA_ERR_CUDA) has its text */
  FA_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (from fa_get_device_status) */
  FA_ERR_WORKSPACE = 5    /* backward workspace missing, misaligned or too small for the path */
};

/*
 * Forward pass.  Writes o [B][H][N][d] (dtype) and lse [B][H][N] (fp32).
 * q, k, v, o must be 16-byte aligned device pointers, lse 4-byte aligned.
 * scale must be finite and > 0 (1/sqrt(d) is the usual value); B and H are
 * at most 65535.  causal is 0 or 1.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
           int Hkv, int N, int d, int causal, float scale, int dtype, fa_stream_t stream);

/*
 * Forward pass with separate query and key lengths (prefill with a cached
 * prefix, decode, cross-attention): q, o [B][H][Nq][d], k, v [B][Hkv][Nk][d],
 * lse [B][H][Nq].  Under the causal mask query i sees keys k <= i + Nk - Nq
 * (the mask anchored at the bottom-right corner, so the last query sees every
 * key; with Nq == Nk this is fa_fwd).  A query row that sees no key (only
 * when Nq > Nk) gets O = 0 and L = -inf.  Otherwise as fa_fwd.
 */
int fa_fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
              int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
              fa_stream_t stream);
/* (For Nq <= 64 and H > Hkv the G = H / Hkv query heads of a key/value head,
 * G * Nq consecutive rows of q in memory, are processed as one row block.) */

/*
 * Forward pass split over the key axis, for short queries and long keys
 * (decoding): each CTA covers one contiguous range of key tiles and writes a
 * normalised partial output O_s and its logsumexp L_s (fp32) to `workspace`;
 * a second kernel merges them exactly, L = ln sum_s exp(L_s) and
 * O = sum_s exp(L_s - L) O_s, so the result equals fa_fwd_qk's up to
 * rounding.  More CTAs stream K and V at once, which is what a few query rows
 * over many keys need to reach memory bandwidth.  num_splits >= 1 fixes the
 * split count (1 = no split, workspace may be NULL), 0 picks one from the
 * device's SM count.  workspace: device memory of at least
 * fa_fwd_splitkv_workspace_size(...) bytes for the same num_splits, 256-byte
 * aligned.  Otherwise as fa_fwd_qk.
 */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                   int num_splits, void *workspace, size_t workspace_bytes, fa_stream_t stream);

/* Bytes of workspace fa_fwd_splitkv needs (0 when it does not split); 0 for
 * invalid sizes as well. */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d,
                                     int num_splits);

/*
 * Bytes of device scratch fa_bwd needs for this shape: the fp32 row vector
 * D = rowsum(dO o O) [B][H][N] and an fp32 dQ accumulator [B][H][N][d]
 * (N = the query length), each rounded up to 256 bytes, then 256 bytes for
 * the work counter of the persistent d = 128 kernel.  This is enough for
 * every backward entry point.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Bytes of scratch the backward path selected by `deterministic` needs
 * (0 or 1, as in fa_bwd_qk): with deterministic = 1 dQ is written directly by
 * the query-outer kernel and only D is needed (B * H * Nq * 4 bytes, rounded
 * up to 256); with 0 D, the fp32 dQ accumulator and the work counter
 * (fa_bwd_workspace_size).
 * fa_bwd, fa_bwd_qk, fa_bwd_deterministic, fa_bwd_strided and
 * fa_bwd_blocksparse check their workspace_bytes against this size for the
 * path they run.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size_for(int B, int H, int Hkv, int Nq, int d, int deterministic);

/*
 * Backward pass of the forward above, for the same arguments.  o and lse are
 * the forward's outputs; dout is the upstream gradient dO.  Writes dq
 * [B][H][N][d], dk and dv [B][Hkv][N][d] (dtype; dk/dv summed over the query
 * heads that share each key/value head).  workspace must be a device buffer
 * of at least fa_bwd_workspace_size(...) bytes (= fa_bwd_workspace_size_for
 * with deterministic = 0), 256-byte aligned; its contents on entry do not
 * matter and are garbage on exit.
 * dQ strategy (chosen by measurement): each key tile's contribution is added
 * to an fp32 accumulator in the workspace, the pages' scheme; at d = 128 one
 * fused kernel forms all five products of a tile and hands each dQ tile to
 * the tensor memory accelerator as bulk reduce-adds.  The order of those
 * additions varies from run to run, so dQ is reproducible only up to fp32
 * rounding; fa_bwd_deterministic gives the same bits on every run.  At
 * d = 256 (without a block mask) dK and dV come from a kernel run by pairs of
 * CTAs (a thread-block cluster of two per key tile) and dQ from the
 * query-outer kernel of fa_bwd_deterministic: no atomics, every output the
 * same bits on every run, and only D of the workspace is used.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int N, int d,
           int causal, float scale, int dtype, void *workspace, size_t workspace_bytes,
           fa_stream_t stream);

/*
 * Backward pass of fa_fwd_qk: separate query and key lengths, the same mask.
 * dq [B][H][Nq][d], dk, dv [B][Hkv][Nk][d].  deterministic = 1 selects the
 * reproducible dQ path of fa_bwd_deterministic for every head dim, 0 the
 * choice of fa_bwd.  The workspace is fa_bwd_workspace_size_for(B, H, Hkv,
 * Nq, d, deterministic) bytes.
 */
int fa_bwd_qk(const void *q, const void *k, const void *v, const void *o, const float *lse,
              const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int Nq,
              int Nk, int d, int causal, float scale, int dtype, int deterministic,
              void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd with a bitwise reproducible dQ.  fa_bwd sums the dQ contributions
 * of the key/value tiles with atomic adds, whose order varies from run to run
 * (the pages use atomic adds here and do not discuss the non-determinism:
 * "FlashAttention-2: Faster Attention with Better Parallelism and Work
 * Partitioning", paper digest, section 7).  This entry point instead computes
 * dQ in a query-outer kernel that owns each query tile and walks the key
 * tiles in a fixed order (two extra products per tile: S and dP are formed
 * again); dK and dV come from the same key-outer kernel as in fa_bwd, in a
 * mode without dQ.  Same arguments and layouts as fa_bwd; the workspace
 * needs only fa_bwd_workspace_size_for(..., deterministic = 1) bytes (D);
 * every output is the same bits on every run.
 */
int fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                         int H, int Hkv, int N, int d, int causal, float scale, int dtype,
                         void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * fa_bwd for callers that cannot allocate device memory (no counterpart in
 * the paper: it exists for the caller's memory rules, not for the method).
 * Plugins whose host interface passes only inputs and outputs, and processes
 * that must not call cudaMalloc after start-up, have no way to hand fa_bwd
 * its workspace; this entry point uses a fixed array of
 * FA_BWD_NOALLOC_SCRATCH_BYTES in the library's own device memory instead
 * (held on every GPU that loads the library until exit) and allocates
 * nothing.  Arguments, outputs and semantics are those of fa_bwd without the
 * workspace.  Problems with fa_bwd_workspace_size(...) above the maximum are
 * rejected with FA_ERR_WORKSPACE before anything is enqueued.  All calls
 * share the one array: calls whose work overlaps on the GPU (two streams,
 * two threads) race and must be ordered by the caller.  The first call on a
 * device looks up the array's address with that device current, so make it
 * before any stream capture.  That address is kept for the life of the
 * process: after cudaDeviceReset (or anything else that destroys the
 * device's primary context) this entry point must not be called again in the
 * same process.  Devices with an ordinal of 64 or more are not served
 * (FA_ERR_UNSUPPORTED).
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64u << 20)
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int N,
                   int d, int causal, float scale, int dtype, fa_stream_t stream);

/*
 * Strided views (no counterpart on the pages: they let framework tensors,
 * e.g. [B][N][H][d] or a packed [B][N][3][H][d] QKV buffer, be used without
 * a copy).  Each of q, k, v, o (and dout, dq, dk, dv) is described as the
 * logical [B][heads][N][d] view with the d elements contiguous and element
 * strides
 *     element (b, h, n, c) at  base + b * batch + h * head + n * row + c.
 * Every stride must be a positive multiple of 8 elements (16 bytes) below
 * 2^39; base pointers 16-byte aligned.  The contiguous layout of fa_fwd is
 * {H * N * d, N * d, d}; [B][N][H][d] is {N * H * d, d, H * d}.  lse stays
 * contiguous [B][H][Nq] fp32.  Output views must not overlap themselves or
 * the inputs.  The results are those of fa_fwd_qk / fa_bwd_qk on the same
 * values (the same bits: only the addressing differs).
 */
typedef struct fa_strides {
  long long batch, head, row; /* element strides */
} fa_strides;

/* strides[4]: q, k, v, o.  Otherwise as fa_fwd_qk. */
int fa_fwd_strided(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                   const fa_strides *strides, fa_stream_t stream);

/* strides[8]: q, k, v, o, dout, dq, dk, dv.  Otherwise as fa_bwd_qk (the
 * workspace is fa_bwd_workspace_size_for(B, H, Hkv, Nq, d, deterministic)
 * bytes). */
int fa_bwd_strided(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int Nq,
                   int Nk, int d, int causal, float scale, int dtype, const fa_strides *strides,
                   int deterministic, void *workspace, size_t workspace_bytes,
                   fa_stream_t stream);

/*
 * Block-sparse attention ("FlashAttention: Fast and Memory-Efficient Exact
 * Attention with IO-Awareness", abstract and "Key contributions": block-sparse
 * FlashAttention computes attention only on the nonzero blocks of a given
 * block pattern).  Read here as exact attention restricted to the kept
 * blocks: query i of head h sees key k only where
 *     block_mask[hm][i / 128][k / 128] != 0      (hm = 0 if mask_heads == 1, else h)
 * and, when causal, k <= i + Nk - Nq.  The result is exact for that mask (an
 * approximation of dense attention only through the mask itself); blocks
 * whose mask byte is zero cost no loads and no products.  A query row that
 * sees no key gets O = 0 and L = -inf; a key that no query sees gets
 * dK = dV = 0.
 *
 * block_mask: device memory, bytes [mask_heads][ceil(Nq/128)][ceil(Nk/128)],
 * row-major, any alignment, read-only, nonzero = the block is computed.
 * mask_heads is 1 (one pattern for every query head) or H (one per query
 * head).  Other arguments, layouts and outputs as fa_fwd_qk / fa_bwd_qk; the
 * backward must get the forward's mask.  Limits (FA_ERR_INVALID_ARG beyond
 * them, for the per-CTA work lists): ceil(Nk / 128) <= 8192 for the forward
 * at d <= 128 (ceil(Nk / 64) <= 8192 at d = 256); for the backward,
 * (H / Hkv) * ceil(Nq / 128) <= 8192 (d = 64 and 128), (H / Hkv) *
 * ceil(Nq / 64) <= 4096 (d = 256), and with deterministic = 1 also
 * ceil(Nk / 64) <= 8192.
 */
int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                       const unsigned char *block_mask, int mask_heads, fa_stream_t stream);

int fa_bwd_blocksparse(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                       int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, int dtype,
                       const unsigned char *block_mask, int mask_heads, int deterministic,
                       void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Synchronises `stream`, then reports (and clears) the device-side error
 * word: FA_ERR_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, FA_ERR_CUDA if the stream itself failed, FA_OK otherwise.
 */
int fa_get_device_status(fa_stream_t stream);

/* Static text for a status; for FA_ERR_CUDA, the text of the last CUDA error
 * seen by this thread. */
const char *fa_strerror(int status);

/*
 * Diagnostics: per-kernel timing with CUDA events (not part of the
 * attention operation; used by the benchmark to time single kernels).
 *
 * fa_timing_enable(capacity), capacity > 0, creates `capacity` pairs of CUDA
 * events on the current device and clears the record; from then on every
 * kernel launched by fa_fwd / fa_bwd is bracketed by one pair, recorded on
 * the call's stream, until the pairs run out.  fa_timing_enable(0) stops
 * recording and destroys the events.  fa_timing_read() waits for the
 * recorded events, writes the summed elapsed milliseconds and the number of
 * timed launches per kernel kind into ms[FA_NUM_KERNEL_KINDS] and
 * launches[FA_NUM_KERNEL_KINDS], and clears the record (recording goes on).
 * Both return an fa_status.  Timing is process-wide, not per thread.
 */
/*
 * Diagnostics: checks the failure-detection path.  Launches one thread that
 * waits, through the same bounded wait the attention kernels use, on an
 * mbarrier that nothing ever completes; after limit_us microseconds (1 to
 * 2,000,000) the wait gives up and records the expiry in the device error
 * word, so the next fa_get_device_status(stream) returns FA_ERR_TIMEOUT and
 * the CUDA context stays usable.  Returns an fa_status for the launch.
 */
int fa_selftest_expired_wait(int limit_us, fa_stream_t stream);

/*
 * Diagnostics: measures the throughput of the GPU's exponential unit
 * (ex2.approx, the instruction the softmax steps use for every score), the
 * secondary bound of the attention kernels ("FlashAttention-2: Faster
 * Attention with Better Parallelism and Work Partitioning", paper digest,
 * section 2 Q1: the non-matmul work).  Runs a kernel of independent ex2
 * chains on every SM of the current device, synchronises `stream`, and
 * writes the exponentials per second (best of three timed runs) to
 * *exps_per_s.  Returns an fa_status.
 */
int fa_measure_ex2_rate(double *exps_per_s, fa_stream_t stream);

/*
 * Diagnostics: measures how many bytes per second of fp32 reduce-adds the
 * SMs of the current device push into global memory together (one CTA per
 * SM, 16 KB bulk reduce-adds of shared-memory tiles, two in flight per SM),
 * the resource that bounds the backward's dQ accumulation (dQ is
 * accumulated across key/value tiles with atomic adds: "FlashAttention-2:
 * Faster Attention with Better Parallelism and Work Partitioning", paper
 * digest, section 2 Q2, improvement 2).  scratch: device buffer of
 * scratch_bytes (at least 1 MiB, 256-byte aligned) the tiles are added into;
 * zeros are added, so its values are unchanged (a negative zero may become
 * a positive one).  Synchronises `stream`
 * and writes the best of three timed runs to *bytes_per_s.  Returns an
 * fa_status (FA_ERR_INVALID_ARG for a missing, small or misaligned buffer).
 */
int fa_measure_reduce_rate(void *scratch, size_t scratch_bytes, double *bytes_per_s,
                           fa_stream_t stream);

enum fa_kernel_kind {
  FA_KERNEL_FWD = 0,         /* the forward kernel */
  FA_KERNEL_BWD_PRE = 1,     /* backward preprocess: D and the zeroed dQ accumulator */
  FA_KERNEL_BWD_MAIN = 2,    /* backward main kernel: dK, dV and dQ accumulation */
  FA_KERNEL_BWD_CONVERT = 3, /* backward dQ conversion */
  FA_KERNEL_BWD_DQ = 4,      /* deterministic backward: query-outer dQ kernel */
  FA_NUM_KERNEL_KINDS = 5
};
int fa_timing_enable(int capacity);
int fa_timing_read(double *ms, int *launches);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
