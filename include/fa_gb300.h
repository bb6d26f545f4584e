/*
 * fa_gb300.h - C ABI of exact tiled attention for GB300 (sm_103a): forward,
 * backward, split-KV and paged decode, prefix attention and row statistics.
 *
 * What is computed.  For every query row i of every (batch, head):
 *     s_j = scale * <q_i, k_j>,     O_i = sum_j e^{s_j} v_j / sum_j e^{s_j},
 *     LSE_i = ln sum_j e^{s_j}      (natural log, fp32),
 * over the keys j visible to i (all keys; with causal, keys j <= i of the
 * same sequence).  This is the attention of "Learning FlashAttention the
 * Hard Way - Part 1" (cloudrift.ai), section "FlashAttention: Not So
 * Special", computed per row as a fold of the state (m, d, o) of sections
 * "The State" and "The Merge, and the Twist" with identity (-inf, 0, 0), in
 * the base-2 coordinates of section "Alternative Twist: Base 2"
 * (sigma = s log2 e, every exponential a 2^x).  The N x N score matrix is
 * never written to memory.  Split-KV decode and the state combine follow
 * section "Associativity is All You Need" (split-K: chunks reduced by
 * separate thread blocks, partials folded by a second kernel).
 *
 * Conventions shared by every call.
 *  - Pointers named q, k, v, o, lse, cu_seqlens*, part_* are DEVICE pointers
 *    owned by the caller; the library never allocates, frees or keeps them.
 *    Every data pointer must be 16-byte aligned and non-NULL, except that
 *    an empty problem (a zero batch, head, token or row count) returns FA_OK
 *    at once and reads no pointer (empty tensors may have NULL data).
 *  - Tensors are contiguous, row-major, without padding.  bf16 is IEEE
 *    bfloat16 (uint16 storage), f32 is IEEE binary32.
 *  - Outputs (o, lse, part_*, gradients, statistics) must not overlap any
 *    input of the same call: thread blocks write their outputs while other
 *    blocks still read the inputs, so an overlap gives undefined results.
 *  - stream is a cudaStream_t (NULL = legacy default stream).  Every call
 *    only enqueues work on it and returns: nothing synchronises, so errors
 *    raised on the device appear through fa_check_device_status.
 *  - The device current on the calling thread must be an sm_103 GPU.
 *  - scale must be finite and >= 0 (0 gives uniform weights).
 *  - Return value: FA_OK (0) or a negative FA_ERR_* code.  On
 *    FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED_ARCH nothing was launched and no
 *    output was touched.
 *  - When fa_check_device_status reports FA_ERR_DEVICE_BOUNDS or
 *    FA_ERR_DEVICE_TIMEOUT, the outputs of the calls enqueued since the last
 *    check are undefined (the split-KV first passes write the identity
 *    state (-inf, 0, 0) for a sequence whose offsets or length failed the
 *    check, but nothing else is promised).
 *  - The library looks up per-device addresses (its status word, the
 *    no-allocation scratch) once per device and keeps them for the life of
 *    the process: after cudaDeviceReset on a device, do not call the library
 *    on that device again in the same process.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK                    0
#define FA_ERR_INVALID_ARG      -1  /* NULL / misaligned pointer, bad size, bad dtype */
#define FA_ERR_UNSUPPORTED_ARCH -2  /* current device is not sm_103 */
#define FA_ERR_LAUNCH           -3  /* the CUDA launch itself failed; also a D = 64 forward whose
                                       kernel image does not start with the 168 registers per
                                       thread its warpgroup register split assumes
                                       (cudaErrorInvalidKernelImage in fa_last_cuda_error) */
#define FA_ERR_DEVICE_TIMEOUT   -4  /* a device-side pipeline wait ran past its limit */
#define FA_ERR_DEVICE_BOUNDS    -5  /* a device-side index check failed */
#define FA_ERR_DRIVER           -6  /* CUDA driver entry point or tensor-map encoding failed */
#define FA_ERR_CUDA             -7  /* another CUDA runtime error (see fa_last_cuda_error) */
#define FA_ERR_SCRATCH_CAPACITY -8  /* fa_decode_splitkv_noalloc: problem exceeds its static scratch */

#define FA_DTYPE_BF16 0
#define FA_DTYPE_F32  1

/*
 * Dense forward, bf16 in and out: the attention defined above ("FlashAttention:
 * Not So Special"), one (batch, head) per [N, D] slice.
 *   q, k, v : bf16 [B, H, N, D]
 *   o       : bf16 [B, H, N, D]           (written)
 *   lse     : f32  [B, H, N], natural log (written)
 *   B, H, N >= 1; D in {64, 128}; causal != 0 hides keys j > i.
 * Runs the tcgen05 / TMEM / TMA kernel; accumulation in fp32, the softmax
 * weights rounded to bf16 (nearest-even) before the P V product.
 * Range: a row's weights are taken against a reference maximum that may lag
 * the running maximum by up to 2^32 (base 2), so the unnormalised output
 * stays finite while N * 2^32 * max|v| is below fp32's range (|v| < 2^82 at
 * N = 2^14); the same holds for fa_fwd_ex, fa_fwd_window and fa_fwd_varlen.
 * Errors: FA_ERR_INVALID_ARG for a negative size, D not in {64, 128}, a bad
 * scale or a misaligned pointer (nothing launched); FA_ERR_UNSUPPORTED_ARCH
 * off sm_103; a device-side wait that gave up is reported later by
 * fa_check_device_status as FA_ERR_DEVICE_TIMEOUT.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int D, float scale, int causal, void* stream);

/*
 * Dense causal forward with a sliding window, bf16 in and out: query i sees
 * keys max(0, i - window + 1) .. i.  Same layouts as fa_fwd; window >= 1
 * (window >= N is plain causal attention).  Key tiles outside every row's
 * window are not read.  Hidden keys enter the fold as the identity
 * (-inf, 0, 0), the masking of "Associativity is All You Need".
 */
int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int N, int D, float scale, int window, void* stream);

/*
 * Dense forward, fp32 in and out (CUDA-core FFMA kernel, no tensor cores).
 * Same shapes and meaning as fa_fwd with f32 elements.
 */
int fa_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int D, float scale, int causal, void* stream);

/*
 * Dense forward with explicit dtypes: in_dtype is the dtype of q, k and v,
 * o_dtype that of o (FA_DTYPE_BF16 or FA_DTYPE_F32).  in_dtype BF16 runs the
 * tensor-core kernel, F32 the FFMA kernel.  o_dtype F32 with bf16 inputs
 * returns the fp32 result before the final rounding.
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int D, float scale, int causal,
              int in_dtype, int o_dtype, void* stream);

/*
 * Variable-length forward over packed sequences, bf16 in and out.
 *   q, k, v    : bf16 [total_tokens, H, D]; sequence s owns tokens
 *                [cu_seqlens[s], cu_seqlens[s+1])
 *   cu_seqlens : int32 [num_seqs + 1] DEVICE array, cu_seqlens[0] = 0,
 *                non-decreasing, cu_seqlens[num_seqs] = total_tokens
 *   max_seqlen : >= every sequence length (checked against each length)
 *   o          : bf16 [total_tokens, H, D]  (written)
 *   lse        : f32  [H, total_tokens]     (written)
 * Positions restart at 0 in every sequence (causal = keys j <= i of the same
 * sequence).  Tiles never mix sequences: rows beyond a sequence's end are
 * masked with the identity and not stored.  The launch grid is
 * H * (total_tokens / 128 + num_seqs) CTAs (sequence s owns the 128-row tile
 * slots from cu_seqlens[s] / 128 + s on); FA_ERR_INVALID_ARG if that count or
 * num_seqs * H * ceil(max_seqlen / 128) exceeds 2^31 - 1.  The device checks
 * the cu_seqlens it reads against total_tokens and max_seqlen and reports
 * FA_ERR_DEVICE_BOUNDS (through fa_check_device_status) instead of reading
 * out of range; offsets that are in range but inconsistent with
 * total_tokens (cu_seqlens[num_seqs] != total_tokens) leave rows unwritten.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int num_seqs, int total_tokens,
                  int max_seqlen, int H, int D, float scale, int causal,
                  void* stream);

/*
 * Backward of the dense bf16 forward, by recomputation: the attention weights
 * P_ij = e^{s_ij - LSE_i} are rebuilt tile by tile from Q, K and the
 * forward's LSE, never read from or written to memory ("Understanding
 * FlashAttention Pt 1: Personal Notes", Introduction: tiling + online
 * softmax + recomputation).  With dO the gradient of the loss with respect
 * to O:
 *     Delta_i = <dO_i, O_i>,   dS_ij = P_ij (<dO_i, v_j> - Delta_i),
 *     dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO.
 *   q, k, v, o, dout : bf16 [B, H, N, D]  (o and lse as fa_fwd wrote them,
 *                      same scale and causal flag)
 *   lse              : f32 [B, H, N]
 *   dq, dk, dv       : bf16 [B, H, N, D]  (written, not accumulated into)
 *   workspace        : f32, fa_bwd_workspace_bytes(B, H, N) bytes, caller-
 *                      owned DEVICE scratch (Delta is written there)
 *   B, H, N >= 1; D in {64, 128}.
 * Products on the tensor cores in bf16 with fp32 accumulation; P and dS are
 * rounded to bf16 before their products.  Three kernels in stream order
 * (Delta, dK/dV, dQ); no atomics, so the result is deterministic.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N);

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, float* workspace,
           int B, int H, int N, int D, float scale, int causal, void* stream);

/*
 * Backward of the causal sliding-window forward (fa_fwd_window): same layouts
 * and workspace as fa_bwd, query i sees keys max(0, i - window + 1) .. i
 * (window >= 1; window >= N is fa_bwd with causal = 1).  Tiles outside
 * every row's window are skipped; the edge tiles are masked.
 */
int fa_bwd_window(const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                  float* workspace, int B, int H, int N, int D, float scale, int window,
                  void* stream);

/*
 * Backward of the variable-length forward (fa_fwd_varlen) over packed
 * sequences, by the same recomputation.
 *   q, k, v, o, dout : bf16 [total_tokens, H, D]; sequence s owns tokens
 *                      [cu_seqlens[s], cu_seqlens[s+1])
 *   lse              : f32 [H, total_tokens], as fa_fwd_varlen wrote it
 *   dq, dk, dv       : bf16 [total_tokens, H, D] (written)
 *   workspace        : f32, fa_bwd_workspace_bytes(1, H, total_tokens) bytes
 *   cu_seqlens       : int32 [num_seqs + 1] DEVICE array; max_seqlen >= every
 *                      length.  Offsets that fail the device's bounds check
 *                      are reported as FA_ERR_DEVICE_BOUNDS.
 * Positions restart at 0 in every sequence; tiles never mix sequences.  The
 * tile kernels' grids are H * (total_tokens / 128 + num_seqs) CTAs, as in
 * fa_fwd_varlen (FA_ERR_INVALID_ARG past 2^31 - 1).
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                  const void* dout, const float* lse, void* dq, void* dk, void* dv,
                  float* workspace, const int* cu_seqlens, int num_seqs, int total_tokens,
                  int max_seqlen, int H, int D, float scale, int causal, void* stream);

/*
 * Row statistics as a monoid reduction: per row of a [R, C] matrix, the
 * Welford state (n, mu, M2) of "Learning FlashAttention the Hard Way -
 * Part 1", section "The Same Move: Welford's Variance" (a sample injects as
 * (1, x, 0); partials over disjoint chunks merge symmetrically with identity
 * (0, 0, 0); variance = M2 / n), reduced with the split-K + combine
 * structure of the decode above ("only the combine changes").
 *   x      : DEVICE [R, C] row-major, dtype FA_DTYPE_BF16 or FA_DTYPE_F32,
 *            aligned to its element size (16-byte aligned rows are read with
 *            16-byte loads; other rows one element at a time)
 *   mean   : f32 [R]  (written)
 *   var    : f32 [R]  population variance M2 / n (written)
 *   rstd   : f32 [R]  1 / sqrt(var + eps), the LayerNorm scale (written;
 *            may be NULL)
 *   R >= 0, C >= 1, eps finite and >= 0.
 * Accumulation in fp32; the fold order depends only on R, C and the
 * alignment of x, so results are deterministic.
 */
int fa_row_stats(const void* x, int R, int C, int dtype, float eps,
                 float* mean, float* var, float* rstd, void* stream);

/*
 * Bytes of the chunk states fa_row_stats_partials writes:
 * part_n, part_mu, part_m2, each f32 [R, num_splits].  0 for invalid sizes.
 */
size_t fa_row_stats_workspace_bytes(int R, int num_splits);

/*
 * Split-K first pass: chunk c of a row covers columns
 * [c*ceil(C/S), min(C, (c+1)*ceil(C/S))) (may be empty: state (0, 0, 0)),
 * S = num_splits in [1, 65535], R * S <= 2^31 - 1.  Writes each chunk's
 * state (n, mu, M2) to part_n / part_mu / part_m2 [R, S] (caller-owned).
 */
int fa_row_stats_partials(const void* x, int R, int C, int dtype, int num_splits,
                          float* part_n, float* part_mu, float* part_m2, void* stream);

/*
 * Split-K second pass: per row, folds its chunk states left to right, chunk
 * 0 first, with the merge
 *     n = n_a + n_b, delta = mu_b - mu_a, r = n_b / n,
 *     mu = mu_a + delta * r, M2 = (M2_a + M2_b) + ((delta * delta) * n_a) * r
 * (states with n = 0 are skipped), every operation rounded once in binary32
 * in this order, then var = M2 / n and rstd = 1 / sqrt(var + eps) with a
 * correctly rounded sqrt: bit-reproducible by any IEEE fp32 implementation
 * of the same sequence.  Outputs as fa_row_stats.
 */
int fa_row_stats_combine(const float* part_n, const float* part_mu, const float* part_m2,
                         int R, int num_splits, float eps, float* mean, float* var,
                         float* rstd, void* stream);

/*
 * Prefix attention: for every sequence b, head h and key position i of the
 * sequence, the attention of q[b, h] over keys 0..i -- the inclusive scan of
 * the keys' (m, d, o) states under the merge of "Learning FlashAttention the
 * Hard Way - Part 1" ("Why Attention's Combine Still Associates": the merge
 * is associative with identity (-inf, 0, 0), so exact attention runs as a
 * parallel prefix scan).  The last position of a sequence is its decode
 * output; with the query repeated on every row it is causal attention.
 *   q            : bf16 [B, H, D]
 *   k_cache, v_cache : bf16 [T_k, H, D], packed sequences
 *   cu_seqlens_k : int32 [B + 1] DEVICE array (checked against
 *                  total_kv_tokens on the device: FA_ERR_DEVICE_BOUNDS)
 *   o            : bf16 [T_k, H, D]  O_i of the prefix ending at token i (written)
 *   lse          : f32  [H, T_k]     natural-log LSE of that prefix (written)
 *   D in {64, 128}.  K and V are read once (one CTA per (b, h) walks its
 *   sequence in windows of 128 keys; within a window the scan has two
 *   levels: 16 keys per warp, 8 warp totals).
 */
int fa_prefix_attention(const void* q, const void* k_cache, const void* v_cache,
                        const int* cu_seqlens_k, int total_kv_tokens, int B, int H, int D,
                        float scale, void* o, float* lse, void* stream);

/*
 * Prefix attention with each row cut into num_splits chunks (1..256), for
 * few long rows: a split-KV first pass (as fa_decode_splitkv, same chunking)
 * writes every chunk's state to part_m / part_d / part_o (caller-owned,
 * fa_decode_workspace_bytes(B, H, D, num_splits) bytes), then chunk c of a
 * row scans its own keys starting from the fold of chunks 0..c-1, all
 * chunks at once.  K and V are read twice.  Outputs as fa_prefix_attention;
 * num_splits = 1 is fa_prefix_attention.
 */
int fa_prefix_attention_chunked(const void* q, const void* k_cache, const void* v_cache,
                                const int* cu_seqlens_k, int total_kv_tokens, int B, int H,
                                int D, int num_splits, float scale, float* part_m,
                                float* part_d, float* part_o, void* o, float* lse,
                                void* stream);

/*
 * Bytes of the partial-state workspace fa_decode_splitkv writes:
 * part_m and part_d f32 [B, H, num_splits], part_o f32 [B, H, num_splits, D].
 * Returns 0 for invalid sizes.
 */
size_t fa_decode_workspace_bytes(int B, int H, int D, int num_splits);

/*
 * Split-KV decode, first pass: one query token per sequence against its
 * whole KV cache, the keys cut into num_splits chunks; chunk c of a length-L
 * sequence covers keys [c*ceil(L/S), min(L, (c+1)*ceil(L/S))) (may be empty).
 *   q            : bf16 [B, H, D]
 *   k_cache      : bf16 [T_k, H, D], v_cache likewise (packed sequences)
 *   cu_seqlens_k : int32 [B + 1] DEVICE array of cache offsets (as above)
 *   total_kv_tokens : T_k, the number of rows of each cache; the device
 *                  checks every offset it reads against it and reports
 *                  FA_ERR_DEVICE_BOUNDS instead of reading out of range
 *   part_m       : f32 [B, H, S]    max of sigma = scale*log2(e)*<q,k> over the chunk
 *   part_d       : f32 [B, H, S]    sum of 2^(sigma - part_m)
 *   part_o       : f32 [B, H, S, D] sum of 2^(sigma - part_m) * v
 * An empty chunk writes the identity (-inf, 0, 0).  1 <= num_splits <= 256,
 * D in {64, 128}.  Finish with fa_combine_states(rows = B*H).
 */
int fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                      const int* cu_seqlens_k, int total_kv_tokens,
                      int B, int H, int D, int num_splits, float scale, float* part_m, float* part_d,
                      float* part_o, void* stream);

/*
 * Split-KV decode, first pass, over a paged KV cache with grouped query
 * heads.  Same outputs as fa_decode_splitkv (part_m, part_d, part_o for B*H
 * rows; finish with fa_combine_states); the chunking is described below.
 *   q           : bf16 [B, H, D]
 *   k_pages     : bf16 [num_pages, page_size, H_kv, D], v_pages likewise
 *   block_table : int32 [B, max_blocks] DEVICE array: key t of sequence b is
 *                 row t % page_size of page block_table[b][t / page_size];
 *                 page_size is a power of two
 *   seqlens     : int32 [B] DEVICE array, 0 <= seqlens[b] <= max_blocks*page_size
 *   H_kv        : KV heads, H % H_kv == 0; query head h reads KV head
 *                 h / (H / H_kv)
 * The device checks every length and page index it reads (page indices in
 * [0, num_pages)) and reports FA_ERR_DEVICE_BOUNDS through
 * fa_check_device_status instead of reading out of range; such keys are left
 * out of the fold.
 * With D = 128, 2 <= H / H_kv <= 16 and page_size >= 8 the query heads of a
 * group share one tensor-core product per 128-key tile (keys in M, the
 * group's heads in N): each KV row is read once for the whole group.  On
 * that path a chunk is made of whole tiles: its length ceil(L/S) is rounded
 * up to a multiple of 128 keys (trailing chunks may then be empty), so no
 * tile is read twice.  Other shapes fold on the CUDA cores, one query head
 * per warp, with the chunks of fa_decode_splitkv.  Either way the combined
 * output is the same attention; only the chunk boundaries of the partial
 * states differ.
 */
int fa_decode_paged_splitkv(const void* q, const void* k_pages, const void* v_pages,
                            const int* block_table, const int* seqlens, int num_pages,
                            int page_size, int max_blocks, int B, int H, int H_kv, int D,
                            int num_splits, float scale, float* part_m, float* part_d,
                            float* part_o, void* stream);

/*
 * Split-KV second pass: per row, fold chunks 0, 1, ..., num_splits-1 (in that
 * fixed order, no atomics) with the case-split merge, then O = o / d and
 * LSE = ln2 * (m + log2 d).  Every step is one IEEE binary32 operation
 * rounded to nearest, and the two exponentials are computed in software
 * (2^x by range reduction and a degree-7 Taylor polynomial; ln by
 * 2 atanh((x-1)/(x+1))), so the result is bit-reproducible on any launch and
 * equal bit for bit to a serial CPU fold that performs the same steps.
 *   part_*  : as written by fa_decode_splitkv, rows = B*H
 *   o       : [rows, D] in o_dtype (FA_DTYPE_BF16 or FA_DTYPE_F32)
 *   lse     : f32 [rows]
 * A row whose chunks are all empty gets O = 0 and LSE = -inf.
 */
int fa_combine_states(const float* part_m, const float* part_d,
                      const float* part_o, int rows, int num_splits, int D,
                      void* o, int o_dtype, float* lse, void* stream);

/*
 * Split-KV decode (both passes) without any device allocation, for callers
 * that are handed only their input and output buffers and may not allocate:
 * for example a host framework's plugin or custom-op interface that offers
 * no workspace, or a serving loop that fixes all device memory at start-up
 * because cudaMalloc can synchronise the device and fail under
 * fragmentation.  The pages have no counterpart: this is a deployment form
 * of fa_decode_splitkv + fa_combine_states, with the same arguments and
 * results (o_dtype FA_DTYPE_BF16 or FA_DTYPE_F32, lse f32 [B, H]).
 *
 * The partial states live in one static device array of the library,
 * 32 MiB per GPU that loads it (held until the process exits).  A problem
 * needing more than that, i.e. B*H*num_splits*(D+2)*4 bytes > 32 MiB, is
 * refused with FA_ERR_SCRATCH_CAPACITY before anything is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, no allocation); make that first call before
 *    capturing the stream.  The address is kept until the process exits, so
 *    this entry point must not be called on a device after cudaDeviceReset.
 *  - Nothing has to be cleared between calls: the first pass writes every
 *    state the second pass reads, the identity (-inf, 0, 0) for a sequence
 *    whose cache offsets fail the device's bounds check.
 *  - All calls on a device share the one array, so calls whose work
 *    overlaps on the GPU (different streams, no ordering) race on it.
 * The function calls no cudaMalloc, cudaFree or allocating library routine.
 */
int fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                              const int* cu_seqlens_k, int total_kv_tokens, int B,
                              int H, int D, int num_splits, float scale, void* o,
                              int o_dtype, float* lse, void* stream);

/*
 * Test hook for the failure path, not for production use: fa_fwd (bf16 out)
 * with one fault injected.  The producer leaves key tile skip_k_tile (>= 0,
 * counted from each query tile's first key tile) unrequested, as if its copy
 * had been lost, and every pipeline wait gives up after wait_limit_us
 * microseconds (1 .. 2,000,000) instead of 2 s.  A query tile that reaches
 * the missing key tile then records FA_ERR_DEVICE_TIMEOUT, lets its issued
 * copies and products complete, frees its tensor memory and exits, leaving
 * its rows of o and lse unwritten; fa_check_device_status reports the
 * timeout and clears it, and the context stays usable.  Other arguments and
 * errors as fa_fwd.
 */
int fa_fwd_fault_inject(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int N, int D, float scale, int causal, int skip_k_tile,
                        int wait_limit_us, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device that the kernels set on a failed device-side check.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_BOUNDS or FA_ERR_CUDA.
 */
int fa_check_device_status(void* stream);

/* Static English description of a status code. */
const char* fa_status_string(int code);

/* The last CUDA runtime error code seen by the library on this thread. */
int fa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
