// Internal launch interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Arguments of the tensor-core forward (dense and varlen share the kernel).
struct TcFwdArgs {
  int H;             // heads
  int N;             // dense: sequence length (queries = keys); unused for varlen
  int num_mblocks;   // 128-row query tiles per sequence (grid.y)
  int causal;
  int window;        // > 0: causal sliding window, query i sees keys i-window+1 .. i
  float scale_log2;  // softmax scale * log2(e)
  const int* cu_seqlens;  // varlen token offsets [num_seqs + 1]; NULL when dense
  int num_seqs;           // varlen: sequences
  int total_tokens;       // varlen: T
  int max_seqlen;         // varlen: bound checked against every length
  void* o;
  int o_f32;         // 1: o is fp32, 0: bf16
  int o_tma;         // 1: bf16 O (D = 128) is stored through TcMaps::o (32-row boxes)
  float* lse;
  unsigned int* status;
  // Fault injection, used only by the tests of the timeout path (0 and -1 in
  // every other call): wait_limit_ns > 0 replaces the limit of every pipeline
  // wait, and skip_k_tile >= 0 makes the producer leave that key tile
  // unloaded, so the wait for it runs out and every role unwinds.
  unsigned long long wait_limit_ns;
  int skip_k_tile;
  // Set by launch_fwd_tc: the number of work items (query tiles x
  // (sequence, head) pairs) and whether CTAs loop over them persistently.
  int num_items;
  int persistent;
};

// Tensor maps of Q, K, V (128-row boxes) and of O (32-row boxes, used when
// TcFwdArgs::o_tma is set) for the tensor-core kernel (3-D, 128-byte swizzle).
struct TcMaps {
  CUtensorMap q, k, v, o;
};

cudaError_t launch_fwd_tc(const TcMaps& maps, const TcFwdArgs& a, int D, int grid_x,
                          cudaStream_t stream);

struct F32FwdArgs {
  const float* q;
  const float* k;
  const float* v;
  void* o;
  int o_f32;
  float* lse;
  int BH, N, causal;
  float scale_log2;
};
cudaError_t launch_fwd_f32(const F32FwdArgs& a, int D, cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* cu_seqlens_k;
  int total_kv;
  int B, H, S;
  float scale_log2;
  float* part_m;
  float* part_d;
  float* part_o;
  unsigned int* status;
};
cudaError_t launch_decode_splitkv(const DecodeArgs& a, int D, cudaStream_t stream);

struct PagedDecodeArgs {
  const void* q;         // [B, H, D]
  const void* k_pages;   // [num_pages, page_size, Hkv, D]
  const void* v_pages;
  const int* block_table;  // [B, max_blocks]
  const int* seqlens;      // [B]
  int num_pages, page_size, max_blocks;
  int B, H, Hkv, S;
  float scale_log2;
  float* part_m;
  float* part_d;
  float* part_o;
  unsigned int* status;
};
cudaError_t launch_decode_paged(const PagedDecodeArgs& a, int D, cudaStream_t stream);

// Tensor-core paged decode (decode_tc.cu): D = 128, 2 <= H / H_kv <= 16,
// page_size >= 8.  Maps: q (D, H, B) box (64, 16, 1); k and v pools
// (D, H_kv, num_pages * page_size) box (64, 1, min(page_size, 128)).
struct PagedTcMaps {
  CUtensorMap q, k, v;
};
bool decode_paged_tc_supported(int D, int G, int page_size);
cudaError_t launch_decode_paged_tc(const PagedTcMaps& maps, const PagedDecodeArgs& a, int G,
                                   cudaStream_t stream);

// Arguments of the backward kernels (dense bf16 [B, H, N, D], D = 64 or 128).
struct BwdArgs {
  int BH;            // B * H
  int N;             // sequence length (queries = keys)
  int num_tiles;     // 128-row tiles per sequence
  int causal;
  long long rows;    // BH * N
  float scale;       // softmax scale (dQ, dK epilogue)
  float scale_log2;  // scale * log2(e)
  const void* o;     // forward output, bf16
  const void* dout;  // dO, bf16
  const float* lse;  // forward log-sum-exp (natural log) [BH * N]
  float* delta;      // workspace: rowsum(dO * O) [BH * N]
  void* dq;          // bf16 outputs
  void* dk;
  void* dv;
  unsigned int* status;
  // packed sequences (NULL cu_seqlens: dense [B, H, N, D]); BH is then
  // num_seqs * H and num_tiles covers max_seqlen
  const int* cu_seqlens;
  int total_tokens;
  int H;
  int max_seqlen;
  int window;  // > 0 (dense, causal): causal sliding window
};

struct BwdMaps {
  CUtensorMap q, k, v, dout;
};

// Delta, then dK/dV, then dQ, in stream order.
cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& a, int D, cudaStream_t stream);

struct CombineArgs {
  const float* part_m;
  const float* part_d;
  const float* part_o;
  int rows, S;
  void* o;
  int o_f32;
  float* lse;
};
cudaError_t launch_combine(const CombineArgs& a, int D, cudaStream_t stream);

// Per-row Welford statistics of a [R, C] matrix (rowstats.cu).
struct RowStatsArgs {
  const void* x;
  int R, C, S;       // rows, columns, column chunks per row
  int bf16;          // 1: bf16 elements, 0: fp32
  float* part_n;     // chunk states [R, S] (NULL: S == 1, write the statistics)
  float* part_mu;
  float* part_m2;
  float* mean;       // [R]
  float* var;        // [R], population variance
  float* rstd;       // [R], 1 / sqrt(var + eps); may be NULL
  float eps;
};
cudaError_t launch_row_stats(const RowStatsArgs& a, cudaStream_t stream);

struct RowStatsCombineArgs {
  const float* part_n;
  const float* part_mu;
  const float* part_m2;
  int R, S;
  float eps;
  float* mean;
  float* var;
  float* rstd;
};
cudaError_t launch_row_stats_combine(const RowStatsCombineArgs& a, cudaStream_t stream);

// Prefix attention (scan.cu): every prefix of every sequence's keys.
struct ScanArgs {
  const void* q;        // [B, H, D] bf16
  const void* k_cache;  // [T, H, D] bf16, packed sequences
  const void* v_cache;
  const int* cu_seqlens_k;  // [B + 1]
  int total_kv;             // T
  int B, H;
  float scale_log2;
  void* o;                  // [T, H, D] bf16
  float* lse;               // [H, T]
  unsigned int* status;
  int S;                    // chunks per row (1: one CTA walks the whole row)
  const float* part_m;      // S > 1: the chunks' split-KV states [B, H, S] ...
  const float* part_d;
  const float* part_o;      // ... and [B, H, S, D]
};
cudaError_t launch_prefix_scan(const ScanArgs& a, int D, cudaStream_t stream);

// The sm_103 check of the current device and its device status word, as used
// by every entry point of fa_api.cu (returns an FA_* status code).
int checked_current_device(unsigned int** status);

// Remember a CUDA runtime error for fa_last_cuda_error() on this thread and
// return FA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// FA_OK for cudaSuccess; otherwise remember the error for fa_last_cuda_error()
// and return FA_ERR_LAUNCH (the status of a kernel launch).
int launch_status(cudaError_t e);

}  // namespace fa
