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
  int total_tokens;       // varlen: T
  int max_seqlen;         // varlen: bound checked against every length
  void* o;
  int o_f32;         // 1: o is fp32, 0: bf16
  float* lse;
  unsigned int* status;
};

// Tensor maps of Q, K, V for the tensor-core kernel (3-D, 128-byte swizzle).
struct TcMaps {
  CUtensorMap q, k, v;
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

// The sm_103 check of the current device and its device status word, as used
// by every entry point of fa_api.cu (returns an FA_* status code).
int checked_current_device(unsigned int** status);

}  // namespace fa
