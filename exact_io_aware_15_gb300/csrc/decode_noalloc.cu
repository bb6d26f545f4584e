// Split-KV decode that allocates nothing: the partial (m, d, o) states of
// the first pass go to a static device array owned by the library instead of
// a caller-provided workspace.  For callers that receive only their input
// and output buffers and are not allowed to allocate device memory (plugin
// interfaces without a workspace, serving loops whose memory is fixed at
// start-up).  It reuses the decode and combine kernels unchanged.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa_gb300.h"
#include "fa_internal.h"

namespace {

// 32 MiB of partial states per GPU: B*H*S*(D+2) floats.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDev] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  In host code the array's name only
// stands for the symbol; kernels must be given this address instead.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDev) return FA_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fa::record_cuda_error(e);
    if (p == nullptr) return fa::record_cuda_error(cudaErrorInvalidSymbol);
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return FA_OK;
}

bool al16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int fa_decode_splitkv_noalloc(const void* q, const void* k_cache,
                                         const void* v_cache, const int* cu_seqlens_k,
                                         int total_kv_tokens, int B, int H, int D,
                                         int num_splits, float scale, void* o, int o_dtype,
                                         float* lse, void* stream) {
  const bool dims_ok = B >= 0 && H >= 0 && total_kv_tokens >= 0 && (D == 64 || D == 128) &&
                       num_splits >= 1 && num_splits <= 256 && B <= 65535 &&
                       H <= 8 * 65535 && isfinite(scale) && scale >= 0.f &&
                       (o_dtype == FA_DTYPE_BF16 || o_dtype == FA_DTYPE_F32);
  if (!dims_ok) return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return FA_OK;
  if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al4(cu_seqlens_k) || !al16(o) ||
      !al4(lse))
    return FA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(B) * H;
  const size_t states = rows * num_splits;
  const size_t o_bytes = states * D * sizeof(float);
  const size_t md_bytes = states * sizeof(float);
  if (o_bytes + 2 * md_bytes > kNoAllocScratchBytes) return FA_ERR_SCRATCH_CAPACITY;

  unsigned int* status = nullptr;
  int rc = fa::checked_current_device(&status);
  if (rc != FA_OK) return rc;
  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc != FA_OK) return rc;
  // [part_o | part_m | part_d]; part_o starts on the array's 256-byte boundary.
  float* part_o = static_cast<float*>(base);
  float* part_m = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + o_bytes);
  float* part_d = part_m + states;

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  fa::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_kv = total_kv_tokens;
  a.B = B;
  a.H = H;
  a.S = num_splits;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634073599);
  a.part_m = part_m;
  a.part_d = part_d;
  a.part_o = part_o;
  a.status = status;
  rc = fa::launch_status(fa::launch_decode_splitkv(a, D, st));
  if (rc != FA_OK) return rc;
  fa::CombineArgs c{};
  c.part_m = part_m;
  c.part_d = part_d;
  c.part_o = part_o;
  c.rows = static_cast<int>(rows);
  c.S = num_splits;
  c.o = o;
  c.o_f32 = o_dtype == FA_DTYPE_F32 ? 1 : 0;
  c.lse = lse;
  return fa::launch_status(fa::launch_combine(c, D, st));
}
