// C ABI of the library (declared in include/fa_gb300.h): argument checks,
// TMA tensor-map encoding and dispatch to the kernels.  Nothing here
// allocates device memory or synchronises, except fa_check_device_status.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fa_device.cuh"
#include "fa_gb300.h"
#include "fa_internal.h"

namespace {

// Device status word: kernels OR fa::kStatus* bits into it.
__device__ unsigned int g_fa_status;

constexpr int kMaxDevices = 64;
thread_local int t_last_cuda_error = 0;

struct DeviceInfo {
  bool probed = false;
  bool sm103 = false;
  unsigned int* status = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int record(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_CUDA;
}

// Checks that the current device is sm_103 and returns its status word.
int current_device(unsigned int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record(e);
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& info = g_devices[dev];
  if (!info.probed) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess) return record(e);
    e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return record(e);
    info.sm103 = (major == 10 && minor == 3);
    if (info.sm103) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_fa_status);
      if (e != cudaSuccess) return record(e);
      info.status = static_cast<unsigned int*>(p);
    }
    info.probed = true;
  }
  if (!info.sm103) return FA_ERR_UNSUPPORTED_ARCH;
  *status = info.status;
  return FA_OK;
}

int get_encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode) return FA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    t_last_cuda_error = static_cast<int>(e);
    return FA_ERR_DRIVER;
  }
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return FA_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool good_scale(float s) { return isfinite(s) && s >= 0.f; }
float scale_log2(float s) {
  return static_cast<float>(static_cast<double>(s) * 1.4426950408889634073599);
}

// 3-D bf16 map with a (64, box1, box2) box and 128-byte swizzle.
int encode_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1, uint32_t box2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {64u, box1, box2};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_DRIVER;
}

int launched(cudaError_t e) {
  if (e == cudaSuccess) return FA_OK;
  t_last_cuda_error = static_cast<int>(e);
  return FA_ERR_LAUNCH;
}

int fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int D, float scale, int causal, int o_f32, void* stream, int window = 0,
             int skip_k_tile = -1, unsigned long long wait_limit_ns = 0) {
  if (B >= 0 && H >= 0 && N >= 0 && (B == 0 || H == 0 || N == 0) &&
      (D == 64 || D == 128) && good_scale(scale))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
    return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128) || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long mblocks = (static_cast<long long>(N) + 127) / 128;
  if (BH > 0x7fffffffLL || BH * mblocks > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (BH == 0 || N == 0) return FA_OK;
  rc = get_encoder();
  if (rc != FA_OK) return rc;
  fa::TcMaps maps{};
  const uint64_t rs = static_cast<uint64_t>(D) * 2u;
  const uint64_t hs = rs * static_cast<uint64_t>(N);
  if (encode_map(&maps.q, q, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      encode_map(&maps.k, k, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      encode_map(&maps.v, v, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      (!o_f32 && D == 128 && encode_map(&maps.o, o, D, N, BH, rs, hs, 32u, 1u) != FA_OK))
    return FA_ERR_DRIVER;
  fa::TcFwdArgs a{};
  a.o_tma = (!o_f32 && D == 128) ? 1 : 0;
  a.H = H;
  a.N = N;
  a.num_mblocks = static_cast<int>(mblocks);
  a.causal = causal ? 1 : 0;
  a.window = window;
  a.scale_log2 = scale_log2(scale);
  a.cu_seqlens = nullptr;
  a.o = o;
  a.o_f32 = o_f32;
  a.lse = lse;
  a.status = status;
  a.wait_limit_ns = wait_limit_ns;
  a.skip_k_tile = skip_k_tile;
  return launched(fa::launch_fwd_tc(maps, a, D, static_cast<int>(BH),
                                    static_cast<cudaStream_t>(stream)));
}

int fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
            int N, int D, float scale, int causal, int o_f32, void* stream) {
  if (B >= 0 && H >= 0 && N >= 0 && (B == 0 || H == 0 || N == 0) &&
      (D == 64 || D == 128) && good_scale(scale))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
    return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128) || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long mblocks = (static_cast<long long>(N) + 63) / 64;
  if (BH > 0x7fffffffLL || mblocks > 65535) return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (BH == 0 || N == 0) return FA_OK;
  fa::F32FwdArgs a{};
  a.q = static_cast<const float*>(q);
  a.k = static_cast<const float*>(k);
  a.v = static_cast<const float*>(v);
  a.o = o;
  a.o_f32 = o_f32;
  a.lse = lse;
  a.BH = static_cast<int>(BH);
  a.N = N;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale_log2(scale);
  return launched(fa::launch_fwd_f32(a, D, static_cast<cudaStream_t>(stream)));
}

int bwd_bf16(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, float* workspace, int B, int H,
             int N, int D, float scale, int causal, void* stream, int window = 0) {
  if (B >= 0 && H >= 0 && N >= 0 && (B == 0 || H == 0 || N == 0) &&
      (D == 64 || D == 128) && good_scale(scale))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned4(lse) ||
      !aligned4(workspace))
    return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128) || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  if (BH > 0x7fffffffLL || BH * tiles > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  rc = get_encoder();
  if (rc != FA_OK) return rc;
  fa::BwdMaps maps;
  const uint64_t rs = static_cast<uint64_t>(D) * 2u;
  const uint64_t hs = rs * static_cast<uint64_t>(N);
  if (encode_map(&maps.q, q, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      encode_map(&maps.k, k, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      encode_map(&maps.v, v, D, N, BH, rs, hs, 128u, 1u) != FA_OK ||
      encode_map(&maps.dout, dout, D, N, BH, rs, hs, 128u, 1u) != FA_OK)
    return FA_ERR_DRIVER;
  fa::BwdArgs a{};
  a.BH = static_cast<int>(BH);
  a.N = N;
  a.num_tiles = static_cast<int>(tiles);
  a.causal = causal ? 1 : 0;
  a.rows = BH * N;
  a.scale = scale;
  a.scale_log2 = scale_log2(scale);
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.delta = workspace;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.window = window;
  return launched(fa::launch_bwd(maps, a, D, static_cast<cudaStream_t>(stream)));
}

bool aligned_to(const void* p, unsigned int a) {
  return p && (reinterpret_cast<uintptr_t>(p) & (a - 1u)) == 0;
}

int row_stats(const void* x, int R, int C, int dtype, int S, float eps, float* part_n,
              float* part_mu, float* part_m2, float* mean, float* var, float* rstd,
              void* stream) {
  if (R < 0 || C < 1 || S < 1 || S > 65535 || (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_F32))
    return FA_ERR_INVALID_ARG;
  if (!isfinite(eps) || eps < 0.f) return FA_ERR_INVALID_ARG;
  if (R == 0) return FA_OK;
  if (!aligned_to(x, dtype == FA_DTYPE_BF16 ? 2u : 4u)) return FA_ERR_INVALID_ARG;
  if (part_n ? (!aligned4(part_n) || !aligned4(part_mu) || !aligned4(part_m2))
             : (!aligned4(mean) || !aligned4(var) || (rstd && !aligned4(rstd))))
    return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(R) * S > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  fa::RowStatsArgs a{};
  a.x = x;
  a.R = R;
  a.C = C;
  a.S = S;
  a.bf16 = dtype == FA_DTYPE_BF16 ? 1 : 0;
  a.part_n = part_n;
  a.part_mu = part_mu;
  a.part_m2 = part_m2;
  a.mean = mean;
  a.var = var;
  a.rstd = rstd;
  a.eps = eps;
  return launched(fa::launch_row_stats(a, static_cast<cudaStream_t>(stream)));
}

int bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
               const float* lse, void* dq, void* dk, void* dv, float* workspace,
               const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int H,
               int D, float scale, int causal, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H < 0 || (D != 64 && D != 128) ||
      !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  if (num_seqs == 0 || H == 0 || total_tokens == 0) return FA_OK;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned4(lse) ||
      !aligned4(workspace) || !aligned4(cu_seqlens))
    return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(num_seqs) * H;
  const long long tiles = (static_cast<long long>(max_seqlen) + 127) / 128;
  // (the tile kernels' grid: H x (total_tokens / 128 + num_seqs) tile slots)
  const long long slots = static_cast<long long>(total_tokens) / 128 + num_seqs;
  if (max_seqlen < 1 || BH * tiles > 0x7fffffffLL || slots * H > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  rc = get_encoder();
  if (rc != FA_OK) return rc;
  fa::BwdMaps maps;
  const uint64_t rs = static_cast<uint64_t>(D) * 2u;
  const uint64_t ts = rs * static_cast<uint64_t>(H);
  if (encode_map(&maps.q, q, D, H, total_tokens, rs, ts, 1u, 128u) != FA_OK ||
      encode_map(&maps.k, k, D, H, total_tokens, rs, ts, 1u, 128u) != FA_OK ||
      encode_map(&maps.v, v, D, H, total_tokens, rs, ts, 1u, 128u) != FA_OK ||
      encode_map(&maps.dout, dout, D, H, total_tokens, rs, ts, 1u, 128u) != FA_OK)
    return FA_ERR_DRIVER;
  fa::BwdArgs a{};
  a.BH = static_cast<int>(BH);
  a.N = 0;
  a.num_tiles = static_cast<int>(tiles);
  a.causal = causal ? 1 : 0;
  a.rows = static_cast<long long>(total_tokens) * H;
  a.scale = scale;
  a.scale_log2 = scale_log2(scale);
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.delta = workspace;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.cu_seqlens = cu_seqlens;
  a.total_tokens = total_tokens;
  a.H = H;
  a.max_seqlen = max_seqlen;
  return launched(fa::launch_bwd(maps, a, D, static_cast<cudaStream_t>(stream)));
}

}  // namespace

int fa::checked_current_device(unsigned int** status) { return current_device(status); }
int fa::record_cuda_error(cudaError_t e) { return record(e); }
int fa::launch_status(cudaError_t e) { return launched(e); }

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int D, float scale, int causal, void* stream) {
  return fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, causal, 0, stream);
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int D, float scale, int window, void* stream) {
  if (window < 1) return FA_ERR_INVALID_ARG;
  return fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, 1, 0, stream, window);
}

int fa_fwd_fault_inject(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int N, int D, float scale, int causal, int skip_k_tile,
                        int wait_limit_us, void* stream) {
  if (skip_k_tile < 0 || wait_limit_us < 1 || wait_limit_us > 2000000) return FA_ERR_INVALID_ARG;
  return fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, causal, 0, stream, 0, skip_k_tile,
                  static_cast<unsigned long long>(wait_limit_us) * 1000ull);
}

int fa_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int D, float scale, int causal, void* stream) {
  return fwd_f32(q, k, v, o, lse, B, H, N, D, scale, causal, 1, stream);
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int D, float scale, int causal, int in_dtype, int o_dtype, void* stream) {
  if (o_dtype != FA_DTYPE_BF16 && o_dtype != FA_DTYPE_F32) return FA_ERR_INVALID_ARG;
  const int o_f32 = o_dtype == FA_DTYPE_F32 ? 1 : 0;
  if (in_dtype == FA_DTYPE_BF16)
    return fwd_bf16(q, k, v, o, lse, B, H, N, D, scale, causal, o_f32, stream);
  if (in_dtype == FA_DTYPE_F32)
    return fwd_f32(q, k, v, o, lse, B, H, N, D, scale, causal, o_f32, stream);
  return FA_ERR_INVALID_ARG;
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int H,
                  int D, float scale, int causal, void* stream) {
  if (num_seqs >= 0 && H >= 0 && total_tokens >= 0 && max_seqlen >= 0 &&
      (num_seqs == 0 || H == 0 || total_tokens == 0) && (D == 64 || D == 128) &&
      good_scale(scale))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
      !aligned4(cu_seqlens))
    return FA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H < 0 ||
      (D != 64 && D != 128) || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  const long long SH = static_cast<long long>(num_seqs) * H;
  const long long mblocks = (static_cast<long long>(max_seqlen) + 127) / 128;
  // (the launch's grid: H x (total_tokens / 128 + num_seqs) query-tile slots)
  const long long slots = static_cast<long long>(total_tokens) / 128 + num_seqs;
  if (SH > 0x7fffffffLL || SH * mblocks > 0x7fffffffLL || slots * H > 0x7fffffffLL)
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (SH == 0 || total_tokens == 0 || max_seqlen == 0) return FA_OK;
  rc = get_encoder();
  if (rc != FA_OK) return rc;
  fa::TcMaps maps{};
  const uint64_t hs = static_cast<uint64_t>(D) * 2u;
  const uint64_t ts = hs * static_cast<uint64_t>(H);
  if (encode_map(&maps.q, q, D, H, total_tokens, hs, ts, 1u, 128u) != FA_OK ||
      encode_map(&maps.k, k, D, H, total_tokens, hs, ts, 1u, 128u) != FA_OK ||
      encode_map(&maps.v, v, D, H, total_tokens, hs, ts, 1u, 128u) != FA_OK ||
      (D == 128 && encode_map(&maps.o, o, D, H, total_tokens, hs, ts, 1u, 32u) != FA_OK))
    return FA_ERR_DRIVER;
  fa::TcFwdArgs a{};
  a.o_tma = D == 128 ? 1 : 0;
  a.H = H;
  a.N = 0;
  a.num_mblocks = static_cast<int>(mblocks);
  a.causal = causal ? 1 : 0;
  a.window = 0;
  a.scale_log2 = scale_log2(scale);
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.total_tokens = total_tokens;
  a.max_seqlen = max_seqlen;
  a.o = o;
  a.o_f32 = 0;
  a.lse = lse;
  a.status = status;
  a.wait_limit_ns = 0;
  a.skip_k_tile = -1;
  return launched(fa::launch_fwd_tc(maps, a, D, static_cast<int>(SH),
                                    static_cast<cudaStream_t>(stream)));
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 0 || H < 0 || N < 0) return 0;
  return static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(N) *
         sizeof(float);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, float* workspace, int B, int H,
           int N, int D, float scale, int causal, void* stream) {
  return bwd_bf16(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, N, D, scale, causal,
                  stream);
}

int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, float* workspace, int B, int H,
                  int N, int D, float scale, int window, void* stream) {
  if (window < 1) return FA_ERR_INVALID_ARG;
  return bwd_bf16(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, H, N, D, scale, 1, stream,
                  window);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, float* workspace,
                  const int* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int H,
                  int D, float scale, int causal, void* stream) {
  return bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, num_seqs,
                    total_tokens, max_seqlen, H, D, scale, causal, stream);
}

size_t fa_decode_workspace_bytes(int B, int H, int D, int num_splits) {
  if (B < 0 || H < 0 || (D != 64 && D != 128) || num_splits < 1 || num_splits > 256) return 0;
  const size_t rows = static_cast<size_t>(B) * H * num_splits;
  return rows * sizeof(float) * (2 + static_cast<size_t>(D));
}

int fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                      const int* cu_seqlens_k, int total_kv_tokens, int B, int H, int D,
                      int num_splits, float scale, float* part_m, float* part_d, float* part_o,
                      void* stream) {
  if (B >= 0 && H >= 0 && (B == 0 || H == 0) && (D == 64 || D == 128) && num_splits >= 1 &&
      num_splits <= 256 && good_scale(scale))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned4(cu_seqlens_k) ||
      !aligned4(part_m) || !aligned4(part_d) || !aligned16(part_o))
    return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || total_kv_tokens < 0 || (D != 64 && D != 128) || num_splits < 1 ||
      num_splits > 256 || B > 65535 || H > 8 * 65535 || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (B == 0 || H == 0) return FA_OK;
  fa::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_kv = total_kv_tokens;
  a.B = B;
  a.H = H;
  a.S = num_splits;
  a.scale_log2 = scale_log2(scale);
  a.part_m = part_m;
  a.part_d = part_d;
  a.part_o = part_o;
  a.status = status;
  return launched(fa::launch_decode_splitkv(a, D, static_cast<cudaStream_t>(stream)));
}

int fa_decode_paged_splitkv(const void* q, const void* k_pages, const void* v_pages,
                            const int* block_table, const int* seqlens, int num_pages,
                            int page_size, int max_blocks, int B, int H, int H_kv, int D,
                            int num_splits, float scale, float* part_m, float* part_d,
                            float* part_o, void* stream) {
  if (B < 0 || H < 0 || H_kv < 1 || num_pages < 0 || page_size < 1 ||
      (page_size & (page_size - 1)) != 0 || max_blocks < 0 ||
      (D != 64 && D != 128) || num_splits < 1 || num_splits > 256 || B > 65535 ||
      H > 8 * 65535 || !good_scale(scale) || (H > 0 && H % H_kv != 0))
    return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return FA_OK;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned4(block_table) ||
      !aligned4(seqlens) || !aligned4(part_m) || !aligned4(part_d) || !aligned16(part_o))
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  fa::PagedDecodeArgs a{};
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.block_table = block_table;
  a.seqlens = seqlens;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.max_blocks = max_blocks;
  a.B = B;
  a.H = H;
  a.Hkv = H_kv;
  a.S = num_splits;
  a.scale_log2 = scale_log2(scale);
  a.part_m = part_m;
  a.part_d = part_d;
  a.part_o = part_o;
  a.status = status;
  const int G = H / H_kv;
  const long long pool_rows = static_cast<long long>(num_pages) * page_size;
  if (fa::decode_paged_tc_supported(D, G, page_size) && num_pages > 0 &&
      pool_rows <= 0x7fffffffLL - 256) {
    // query heads of a group packed into one tensor-core product
    rc = get_encoder();
    if (rc != FA_OK) return rc;
    fa::PagedTcMaps maps;
    const uint64_t rs = static_cast<uint64_t>(D) * 2u;
    const uint32_t R = static_cast<uint32_t>(page_size < 128 ? page_size : 128);
    if (encode_map(&maps.q, q, D, H, B, rs, rs * H, 16u, 1u) != FA_OK ||
        encode_map(&maps.k, k_pages, D, H_kv, pool_rows, rs, rs * H_kv, 1u, R) != FA_OK ||
        encode_map(&maps.v, v_pages, D, H_kv, pool_rows, rs, rs * H_kv, 1u, R) != FA_OK)
      return FA_ERR_DRIVER;
    return launched(fa::launch_decode_paged_tc(maps, a, G, static_cast<cudaStream_t>(stream)));
  }
  return launched(fa::launch_decode_paged(a, D, static_cast<cudaStream_t>(stream)));
}

int fa_combine_states(const float* part_m, const float* part_d, const float* part_o, int rows,
                      int num_splits, int D, void* o, int o_dtype, float* lse, void* stream) {
  if (rows == 0 && num_splits >= 1 && num_splits <= 256 && (D == 64 || D == 128) &&
      (o_dtype == FA_DTYPE_BF16 || o_dtype == FA_DTYPE_F32))
    return FA_OK;  // empty problem: nothing to read or write
  if (!aligned4(part_m) || !aligned4(part_d) || !aligned16(part_o) || !aligned16(o) ||
      !aligned4(lse))
    return FA_ERR_INVALID_ARG;
  if (rows < 0 || num_splits < 1 || num_splits > 256 || (D != 64 && D != 128) ||
      (o_dtype != FA_DTYPE_BF16 && o_dtype != FA_DTYPE_F32))
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (rows == 0) return FA_OK;
  fa::CombineArgs a{};
  a.part_m = part_m;
  a.part_d = part_d;
  a.part_o = part_o;
  a.rows = rows;
  a.S = num_splits;
  a.o = o;
  a.o_f32 = o_dtype == FA_DTYPE_F32 ? 1 : 0;
  a.lse = lse;
  return launched(fa::launch_combine(a, D, static_cast<cudaStream_t>(stream)));
}

int fa_row_stats(const void* x, int R, int C, int dtype, float eps, float* mean, float* var,
                 float* rstd, void* stream) {
  return row_stats(x, R, C, dtype, 1, eps, nullptr, nullptr, nullptr, mean, var, rstd, stream);
}

size_t fa_row_stats_workspace_bytes(int R, int num_splits) {
  if (R < 0 || num_splits < 1) return 0;
  return 3u * static_cast<size_t>(R) * static_cast<size_t>(num_splits) * sizeof(float);
}

int fa_row_stats_partials(const void* x, int R, int C, int dtype, int num_splits,
                          float* part_n, float* part_mu, float* part_m2, void* stream) {
  if (R > 0 && (!part_n || !part_mu || !part_m2)) return FA_ERR_INVALID_ARG;
  return row_stats(x, R, C, dtype, num_splits, 0.f, part_n, part_mu, part_m2, nullptr, nullptr,
                   nullptr, stream);
}

int fa_row_stats_combine(const float* part_n, const float* part_mu, const float* part_m2, int R,
                         int num_splits, float eps, float* mean, float* var, float* rstd,
                         void* stream) {
  if (R < 0 || num_splits < 1 || num_splits > 65535 || !isfinite(eps) || eps < 0.f)
    return FA_ERR_INVALID_ARG;
  if (R == 0) return FA_OK;
  if (!aligned4(part_n) || !aligned4(part_mu) || !aligned4(part_m2) || !aligned4(mean) ||
      !aligned4(var) || (rstd && !aligned4(rstd)))
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  fa::RowStatsCombineArgs a{};
  a.part_n = part_n;
  a.part_mu = part_mu;
  a.part_m2 = part_m2;
  a.R = R;
  a.S = num_splits;
  a.eps = eps;
  a.mean = mean;
  a.var = var;
  a.rstd = rstd;
  return launched(fa::launch_row_stats_combine(a, static_cast<cudaStream_t>(stream)));
}

int fa_prefix_attention(const void* q, const void* k_cache, const void* v_cache,
                        const int* cu_seqlens_k, int total_kv_tokens, int B, int H, int D,
                        float scale, void* o, float* lse, void* stream) {
  return fa_prefix_attention_chunked(q, k_cache, v_cache, cu_seqlens_k, total_kv_tokens, B, H,
                                     D, 1, scale, nullptr, nullptr, nullptr, o, lse, stream);
}

int fa_prefix_attention_chunked(const void* q, const void* k_cache, const void* v_cache,
                                const int* cu_seqlens_k, int total_kv_tokens, int B, int H,
                                int D, int num_splits, float scale, float* part_m,
                                float* part_d, float* part_o, void* o, float* lse,
                                void* stream) {
  if (num_splits < 1 || num_splits > 256) return FA_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || total_kv_tokens < 0 || (D != 64 && D != 128) || !good_scale(scale))
    return FA_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return FA_OK;
  if (!aligned16(q) || !aligned4(cu_seqlens_k)) return FA_ERR_INVALID_ARG;
  if (total_kv_tokens > 0 && (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
                              !aligned4(lse)))
    return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * num_splits > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (num_splits > 1 && (!aligned4(part_m) || !aligned4(part_d) || !aligned16(part_o) ||
                         B > 65535 || H > 8 * 65535))
    return FA_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  if (num_splits > 1) {  // the chunks' states: the split-KV first pass
    fa::DecodeArgs d{};
    d.q = q;
    d.k_cache = k_cache;
    d.v_cache = v_cache;
    d.cu_seqlens_k = cu_seqlens_k;
    d.total_kv = total_kv_tokens;
    d.B = B;
    d.H = H;
    d.S = num_splits;
    d.scale_log2 = scale_log2(scale);
    d.part_m = part_m;
    d.part_d = part_d;
    d.part_o = part_o;
    d.status = status;
    rc = launched(fa::launch_decode_splitkv(d, D, static_cast<cudaStream_t>(stream)));
    if (rc != FA_OK) return rc;
  }
  fa::ScanArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_kv = total_kv_tokens;
  a.B = B;
  a.H = H;
  a.scale_log2 = scale_log2(scale);
  a.o = o;
  a.lse = lse;
  a.status = status;
  a.S = num_splits;
  a.part_m = part_m;
  a.part_d = part_d;
  a.part_o = part_o;
  return launched(fa::launch_prefix_scan(a, D, static_cast<cudaStream_t>(stream)));
}

int fa_check_device_status(void* stream) {
  unsigned int* status = nullptr;
  int rc = current_device(&status);
  if (rc != FA_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record(e);
  unsigned int word = 0;
  e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record(e);
  if (word != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return record(e);
  }
  if (word & fa::kStatusTimeout) return FA_ERR_DEVICE_TIMEOUT;
  if (word & fa::kStatusBounds) return FA_ERR_DEVICE_BOUNDS;
  return FA_OK;
}

const char* fa_status_string(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument (pointer, alignment, size, dtype or scale)";
    case FA_ERR_UNSUPPORTED_ARCH: return "current device is not an sm_103 GPU";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a device pipeline wait exceeded its limit";
    case FA_ERR_DEVICE_BOUNDS: return "a device-side bounds check failed";
    case FA_ERR_DRIVER: return "CUDA driver entry point or tensor-map encoding failed";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_SCRATCH_CAPACITY:
      return "problem needs more scratch than the no-allocation entry point's static array holds";
    default: return "unknown status code";
  }
}

int fa_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
