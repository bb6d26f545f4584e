// Split-KV second pass: fold the per-chunk states of every row.
//
// "Learning FlashAttention the Hard Way - Part 1": split-K folds the partials
// "in a small second kernel" ("Associativity is All You Need"), with the merge
// of "The Merge, and the Twist" written as its case split so that the
// exponent is never positive, in base 2 ("Alternative Twist: Base 2"); the
// row is read off as o / d ("The State").
//
// One warp per row; lane l owns D/32 consecutive columns, so each chunk's
// partial o row is one coalesced 512-byte (D = 128) read.  A warp loads the
// states of 16 chunks at a time before folding them, so a row waits for
// memory once per 16 chunks rather than once per chunk, and the 16 merge
// factors of a batch are computed at once, one per lane.  Chunks are folded
// in index order 0, 1, ..., S-1 starting from the identity, with no atomics,
// so the result does not depend on the launch.  Every arithmetic step is a
// single IEEE binary32 operation with round-to-nearest (the __f*_rn
// intrinsics keep the compiler from fusing or reassociating), and the two
// transcendental steps are computed here rather than by the special-function
// unit:
//   2^x  : x = n + f with n = rint(x), |f| <= 1/2 (exact), then the Taylor
//          polynomial of 2^f = sum_k (f ln 2)^k / k! through k = 7, in Horner
//          form, times 2^n assembled from exponent bits; x < -126 gives 0.
//   ln d : d = 2^e x with x in [1/sqrt2, sqrt2], ln x = 2 atanh(t) with
//          t = (x - 1)/(x + 1) and atanh(t) = t (1 + t^2/3 + ... + t^10/11).
// A serial CPU fold that performs the same operations therefore reproduces the
// output bits exactly.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"

namespace fa {
namespace {

// Taylor coefficients (ln 2)^k / k!, formed in double by the recurrence
// c_k = c_{k-1} * ln2 / k and rounded to binary32 once.
constexpr double kLn2d = 0.693147180559945309417232121458;
constexpr double taylor_coef(int k) { return k == 0 ? 1.0 : taylor_coef(k - 1) * kLn2d / k; }
constexpr float kE0 = 1.0f;
constexpr float kE1 = static_cast<float>(taylor_coef(1));
constexpr float kE2 = static_cast<float>(taylor_coef(2));
constexpr float kE3 = static_cast<float>(taylor_coef(3));
constexpr float kE4 = static_cast<float>(taylor_coef(4));
constexpr float kE5 = static_cast<float>(taylor_coef(5));
constexpr float kE6 = static_cast<float>(taylor_coef(6));
constexpr float kE7 = static_cast<float>(taylor_coef(7));
// atanh series coefficients 1/(2j+1).
constexpr float kA0 = 1.0f;
constexpr float kA1 = static_cast<float>(1.0 / 3.0);
constexpr float kA2 = static_cast<float>(1.0 / 5.0);
constexpr float kA3 = static_cast<float>(1.0 / 7.0);
constexpr float kA4 = static_cast<float>(1.0 / 9.0);
constexpr float kA5 = static_cast<float>(1.0 / 11.0);
constexpr float kLn2f = static_cast<float>(kLn2d);
constexpr float kSqrt2f = static_cast<float>(1.41421356237309504880);

__device__ __forceinline__ float sw_exp2(float x) {
  if (x != x) return x;
  if (x < -126.0f) return 0.0f;
  if (x >= 128.0f) return INFINITY;
  const float n = rintf(x);
  const float f = __fsub_rn(x, n);
  float p = kE7;
  p = __fmaf_rn(p, f, kE6);
  p = __fmaf_rn(p, f, kE5);
  p = __fmaf_rn(p, f, kE4);
  p = __fmaf_rn(p, f, kE3);
  p = __fmaf_rn(p, f, kE2);
  p = __fmaf_rn(p, f, kE1);
  p = __fmaf_rn(p, f, kE0);
  const float two_n = __uint_as_float(static_cast<uint32_t>(static_cast<int>(n) + 127) << 23);
  return __fmul_rn(p, two_n);
}

// ln(d) = e*ln2 + ln(x) for positive normal d; returns e and ln(x).
__device__ __forceinline__ void sw_ln_split(float d, int& e, float& lnx) {
  const uint32_t u = __float_as_uint(d);
  e = static_cast<int>((u >> 23) & 0xffu) - 127;
  float x = __uint_as_float((u & 0x7fffffu) | 0x3f800000u);
  if (x > kSqrt2f) {
    x = __fmul_rn(x, 0.5f);
    e += 1;
  }
  const float t = __fdiv_rn(__fsub_rn(x, 1.0f), __fadd_rn(x, 1.0f));
  const float w = __fmul_rn(t, t);
  float p = kA5;
  p = __fmaf_rn(p, w, kA4);
  p = __fmaf_rn(p, w, kA3);
  p = __fmaf_rn(p, w, kA2);
  p = __fmaf_rn(p, w, kA1);
  p = __fmaf_rn(p, w, kA0);
  lnx = __fmul_rn(__fadd_rn(t, t), p);
}

// Chunks whose states one lane loads before folding them (a batch).
constexpr int kBatch = 16;

template <int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const CombineArgs a) {
  constexpr int VPL = D / 32;  // columns per lane
  // Launched as a programmatic dependent of the split-KV pass: wait until
  // that grid has finished and its partial states are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  if (row >= a.rows) return;
  const int S = a.S;
  const float* pm = a.part_m + static_cast<size_t>(row) * S;
  const float* pd = a.part_d + static_cast<size_t>(row) * S;
  const float* po = a.part_o + static_cast<size_t>(row) * S * D + lane * VPL;

  float m = -INFINITY, d = 0.0f;
  float o[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) o[i] = 0.0f;

  for (int c0 = 0; c0 < S; c0 += kBatch) {
    // All loads of the batch first (one memory latency per batch): every
    // lane its columns of the 16 partial o rows, lane i < 16 the m and d of
    // chunk c0 + i.
    float ob[kBatch][VPL];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
#pragma unroll
      for (int k = 0; k < VPL; ++k) ob[i][k] = 0.0f;
      if (c0 + i < S) {
        const size_t c = static_cast<size_t>(c0 + i);
        if constexpr (VPL == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(po + c * D));
          ob[i][0] = x.x; ob[i][1] = x.y; ob[i][2] = x.z; ob[i][3] = x.w;
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(po + c * D));
          ob[i][0] = x.x; ob[i][1] = x.y;
        }
      }
    }
    float my_m = -INFINITY, my_d = 0.0f;  // past the last chunk: the identity
    if (lane < kBatch && c0 + lane < S) {
      my_m = __ldg(pm + c0 + lane);
      my_d = __ldg(pd + c0 + lane);
    }
    // The running maximum before each chunk follows from the chunks' m alone
    // (the merge keeps the larger one), so lane i can compute chunk c0 + i's
    // merge factor while the other lanes compute theirs; the fold below then
    // applies them in chunk order.  Each factor is the same operation on the
    // same operands as in a serial fold.
    float my_mprev = m;
    {
      float mr = m;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float mbi = __shfl_sync(0xffffffffu, my_m, i);
        if (lane == i) my_mprev = mr;
        if (mbi != -INFINITY && (mr == -INFINITY || !(mr >= mbi))) mr = mbi;
      }
    }
    const float my_f = sw_exp2(my_mprev >= my_m ? __fsub_rn(my_m, my_mprev)
                                                : __fsub_rn(my_mprev, my_m));
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const float mbi = __shfl_sync(0xffffffffu, my_m, i);
      const float dbi = __shfl_sync(0xffffffffu, my_d, i);
      const float fi = __shfl_sync(0xffffffffu, my_f, i);
      if (mbi == -INFINITY) continue;  // chunk c0 + i is the identity
      if (m == -INFINITY) {            // the running state is the identity
        m = mbi;
        d = dbi;
#pragma unroll
        for (int k = 0; k < VPL; ++k) o[k] = ob[i][k];
        continue;
      }
      if (m >= mbi) {
        d = __fmaf_rn(dbi, fi, d);
#pragma unroll
        for (int k = 0; k < VPL; ++k) o[k] = __fmaf_rn(ob[i][k], fi, o[k]);
      } else {
        d = __fmaf_rn(d, fi, dbi);
#pragma unroll
        for (int k = 0; k < VPL; ++k) o[k] = __fmaf_rn(o[k], fi, ob[i][k]);
        m = mbi;
      }
    }
  }

  float lse;
  if (d == 0.0f) {
    lse = -INFINITY;
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = 0.0f;
  } else {
    int e;
    float lnx;
    sw_ln_split(d, e, lnx);
    lse = __fmaf_rn(__fadd_rn(static_cast<float>(e), m), kLn2f, lnx);
#pragma unroll
    for (int i = 0; i < VPL; ++i) o[i] = __fdiv_rn(o[i], d);
  }
  if (lane == 0) a.lse[row] = lse;
  const size_t base = static_cast<size_t>(row) * D + lane * VPL;
  if (a.o_f32) {
    float* dst = static_cast<float*>(a.o) + base;
    if constexpr (VPL == 4)
      *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
    else
      *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.o) + base;
#pragma unroll
    for (int i = 0; i < VPL; ++i) dst[i] = __float2bfloat16_rn(o[i]);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int D, cudaStream_t stream) {
  // Programmatic dependent launch: the CTAs may be scheduled while the
  // preceding kernel on the stream is still finishing (the split-KV pass
  // allows it once all of its CTAs have started) and wait for its results in
  // griddepcontrol.wait, so the launch latency overlaps that kernel's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((a.rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) return cudaLaunchKernelEx(&cfg, fa_combine_kernel<128>, a);
  return cudaLaunchKernelEx(&cfg, fa_combine_kernel<64>, a);
}

}  // namespace fa
