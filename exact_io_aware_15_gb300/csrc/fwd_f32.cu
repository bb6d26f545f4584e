// Exact attention forward in fp32 on the CUDA cores (FFMA; no tensor cores,
// whose tf32 inputs would lose the fp32 accuracy this path exists for).
//
// Same fold as the tensor-core kernel ("Learning FlashAttention the Hard Way -
// Part 1": "The State", "The Merge, and the Twist", "Alternative Twist:
// Base 2"): a CTA of 128 threads owns 128/TPR query rows of one (batch,
// head); TPR threads share a row, each holding D/TPR columns of q and of the
// unnormalised output o (TPR = 2 when the grid fills the GPU, 8 for small
// problems, whose latency the shorter per-thread chains cut).  Key/value
// tiles of 32 rows are staged in shared memory; each tile is folded into the
// row state (m, d, o) by one merge, masked keys entering as the identity
// (sigma = -inf).  The divide o / d is deferred to the end.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

template <int D, int TPR>
__global__ void __launch_bounds__(128) fa_fwd_f32_kernel(const F32FwdArgs a) {
  constexpr int ROWS = 128 / TPR;
  constexpr int KT = 32;
  constexpr int HD = D / TPR;
  constexpr int PAD = HD + 4;  // part offset: avoids bank conflicts between the parts
  __shared__ __align__(16) float ks[KT][TPR * PAD];
  __shared__ __align__(16) float vs[KT][TPR * PAD];

  const int bh = blockIdx.x;
  const int mb = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
  const int tid = threadIdx.x;
  const int row = tid / TPR;
  const int half = tid % TPR;  // this thread's part of the row
  const int N = a.N;
  const int qpos = mb * ROWS + row;
  const bool valid = qpos < N;
  const size_t head = static_cast<size_t>(bh) * N;

  float qr[HD];
  {
    const float* src = a.q + (head + (valid ? qpos : 0)) * D + half * HD;
#pragma unroll
    for (int i = 0; i < HD; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(src + i);
      qr[i] = x.x;
      qr[i + 1] = x.y;
      qr[i + 2] = x.z;
      qr[i + 3] = x.w;
    }
  }
  float acc[HD];
#pragma unroll
  for (int i = 0; i < HD; ++i) acc[i] = 0.f;
  float m = -INFINITY, dsum = 0.f;
  const float c = a.scale_log2;

  const int kend = a.causal ? min(N, (mb + 1) * ROWS) : N;
  for (int k0 = 0; k0 < kend; k0 += KT) {
    __syncthreads();
    // stage K/V rows k0 .. k0+KT-1 (zero rows past the end)
    for (int idx = tid; idx < KT * (D / 4); idx += 128) {
      const int rr = idx / (D / 4);
      const int cc = (idx % (D / 4)) * 4;
      const int key = k0 + rr;
      float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
      if (key < N) {
        kx = *reinterpret_cast<const float4*>(a.k + (head + key) * D + cc);
        vx = *reinterpret_cast<const float4*>(a.v + (head + key) * D + cc);
      }
      const int col = (cc / HD) * PAD + cc % HD;
      *reinterpret_cast<float4*>(&ks[rr][col]) = kx;
      *reinterpret_cast<float4*>(&vs[rr][col]) = vx;
    }
    __syncthreads();

    float t[KT];
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const float* kr = &ks[kk][half * PAD];
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < HD; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(kr + i);
        part = fmaf(qr[i], x.x, part);
        part = fmaf(qr[i + 1], x.y, part);
        part = fmaf(qr[i + 2], x.z, part);
        part = fmaf(qr[i + 3], x.w, part);
      }
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      const int key = k0 + kk;
      const bool vis = key < N && (!a.causal || key <= qpos);
      t[kk] = vis ? part * c : -INFINITY;
    }
    float mx = t[0];
#pragma unroll
    for (int kk = 1; kk < KT; ++kk) mx = fmaxf(mx, t[kk]);
    const float m_new = fmaxf(m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m_new == m) ? 1.f : exp2f(m - m_use);
    float rs = 0.f;
#pragma unroll
    for (int i = 0; i < HD; ++i) acc[i] *= alpha;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const float p = exp2f(t[kk] - m_use);
      rs += p;
      const float* vr = &vs[kk][half * PAD];
#pragma unroll
      for (int i = 0; i < HD; i += 4) {
        const float4 x = *reinterpret_cast<const float4*>(vr + i);
        acc[i] = fmaf(p, x.x, acc[i]);
        acc[i + 1] = fmaf(p, x.y, acc[i + 1]);
        acc[i + 2] = fmaf(p, x.z, acc[i + 2]);
        acc[i + 3] = fmaf(p, x.w, acc[i + 3]);
      }
    }
    dsum = dsum * alpha + rs;
    m = m_new;
  }

  if (!valid) return;
  const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
  const size_t orow = head + qpos;
  if (a.o_f32) {
    float* dst = static_cast<float*>(a.o) + orow * D + half * HD;
#pragma unroll
    for (int i = 0; i < HD; i += 4)
      *reinterpret_cast<float4*>(dst + i) =
          make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
  } else {
    uint16_t* dst = static_cast<uint16_t*>(a.o) + orow * D + half * HD;
#pragma unroll
    for (int i = 0; i < HD; i += 8) {
      uint4 u;
      u.x = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
      u.y = pack_bf16x2(acc[i + 2] * inv, acc[i + 3] * inv);
      u.z = pack_bf16x2(acc[i + 4] * inv, acc[i + 5] * inv);
      u.w = pack_bf16x2(acc[i + 6] * inv, acc[i + 7] * inv);
      *reinterpret_cast<uint4*>(dst + i) = u;
    }
  }
  if (half == 0)
    a.lse[orow] = dsum > 0.f ? (m + log2f(dsum)) * 0.69314718055994530942f : -INFINITY;
}

cudaError_t launch_fwd_f32(const F32FwdArgs& a, int D, cudaStream_t stream) {
  // two threads per row when that grid fills the GPU twice over, else eight
  const long long ctas2 = static_cast<long long>(a.BH) * ((a.N + 63) / 64);
  if (ctas2 >= 304) {
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>((a.N + 63) / 64));
    if (D == 128)
      fa_fwd_f32_kernel<128, 2><<<grid, 128, 0, stream>>>(a);
    else
      fa_fwd_f32_kernel<64, 2><<<grid, 128, 0, stream>>>(a);
  } else {
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>((a.N + 15) / 16));
    if (D == 128)
      fa_fwd_f32_kernel<128, 8><<<grid, 128, 0, stream>>>(a);
    else
      fa_fwd_f32_kernel<64, 8><<<grid, 128, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fa
