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
//
// Small problems at D = 64 (one head of a few hundred rows) take a second
// kernel that cuts the per-row chain instead: a thread owns a whole row of q
// and o for one eighth of the keys (a key group), so a score needs no
// cross-thread reduction, and the eight groups' states are folded together
// at the end, in group order, with the merge of "The Merge, and the Twist"
// (the split-K of "Associativity is All You Need" inside the CTA).

#include <atomic>
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

// ---- small problems, D = 64 ----
// CTA: 16 query rows x 8 key groups = 128 threads; key/value tiles of 64 rows
// double-buffered in shared memory by cp.async (rows padded to 68 floats so
// the eight groups' 16-byte reads fall in distinct banks).
constexpr int kSmRows = 16, kSmGroups = 8, kSmKT = 64, kSmLd = 68;
constexpr int kSmStage = 2 * kSmKT * kSmLd;                   // floats: K and V tile
constexpr int kSmSmemBytes = 2 * kSmStage * 4;                // two stages
static_assert(kSmRows * kSmGroups * 66 <= 2 * kSmStage, "merge area fits the stages");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__global__ void __launch_bounds__(128) fa_fwd_f32_small_kernel(const F32FwdArgs a) {
  constexpr int D = 64;
  extern __shared__ __align__(16) float sm[];
  const int bh = blockIdx.x;
  const int mb = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
  const int tid = threadIdx.x;
  const int r = tid / kSmGroups;  // row within the CTA
  const int g = tid % kSmGroups;  // key group: keys g, g + 8, ... of every tile
  const int N = a.N;
  const int qpos = mb * kSmRows + r;
  const bool valid = qpos < N;
  const size_t head = static_cast<size_t>(bh) * N;

  float q[D], acc[D];
  {
    const float* src = a.q + (head + (valid ? qpos : 0)) * D;
#pragma unroll
    for (int i = 0; i < D; i += 4) {
      const float4 x = *reinterpret_cast<const float4*>(src + i);
      q[i] = x.x;
      q[i + 1] = x.y;
      q[i + 2] = x.z;
      q[i + 3] = x.w;
    }
  }
#pragma unroll
  for (int i = 0; i < D; ++i) acc[i] = 0.f;
  float m = -INFINITY, dsum = 0.f;
  const float c = a.scale_log2;
  const int kend = a.causal ? min(N, (mb + 1) * kSmRows) : N;
  const int ntiles = (kend + kSmKT - 1) / kSmKT;

  // Copy tile t (K then V, zero rows past N) into stage `buf`.
  auto stage = [&](int t, int buf) {
    for (int idx = tid; idx < 2 * kSmKT * (D / 4); idx += 128) {
      const int which = idx / (kSmKT * (D / 4));
      const int rem = idx % (kSmKT * (D / 4));
      const int rr = rem / (D / 4), c4 = rem % (D / 4);
      const int key = t * kSmKT + rr;
      const float* src = (which ? a.v : a.k) + (head + (key < N ? key : 0)) * D + c4 * 4;
      const uint32_t dst =
          smem_u32(sm + buf * kSmStage + (which * kSmKT + rr) * kSmLd + c4 * 4);
      cp_async16(dst, src, key < N ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  if (ntiles > 0) stage(0, 0);
  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) {
      stage(t + 1, (t + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const float* ks = sm + (t & 1) * kSmStage;
    const float* vs = ks + kSmKT * kSmLd;
    float sc[kSmKT / kSmGroups];
#pragma unroll
    for (int i = 0; i < kSmKT / kSmGroups; ++i) {
      const int kr = g + kSmGroups * i;
      const float* kp = ks + kr * kSmLd;
      float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
      for (int e = 0; e < D; e += 4) {
        const float4 x = *reinterpret_cast<const float4*>(kp + e);
        p0 = fmaf(q[e], x.x, p0);
        p1 = fmaf(q[e + 1], x.y, p1);
        p2 = fmaf(q[e + 2], x.z, p2);
        p3 = fmaf(q[e + 3], x.w, p3);
      }
      const int key = t * kSmKT + kr;
      const bool vis = key < N && (!a.causal || key <= qpos);
      sc[i] = vis ? ((p0 + p1) + (p2 + p3)) * c : -INFINITY;
    }
    float mx = sc[0];
#pragma unroll
    for (int i = 1; i < kSmKT / kSmGroups; ++i) mx = fmaxf(mx, sc[i]);
    const float m_new = fmaxf(m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m_new == m) ? 1.f : exp2f(m - m_use);
#pragma unroll
    for (int e = 0; e < D; ++e) acc[e] *= alpha;
    float rs = 0.f;
#pragma unroll
    for (int i = 0; i < kSmKT / kSmGroups; ++i) {
      const float p = exp2f(sc[i] - m_use);
      rs += p;
      const float* vp = vs + (g + kSmGroups * i) * kSmLd;
#pragma unroll
      for (int e = 0; e < D; e += 4) {
        const float4 x = *reinterpret_cast<const float4*>(vp + e);
        acc[e] = fmaf(p, x.x, acc[e]);
        acc[e + 1] = fmaf(p, x.y, acc[e + 1]);
        acc[e + 2] = fmaf(p, x.z, acc[e + 2]);
        acc[e + 3] = fmaf(p, x.w, acc[e + 3]);
      }
    }
    dsum = dsum * alpha + rs;
    m = m_new;
    __syncthreads();  // the stage is refilled two tiles later
  }

  // Fold the eight key groups of each row (group order), thread (r, j)
  // producing columns [8 j, 8 j + 8).
  float* st = sm;  // [row][group][66]: o[64], m, d
  {
    float* my = st + (r * kSmGroups + g) * 66;
#pragma unroll
    for (int e = 0; e < D; ++e) my[e] = acc[e];
    my[64] = m;
    my[65] = dsum;
  }
  __syncthreads();
  const float* rowst = st + r * kSmGroups * 66;
  float M = -INFINITY;
#pragma unroll
  for (int gg = 0; gg < kSmGroups; ++gg) M = fmaxf(M, rowst[gg * 66 + 64]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float dd = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
  for (int gg = 0; gg < kSmGroups; ++gg) {
    const float w = exp2f(rowst[gg * 66 + 64] - Mu);  // 0 for an empty group
    dd = fmaf(rowst[gg * 66 + 65], w, dd);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = fmaf(rowst[gg * 66 + 8 * g + e], w, o[e]);
  }
  if (!valid) return;
  const float inv = dd > 0.f ? 1.f / dd : 0.f;
  const size_t orow = head + qpos;
  if (a.o_f32) {
    float* dst = static_cast<float*>(a.o) + orow * D + 8 * g;
    *reinterpret_cast<float4*>(dst) = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
    *reinterpret_cast<float4*>(dst + 4) =
        make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
  } else {
    uint16_t* dst = static_cast<uint16_t*>(a.o) + orow * D + 8 * g;
    uint4 u;
    u.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    u.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    u.z = pack_bf16x2(o[4] * inv, o[5] * inv);
    u.w = pack_bf16x2(o[6] * inv, o[7] * inv);
    *reinterpret_cast<uint4*>(dst) = u;
  }
  if (g == 0) a.lse[orow] = dd > 0.f ? (M + log2f(dd)) * 0.69314718055994530942f : -INFINITY;
}

cudaError_t launch_fwd_f32(const F32FwdArgs& a, int D, cudaStream_t stream) {
  // two threads per row when that grid fills the GPU twice over; else, at
  // D = 64, a thread per (row, key group), at D = 128 eight threads per row
  const long long ctas2 = static_cast<long long>(a.BH) * ((a.N + 63) / 64);
  if (ctas2 >= 304) {
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>((a.N + 63) / 64));
    if (D == 128)
      fa_fwd_f32_kernel<128, 2><<<grid, 128, 0, stream>>>(a);
    else
      fa_fwd_f32_kernel<64, 2><<<grid, 128, 0, stream>>>(a);
  } else if (D == 64) {
    static std::atomic<bool> attr_set[64];  // per device: shared-memory opt-in done
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(fa_fwd_f32_small_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmSmemBytes);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
    }
    dim3 grid(static_cast<unsigned>(a.BH), static_cast<unsigned>((a.N + kSmRows - 1) / kSmRows));
    fa_fwd_f32_small_kernel<<<grid, 128, kSmSmemBytes, stream>>>(a);
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
