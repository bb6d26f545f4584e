// Split-KV decode, first pass: the per-chunk states (m, d, o).
//
// "Learning FlashAttention the Hard Way - Part 1", "Associativity is All You
// Need": because the merge is associative, separate thread blocks may each
// reduce one chunk of the keys and leave their partial state in scratch for a
// second kernel to fold ("The Merge, and the Twist").  States are in the
// base-2 coordinates of "Alternative Twist: Base 2": m is the chunk maximum
// of sigma = s * log2 e, d = sum 2^(sigma - m), o = sum 2^(sigma - m) v.
//
// The pass streams the whole KV cache once, so it is bound by HBM bandwidth.
// Grid (num_splits, ceil(H / 8), B); a CTA of 8 warps covers 8 consecutive
// heads of one (sequence, chunk), so for each key the CTA reads 8 adjacent
// 256-byte rows (2 KB contiguous at D = 128).  Within a warp, D/8 lanes cover
// one key row with 16-byte loads and the warp covers 32/(D/8) keys per load;
// every lane keeps 8 loads of K and 8 of V in flight.  Each lane group folds
// its keys into its own state; the groups are merged by warp shuffles at the
// end (the same merge, once more).

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

template <int D>
__global__ void __launch_bounds__(256) fa_decode_splitkv_kernel(const DecodeArgs a) {
  constexpr int LPR = D / 8;         // lanes per key row (8 bf16 = 16 B per lane)
  constexpr int GROUPS = 32 / LPR;   // keys per warp-wide load
  constexpr int U = 8;               // loads in flight per lane per operand
  constexpr int KPI = GROUPS * U;    // keys per iteration

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int h = blockIdx.y * 8 + warp;
  const int b = blockIdx.z;
  const int S = a.S;
  const int H = a.H;

  const int k_begin = __ldg(a.cu_seqlens_k + b);
  const int k_end = __ldg(a.cu_seqlens_k + b + 1);
  if (k_begin < 0 || k_end < k_begin || k_end > a.total_kv) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    return;
  }
  if (h >= H) return;
  const int L = k_end - k_begin;
  const int size = (L + S - 1) / S;
  const int k0 = min(L, c * size);
  const int k1 = min(L, (c + 1) * size);
  const size_t out = (static_cast<size_t>(b) * H + h) * S + c;

  const int g = lane / LPR;
  const int dl = lane % LPR;

  if (k0 >= k1) {  // empty chunk: the identity (-inf, 0, 0)
    if (g == 0) {
      float4* po = reinterpret_cast<float4*>(a.part_o + out * D + dl * 8);
      po[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      po[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lane == 0) {
      a.part_m[out] = -INFINITY;
      a.part_d[out] = 0.f;
    }
    return;
  }

  // q pre-multiplied by scale*log2(e): the dot product is sigma directly.
  float qv[8];
  {
    const uint4 qr = *reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(b) * H + h) * D + dl * 8);
    const uint32_t w[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_f2(w[i]);
      qv[2 * i] = f.x * a.scale_log2;
      qv[2 * i + 1] = f.y * a.scale_log2;
    }
  }

  const size_t row_stride = static_cast<size_t>(H) * D;  // elements between keys
  const uint16_t* kbase =
      static_cast<const uint16_t*>(a.k_cache) + static_cast<size_t>(k_begin) * row_stride +
      static_cast<size_t>(h) * D + dl * 8;
  const uint16_t* vbase =
      static_cast<const uint16_t*>(a.v_cache) + static_cast<size_t>(k_begin) * row_stride +
      static_cast<size_t>(h) * D + dl * 8;

  float m = -INFINITY, dsum = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  for (int kb = k0; kb < k1; kb += KPI) {
    uint4 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = kb + u * GROUPS + g;
      if (key < k1) {
        kr[u] = ld_stream_u4(kbase + static_cast<size_t>(key) * row_stride);
        vr[u] = ld_stream_u4(vbase + static_cast<size_t>(key) * row_stride);
      } else {
        kr[u] = make_uint4(0u, 0u, 0u, 0u);
        vr[u] = kr[u];
      }
    }
    float t[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t w[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bf16x2_to_f2(w[i]);
        part = fmaf(qv[2 * i], f.x, part);
        part = fmaf(qv[2 * i + 1], f.y, part);
      }
      t[u] = part;
    }
#pragma unroll
    for (int off = LPR / 2; off >= 1; off >>= 1) {
#pragma unroll
      for (int u = 0; u < U; ++u) t[u] += __shfl_xor_sync(0xffffffffu, t[u], off);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = kb + u * GROUPS + g;
      if (key >= k1) t[u] = -INFINITY;
      mx = fmaxf(mx, t[u]);
    }
    const float m_new = fmaxf(m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_use);
    float rs = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= alpha;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float p = ex2_approx(t[u] - m_use);
      rs += p;
      const uint32_t w[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = bf16x2_to_f2(w[i]);
        acc[2 * i] = fmaf(p, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(p, f.y, acc[2 * i + 1]);
      }
    }
    dsum = dsum * alpha + rs;
    m = m_new;
  }

  // Merge the lane groups' states (each group saw a disjoint subset of keys).
#pragma unroll
  for (int off = LPR; off < 32; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float d_o = __shfl_xor_sync(0xffffffffu, dsum, off);
    float ao[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ao[i] = __shfl_xor_sync(0xffffffffu, acc[i], off);
    if (mo == -INFINITY) {
      // other side is the identity
    } else if (m == -INFINITY) {
      m = mo;
      dsum = d_o;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = ao[i];
    } else if (m >= mo) {
      const float f = ex2_approx(mo - m);
      dsum = fmaf(d_o, f, dsum);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(ao[i], f, acc[i]);
    } else {
      const float f = ex2_approx(m - mo);
      dsum = fmaf(dsum, f, d_o);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(acc[i], f, ao[i]);
      m = mo;
    }
  }

  if (g == 0) {
    float4* po = reinterpret_cast<float4*>(a.part_o + out * D + dl * 8);
    po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (lane == 0) {
    a.part_m[out] = m;
    a.part_d[out] = dsum;
  }
}

cudaError_t launch_decode_splitkv(const DecodeArgs& a, int D, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(a.S), static_cast<unsigned>((a.H + 7) / 8),
            static_cast<unsigned>(a.B));
  if (D == 128)
    fa_decode_splitkv_kernel<128><<<grid, 256, 0, stream>>>(a);
  else
    fa_decode_splitkv_kernel<64><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
