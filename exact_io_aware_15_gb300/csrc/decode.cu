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
// Within a warp, D/8 lanes cover one key row with 16-byte loads and the warp
// covers 32/(D/8) keys per load; every lane keeps 8 loads of K and 8 of V in
// flight.  Each lane group folds its keys into its own state; the groups are
// merged by warp shuffles at the end (the same merge, once more).  Two cache
// layouts share that fold: a packed [T_k, H, D] cache with cu_seqlens, and a
// paged cache (pages [P, page_size, H_kv, D] reached through a block table)
// whose KV heads may each serve a group of query heads.

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

// Where the key rows of one (sequence, KV head) live.  `row` gives the element
// offset of key `key` from the warp's base pointers, or false for a key whose
// page index is out of range.
struct ContigRows {  // packed [T_k, H, D] caches
  const uint16_t* k;
  const uint16_t* v;
  size_t stride;  // elements between consecutive keys (H * D)
  __device__ __forceinline__ bool row(int key, size_t& off) const {
    off = static_cast<size_t>(key) * stride;
    return true;
  }
  // streamed once: no L1 allocation
  __device__ __forceinline__ uint4 load(const uint16_t* p) const { return ld_stream_u4(p); }
};

struct PagedRows {  // pages [num_pages, page_size, H_kv, D] and a block table
  const uint16_t* k;
  const uint16_t* v;
  const int* table;  // this sequence's row of the block table
  int page_shift;    // log2(page_size)
  int num_pages;
  size_t page_stride;  // elements per page (page_size * H_kv * D)
  size_t row_stride;   // elements between keys of one page (H_kv * D)
  __device__ __forceinline__ bool row(int key, size_t& off) const {
    const int pg = __ldg(table + (key >> page_shift));
    if (pg < 0 || pg >= num_pages) return false;
    off = static_cast<size_t>(pg) * page_stride +
          static_cast<size_t>(key & ((1 << page_shift) - 1)) * row_stride;
    return true;
  }
  // the query heads of one KV head read the same rows: keep them in L1
  __device__ __forceinline__ uint4 load(const uint16_t* p) const {
    return __ldg(reinterpret_cast<const uint4*>(p));
  }
};

// Folds keys [k0, k1) of one (sequence, query head) into the base-2 state
// (m, d, o) and writes it to slot `out` of the partial-state arrays; an
// empty range writes the identity (-inf, 0, 0).  One warp: D/8 lanes per
// key row, 16-byte loads, 8 loads of K and 8 of V in flight per lane.
template <int D, class Rows>
__device__ __forceinline__ void fold_chunk(const Rows& rows, const uint16_t* qrow,
                                           float scale_log2, int k0, int k1, size_t out,
                                           float* part_m, float* part_d, float* part_o,
                                           unsigned int* status) {
  constexpr int LPR = D / 8;         // lanes per key row (8 bf16 = 16 B per lane)
  constexpr int GROUPS = 32 / LPR;   // keys per warp-wide load
  constexpr int U = 8;               // loads in flight per lane per operand
  constexpr int KPI = GROUPS * U;    // keys per iteration
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR;
  const int dl = lane % LPR;

  if (k0 >= k1) {  // empty chunk: the identity (-inf, 0, 0)
    if (g == 0) {
      float4* po = reinterpret_cast<float4*>(part_o + out * D + dl * 8);
      po[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      po[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lane == 0) {
      part_m[out] = -INFINITY;
      part_d[out] = 0.f;
    }
    return;
  }

  // q pre-multiplied by scale*log2(e): the dot product is sigma directly.
  float qv[8];
  {
    const uint4 qr = *reinterpret_cast<const uint4*>(qrow + dl * 8);
    const uint32_t w[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_f2(w[i]);
      qv[2 * i] = f.x * scale_log2;
      qv[2 * i + 1] = f.y * scale_log2;
    }
  }
  const uint16_t* kbase = rows.k + dl * 8;
  const uint16_t* vbase = rows.v + dl * 8;

  float m = -INFINITY, dsum = 0.f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool bad = false;

  for (int kb = k0; kb < k1; kb += KPI) {
    uint4 kr[U], vr[U];
    bool vis[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = kb + u * GROUPS + g;
      size_t off = 0;
      vis[u] = key < k1 && rows.row(key, off);
      bad |= key < k1 && !vis[u];
      if (vis[u]) {
        kr[u] = rows.load(kbase + off);
        vr[u] = rows.load(vbase + off);
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
      if (!vis[u]) t[u] = -INFINITY;  // the identity's m
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
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, kStatusBounds);

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
    float4* po = reinterpret_cast<float4*>(part_o + out * D + dl * 8);
    po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (lane == 0) {
    part_m[out] = m;
    part_d[out] = dsum;
  }
}

// Chunk c of a length-L sequence: keys [c*ceil(L/S), min(L, (c+1)*ceil(L/S))).
__device__ __forceinline__ void chunk_range(int L, int S, int c, int& k0, int& k1) {
  const int size = (L + S - 1) / S;
  k0 = min(L, c * size);
  k1 = min(L, (c + 1) * size);
}

// Grid (num_splits, ceil(H / 8), B); a CTA of 8 warps covers 8 consecutive
// heads of one (sequence, chunk), so for each key the CTA reads 8 adjacent
// 256-byte rows (2 KB contiguous at D = 128).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_splitkv_kernel(const DecodeArgs a) {
  // The combine that follows may be scheduled once every CTA of this grid
  // has started (it waits for this grid's results before reading them).
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int h = blockIdx.y * 8 + warp;
  const int b = blockIdx.z;
  const int S = a.S;
  const int H = a.H;

  int k_begin = __ldg(a.cu_seqlens_k + b);
  int k_end = __ldg(a.cu_seqlens_k + b + 1);
  if (k_begin < 0 || k_end < k_begin || k_end > a.total_kv) {
    // Offsets out of range: read nothing, report it, and leave the identity
    // (-inf, 0, 0) in this CTA's states (an empty sequence), so the second
    // pass never folds a state that this launch did not write.
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    k_begin = 0;
    k_end = 0;
  }
  if (h >= H) return;
  int k0, k1;
  chunk_range(k_end - k_begin, S, c, k0, k1);
  const size_t stride = static_cast<size_t>(H) * D;
  const size_t base = static_cast<size_t>(k_begin) * stride + static_cast<size_t>(h) * D;
  ContigRows rows{static_cast<const uint16_t*>(a.k_cache) + base,
                  static_cast<const uint16_t*>(a.v_cache) + base, stride};
  const uint16_t* qrow =
      static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(b) * H + h) * D;
  fold_chunk<D>(rows, qrow, a.scale_log2, k0, k1, (static_cast<size_t>(b) * H + h) * S + c,
                a.part_m, a.part_d, a.part_o, a.status);
}

// Paged cache with grouped query heads: query head h reads KV head
// h / (H / H_kv); the CTA's 8 warps are 8 consecutive query heads, so warps
// of one group read the same rows (served by L1 after the first).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_paged_kernel(const PagedDecodeArgs a) {
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int h = blockIdx.y * 8 + warp;
  const int b = blockIdx.z;
  int L = __ldg(a.seqlens + b);
  if (L < 0 || static_cast<long long>(L) > static_cast<long long>(a.max_blocks) * a.page_size) {
    // A length out of range: report it and write the identity states (as
    // for an empty sequence) instead of reading anything.
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    L = 0;
  }
  if (h >= a.H) return;
  const int hk = h / (a.H / a.Hkv);
  int k0, k1;
  chunk_range(L, a.S, c, k0, k1);
  const size_t row_stride = static_cast<size_t>(a.Hkv) * D;
  PagedRows rows{static_cast<const uint16_t*>(a.k_pages) + static_cast<size_t>(hk) * D,
                 static_cast<const uint16_t*>(a.v_pages) + static_cast<size_t>(hk) * D,
                 a.block_table + static_cast<size_t>(b) * a.max_blocks,
                 __ffs(a.page_size) - 1,
                 a.num_pages,
                 static_cast<size_t>(a.page_size) * row_stride,
                 row_stride};
  const uint16_t* qrow =
      static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(b) * a.H + h) * D;
  fold_chunk<D>(rows, qrow, a.scale_log2, k0, k1,
                (static_cast<size_t>(b) * a.H + h) * a.S + c, a.part_m, a.part_d, a.part_o,
                a.status);
}

cudaError_t launch_decode_paged(const PagedDecodeArgs& a, int D, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(a.S), static_cast<unsigned>((a.H + 7) / 8),
            static_cast<unsigned>(a.B));
  if (D == 128)
    fa_decode_paged_kernel<128><<<grid, 256, 0, stream>>>(a);
  else
    fa_decode_paged_kernel<64><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
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
