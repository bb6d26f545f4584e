// Per-row mean / variance (LayerNorm statistics) as a monoid reduction of
// Welford states (n, mu, M2), with the split-K + combine structure of the
// attention decode.
//
// "Learning FlashAttention the Hard Way - Part 1", section "The Same Move:
// Welford's Variance": a sample injects as (1, x, 0), two partials over
// disjoint chunks merge symmetrically (identity (0, 0, 0)), and the variance
// is M2 / n at the end; section "Why Welford's Combine Associates" shows the
// merge is associative, which is what lets any split and any bracketing give
// the same statistics.  The merge used here:
//     n = n_a + n_b,  delta = mu_b - mu_a,  r = n_b / n,
//     mu = mu_a + delta r,  M2 = M2_a + M2_b + delta^2 n_a r.
//
// fa_row_stats_kernel: a group of WARPS warps (1, or 8 for segments of at
// least 16384 elements) reduces one segment (a row, or one column chunk of a
// row).  Each thread folds 16-byte packs (4 fp32 values, or bf16 in pairs of
// packs, 16 values, in the unrolled loop and 8 in the remainder): the
// pack's own state by its definition (mean of the pack, then the sum of
// squared deviations), merged into the thread's running state; then the lanes merge by shuffles (lane i with lane i + off) and the
// warps of a group in index order through shared memory.  The fold order
// depends only on the sizes, so results are deterministic.  Loads are 16-byte
// and streaming (no L1 allocation); ragged heads and tails of a segment that
// are not 16-byte aligned are folded one element at a time.
//
// fa_row_stats_combine_kernel: one thread per row folds the row's chunk
// states left to right with one IEEE rounding per operation in a fixed
// order (__f*_rn, no contraction), then var = M2 / n and
// rstd = 1 / sqrt(var + eps), so a plain C fold of the same states gives the
// same bits.

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

struct Welford {
  float n, mu, m2;
};

__device__ __forceinline__ Welford merge(const Welford& a, const Welford& b) {
  if (b.n == 0.f) return a;
  if (a.n == 0.f) return b;
  const float n = a.n + b.n;
  const float delta = b.mu - a.mu;
  const float r = __fdividef(b.n, n);
  Welford o;
  o.n = n;
  o.mu = fmaf(delta, r, a.mu);
  o.m2 = fmaf(delta * delta * a.n, r, a.m2 + b.m2);
  return o;
}

// The state of VEC values by its definition.
template <int VEC>
__device__ __forceinline__ Welford pack_state(const float (&v)[VEC]) {
  float s[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) s[i] = v[i];
#pragma unroll
  for (int w = VEC / 2; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) s[i] += s[i + w];
  const float mu = s[0] * (1.f / VEC);  // VEC is a power of two: exact scaling
  float m2 = 0.f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const float d = v[i] - mu;
    m2 = fmaf(d, d, m2);
  }
  return Welford{static_cast<float>(VEC), mu, m2};
}

// The state of the 16 bf16 values of two 16-byte packs by its definition,
// in packed pairs: mean = (sum of the pairs) / 16, then the sum of squared
// deviations.
__device__ __forceinline__ Welford pack_state_bf16x16(const uint4& a, const uint4& b) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float2 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    v[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  float2 s[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = __fadd2_rn(v[i], v[i + 4]);
  s[0] = __fadd2_rn(s[0], s[2]);
  s[1] = __fadd2_rn(s[1], s[3]);
  s[0] = __fadd2_rn(s[0], s[1]);
  const float mu = (s[0].x + s[0].y) * (1.f / 16.f);  // exact scaling by a power of two
  const float2 nm = make_float2(-mu, -mu);
  float2 q0 = make_float2(0.f, 0.f), q1 = q0;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const float2 d0 = __fadd2_rn(v[i], nm), d1 = __fadd2_rn(v[i + 1], nm);
    q0 = __ffma2_rn(d0, d0, q0);
    q1 = __ffma2_rn(d1, d1, q1);
  }
  q0 = __fadd2_rn(q0, q1);
  return Welford{16.f, mu, q0.x + q0.y};
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <bool BF16>
__device__ __forceinline__ float load_one(const void* base, long long i) {
  if constexpr (BF16)
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[i]) << 16);
  return static_cast<const float*>(base)[i];
}

template <bool BF16, int VEC>
__device__ __forceinline__ void unpack(const uint4& u, float (&v)[VEC]) {
  if constexpr (BF16) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
  }
}

template <int WARPS, bool BF16>
__global__ void __launch_bounds__(256) fa_row_stats_kernel(const RowStatsArgs a) {
  constexpr int VEC = BF16 ? 8 : 4;        // elements per 16-byte pack
  constexpr int ESZ = BF16 ? 2 : 4;        // element bytes
  constexpr int G = WARPS * 32;            // threads per segment
  constexpr int GROUPS = 8 / WARPS;        // segments per CTA
  constexpr int UNROLL = WARPS == 1 ? 8 : 4;  // packs in flight per thread
  __shared__ Welford part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WARPS;
  const int tg = (warp % WARPS) * 32 + lane;
  const long long seg = static_cast<long long>(blockIdx.x) * GROUPS + grp;
  const bool live = seg < static_cast<long long>(a.R) * a.S;
  Welford st{0.f, 0.f, 0.f};
  long long r = 0;
  int c = 0;
  if (live) {
    r = seg / a.S;
    c = static_cast<int>(seg % a.S);
    const long long step = (static_cast<long long>(a.C) + a.S - 1) / a.S;
    const long long lo = min(static_cast<long long>(a.C), c * step);
    const long long hi = min(static_cast<long long>(a.C), lo + step);
    const char* row = static_cast<const char*>(a.x) + r * static_cast<long long>(a.C) * ESZ;
    // first 16-byte aligned element at or after lo
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row) + lo * ESZ;
    long long a0 = lo + static_cast<long long>(((16u - (addr & 15u)) & 15u) / ESZ);
    if ((addr & (ESZ - 1)) != 0 || a0 > hi) a0 = hi;  // (element-misaligned: all scalar)
    const long long npk = (hi - a0) / VEC;
    const long long a1 = a0 + npk * VEC;
    for (long long i = lo + tg; i < a0; i += G)
      st = merge(st, Welford{1.f, load_one<BF16>(row, i), 0.f});
    const uint4* body = reinterpret_cast<const uint4*>(row + a0 * ESZ);
    long long p = tg;
    for (; p + (UNROLL - 1) * G < npk; p += UNROLL * G) {
      uint4 u[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) u[k] = ld_stream(body + p + k * G);
      if constexpr (BF16) {
#pragma unroll
        for (int k = 0; k < UNROLL; k += 2) st = merge(st, pack_state_bf16x16(u[k], u[k + 1]));
      } else {
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          float v[VEC];
          unpack<BF16, VEC>(u[k], v);
          st = merge(st, pack_state<VEC>(v));
        }
      }
    }
    for (; p < npk; p += G) {
      float v[VEC];
      unpack<BF16, VEC>(ld_stream(body + p), v);
      st = merge(st, pack_state<VEC>(v));
    }
    for (long long i = a1 + tg; i < hi; i += G)
      st = merge(st, Welford{1.f, load_one<BF16>(row, i), 0.f});
  }
#pragma unroll
  for (int off = 1; off < 32; off *= 2) {
    Welford o;
    o.n = __shfl_down_sync(0xffffffffu, st.n, off);
    o.mu = __shfl_down_sync(0xffffffffu, st.mu, off);
    o.m2 = __shfl_down_sync(0xffffffffu, st.m2, off);
    if ((lane & (2 * off - 1)) == 0) st = merge(st, o);
  }
  if (WARPS > 1) {
    if (lane == 0) part[warp] = st;
    __syncthreads();
    if (tg == 0) {
      for (int w = 1; w < WARPS; ++w) st = merge(st, part[grp * WARPS + w]);
    }
  }
  if (!live || tg != 0) return;
  if (a.part_n) {
    const long long i = r * a.S + c;
    a.part_n[i] = st.n;
    a.part_mu[i] = st.mu;
    a.part_m2[i] = st.m2;
  } else {
    const float var = __fdiv_rn(st.m2, st.n);
    a.mean[r] = st.mu;
    a.var[r] = var;
    if (a.rstd) a.rstd[r] = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(var, a.eps)));
  }
}

__global__ void __launch_bounds__(256) fa_row_stats_combine_kernel(const RowStatsCombineArgs a) {
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= a.R) return;
  float n = 0.f, mu = 0.f, m2 = 0.f;
  for (int c = 0; c < a.S; ++c) {
    const long long i = r * a.S + c;
    const float nb = a.part_n[i], mub = a.part_mu[i], m2b = a.part_m2[i];
    if (nb == 0.f) continue;
    if (n == 0.f) {
      n = nb;
      mu = mub;
      m2 = m2b;
      continue;
    }
    const float na = n;
    const float nn = __fadd_rn(na, nb);
    const float delta = __fsub_rn(mub, mu);
    const float rr = __fdiv_rn(nb, nn);
    mu = __fadd_rn(mu, __fmul_rn(delta, rr));
    m2 = __fadd_rn(__fadd_rn(m2, m2b), __fmul_rn(__fmul_rn(__fmul_rn(delta, delta), na), rr));
    n = nn;
  }
  const float var = __fdiv_rn(m2, n);
  a.mean[r] = mu;
  a.var[r] = var;
  if (a.rstd) a.rstd[r] = __fdiv_rn(1.f, __fsqrt_rn(__fadd_rn(var, a.eps)));
}

template <int WARPS, bool BF16>
cudaError_t launch_stats(const RowStatsArgs& a, cudaStream_t stream) {
  constexpr int GROUPS = 8 / WARPS;
  const long long segs = static_cast<long long>(a.R) * a.S;
  const unsigned blocks = static_cast<unsigned>((segs + GROUPS - 1) / GROUPS);
  fa_row_stats_kernel<WARPS, BF16><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_stats(const RowStatsArgs& a, cudaStream_t stream) {
  // A warp per segment keeps 8 packs (128 bytes) per lane in flight; only
  // segments of at least 16384 elements get a whole CTA (8 warps).
  const long long seg_len = (static_cast<long long>(a.C) + a.S - 1) / a.S;
  const bool wide = seg_len >= 16384;
  if (a.bf16) return wide ? launch_stats<8, true>(a, stream) : launch_stats<1, true>(a, stream);
  return wide ? launch_stats<8, false>(a, stream) : launch_stats<1, false>(a, stream);
}

cudaError_t launch_row_stats_combine(const RowStatsCombineArgs& a, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((static_cast<long long>(a.R) + 255) / 256);
  fa_row_stats_combine_kernel<<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
