// Prefix attention: for one query vector per (sequence, head) and every key
// position i of the sequence, the attention over keys 0..i -- the inclusive
// scan of the keys' online-softmax states under the merge (+).
//
// "Learning FlashAttention the Hard Way - Part 1", section "Why Attention's
// Combine Still Associates": the merge of (m, d, o) states is associative
// with identity (-inf, 0, 0), which is what lets exact attention run as a
// parallel prefix scan (the ELSA reference).  States are kept in the base-2
// coordinates of section "Alternative Twist: Base 2" (sigma = s log2 e).
//
// fa_prefix_scan_kernel<D>: one CTA (8 warps) per (sequence, head), longest
// sequences first.  The
// sequence is walked in windows of 128 keys, 16 per warp, in two phases:
//   A. each warp loads its 16 key and value rows into registers (lane l owns
//      columns [l*D/32, (l+1)*D/32)), computes the 16 scores (warp-reduced
//      dot products) and folds them into its segment total (m, d, o);
//   B. after a CTA barrier each warp forms its carry-in: the carry of all
//      earlier windows (+) the totals of the warps to its left, in index
//      order; then it rescans its 16 keys from registers, emitting
//      O_i = o / d and LSE_i = ln2 (m + log2 d) for every key.
// The carry of the next window is warp 7's running state after its rescan
// (the carry (+) every key of the window), shared through shared memory.
//
// Chunked rows (S > 1): the row's keys are cut into S chunks with the
// split-KV chunking; the chunks' states come from the split-KV first pass,
// and CTA (row, c) starts from the fold of chunks 0..c-1 and scans chunk c
// only, so S CTAs work on one row at once (depth L/S windows + S merges
// instead of L windows, for two reads of K and V instead of one).  K and V are read from HBM
// once; the depth per window is that of a two-level scan (16 sequential
// steps per warp, 8 totals across warps).

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kKeysPerWarp = 16;
constexpr int kWindow = 8 * kKeysPerWarp;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRankedSeqs = 256;

template <int VPL>
struct Cols;  // a lane's VPL bf16 columns of one row
template <>
struct Cols<4> {
  uint2 u;
};
template <>
struct Cols<2> {
  uint32_t u;
};

template <int VPL>
__device__ __forceinline__ Cols<VPL> ld_cols(const uint16_t* p) {
  Cols<VPL> c;
  if constexpr (VPL == 4) {
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(c.u.x), "=r"(c.u.y)
                 : "l"(p));
  } else {
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(c.u) : "l"(p));
  }
  return c;
}

template <int VPL>
__device__ __forceinline__ void to_f32(const Cols<VPL>& c, float (&x)[VPL]) {
  if constexpr (VPL == 4) {
    x[0] = __uint_as_float(c.u.x << 16);
    x[1] = __uint_as_float(c.u.x & 0xffff0000u);
    x[2] = __uint_as_float(c.u.y << 16);
    x[3] = __uint_as_float(c.u.y & 0xffff0000u);
  } else {
    x[0] = __uint_as_float(c.u << 16);
    x[1] = __uint_as_float(c.u & 0xffff0000u);
  }
}

// (m, d, o) (+)= (mb, db, ob) in base 2; an operand with m = -inf is the
// identity.
template <int VPL>
__device__ __forceinline__ void merge_into(float& m, float& d, float (&o)[VPL], float mb,
                                           float db, const float* ob) {
  if (mb == -INFINITY) return;
  if (m == -INFINITY) {
    m = mb;
    d = db;
#pragma unroll
    for (int c = 0; c < VPL; ++c) o[c] = ob[c];
    return;
  }
  const float mn = fmaxf(m, mb);
  const float a = ex2_approx(m - mn), b = ex2_approx(mb - mn);
  m = mn;
  d = fmaf(d, a, db * b);
#pragma unroll
  for (int c = 0; c < VPL; ++c) o[c] = fmaf(o[c], a, ob[c] * b);
}

template <int D>
__global__ void __launch_bounds__(256, 2) fa_prefix_scan_kernel(const ScanArgs a) {
  constexpr int VPL = D / 32;
  __shared__ float tot_m[8], tot_d[8];
  __shared__ __align__(16) float tot_o[8][D];
  __shared__ float car_m, car_d;  // carry of the windows so far (written by warp 7)
  __shared__ __align__(16) float car_o[D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H;
  const int S = a.S;                                  // chunks per row
  const int chunk = static_cast<int>(blockIdx.x) % S;
  const int rowid = static_cast<int>(blockIdx.x) / S;
  const int h = rowid % H;
  // Longest sequences first (ties by index), so the longest rows do not
  // start last: with up to kRankedSeqs sequences every CTA ranks the lengths
  // itself (a permutation for any values read); beyond that, index order.
  int b = rowid / H;
  if (a.B <= kRankedSeqs) {
    __shared__ int s_len[kRankedSeqs];
    __shared__ int s_seq;
    for (int i = threadIdx.x; i < a.B; i += blockDim.x)
      s_len[i] = __ldg(a.cu_seqlens_k + i + 1) - __ldg(a.cu_seqlens_k + i);
    __syncthreads();
    for (int i = threadIdx.x; i < a.B; i += blockDim.x) {
      const int li = s_len[i];
      int rank = 0;
      for (int j = 0; j < a.B; ++j) rank += (s_len[j] > li) || (s_len[j] == li && j < i);
      if (rank == b) s_seq = i;
    }
    __syncthreads();
    b = s_seq;
  }
  const int k_begin = __ldg(a.cu_seqlens_k + b);
  const int k_end = __ldg(a.cu_seqlens_k + b + 1);
  if (k_begin < 0 || k_end < k_begin || k_end > a.total_kv) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    return;
  }
  const int L = k_end - k_begin;
  // this CTA's keys: chunk `chunk` of S, [k0, k1) (the split-KV chunking)
  const int csize = (L + S - 1) / S;
  const int k0 = min(L, chunk * csize), k1 = min(L, (chunk + 1) * csize);
  const size_t stride = static_cast<size_t>(H) * D;
  const size_t col0 = static_cast<size_t>(h) * D + lane * VPL;
  const uint16_t* kp = static_cast<const uint16_t*>(a.k_cache) + k_begin * stride + col0;
  const uint16_t* vp = static_cast<const uint16_t*>(a.v_cache) + k_begin * stride + col0;
  uint16_t* op = static_cast<uint16_t*>(a.o) + k_begin * stride + col0;
  float* lp = a.lse + static_cast<size_t>(h) * a.total_kv + k_begin;
  float q[VPL];
  {
    const Cols<VPL> qc =
        ld_cols<VPL>(static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(b) * H + h) * D +
                     lane * VPL);
    to_f32<VPL>(qc, q);
  }
  const float c = a.scale_log2;
  // carry of all earlier keys: the fold of the earlier chunks' states (the
  // split-KV first pass), then of the earlier windows
  float cm = -INFINITY, cd = 0.f, co[VPL];
#pragma unroll
  for (int j = 0; j < VPL; ++j) co[j] = 0.f;
  if (chunk > 0) {
    const size_t row = (static_cast<size_t>(b) * H + h) * S;
    for (int c2 = 0; c2 < chunk; ++c2)
      merge_into<VPL>(cm, cd, co, a.part_m[row + c2], a.part_d[row + c2],
                      a.part_o + (row + c2) * D + lane * VPL);
  }

  // This warp's rows of window w0: K is consumed by the scores and V by the
  // rescan, so the next window's K is loaded right after the scores and its
  // V right after the rescan (the loads overlap the rest of the window).
  Cols<VPL> kr[kKeysPerWarp], vr[kKeysPerWarp];
  auto load_rows = [&](Cols<VPL>(&r)[kKeysPerWarp], const uint16_t* base, int w0) {
    const int kw = w0 + warp * kKeysPerWarp;
    const uint16_t* p = base + static_cast<size_t>(kw) * stride;
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i, p += stride)
      if (kw + i < k1) r[i] = ld_cols<VPL>(p);
  };
  load_rows(kr, kp, k0);
  load_rows(vr, vp, k0);
  for (int w0 = k0; w0 < k1; w0 += kWindow) {
    const int kw = w0 + warp * kKeysPerWarp;  // this warp's first key
    const int nk = max(0, min(kKeysPerWarp, k1 - kw));
    // phase A: scores and the segment total
    // Dot products: each lane's partial sums of the 16 keys, reduced across
    // the warp by halving -- at offset 16 a lane keeps 8 keys and adds its
    // partner's partials of those, at 8 it keeps 4, ... -- so that lane l
    // ends with the full sum of key l >> 1; then every lane takes all 16.
    float v[kKeysPerWarp];
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i) {
      float x[VPL];
      to_f32<VPL>(kr[i], x);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) s = fmaf(q[j], x[j], s);
      v[i] = s;
    }
#pragma unroll
    for (int w = kKeysPerWarp / 2, off = 16; w >= 1; w >>= 1, off >>= 1) {
      const bool hi = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < w; ++i) {
        const float send = hi ? v[i] : v[i + w];
        const float keep = hi ? v[i + w] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    float sg[kKeysPerWarp];
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i) {
      const float s = __shfl_sync(0xffffffffu, v[0], 2 * i);
      sg[i] = i < nk ? s * c : -INFINITY;
    }
    load_rows(kr, kp, w0 + kWindow);
    float lm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i) lm = fmaxf(lm, sg[i]);
    float ld = 0.f, lo[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) lo[j] = 0.f;
    if (nk > 0) {
#pragma unroll
      for (int i = 0; i < kKeysPerWarp; ++i) {
        const float p = ex2_approx(sg[i] - lm);  // 0 for the masked keys
        float x[VPL];
        to_f32<VPL>(vr[i], x);
        ld += p;
#pragma unroll
        for (int j = 0; j < VPL; ++j) lo[j] = fmaf(p, x[j], lo[j]);
      }
    }
    if (lane == 0) {
      tot_m[warp] = lm;
      tot_d[warp] = ld;
    }
#pragma unroll
    for (int j = 0; j < VPL; ++j) tot_o[warp][lane * VPL + j] = lo[j];
    __syncthreads();
    // phase B: carry-in, then every prefix of this warp's keys
    float m = cm, d = cd, o[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) o[j] = co[j];
    for (int w = 0; w < warp; ++w) merge_into<VPL>(m, d, o, tot_m[w], tot_d[w], &tot_o[w][lane * VPL]);
    // Lane i keeps key i's LSE and stores it after the rescan (one coalesced
    // store instead of a lane-0 store per key).
    float lse_mine = 0.f;
    uint16_t* dst = op + static_cast<size_t>(kw) * stride;
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i, dst += stride) {
      if (i < nk) {
        const float mn = fmaxf(m, sg[i]);
        const float al = ex2_approx(m - mn);  // m = -inf before the first key: 0
        const float p = ex2_approx(sg[i] - mn);
        float x[VPL];
        to_f32<VPL>(vr[i], x);
        d = fmaf(d, al, p);
        const float inv = __fdividef(1.f, d);
        uint32_t pk[VPL / 2];
#pragma unroll
        for (int j = 0; j < VPL; j += 2) {
          o[j] = fmaf(o[j], al, p * x[j]);
          o[j + 1] = fmaf(o[j + 1], al, p * x[j + 1]);
          pk[j / 2] = pack_bf16x2(o[j] * inv, o[j + 1] * inv);
        }
        m = mn;
        if constexpr (VPL == 4) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
        } else {
          *reinterpret_cast<uint32_t*>(dst) = pk[0];
        }
        const float lv = kLn2 * (m + __log2f(d));
        if (lane == i) lse_mine = lv;
      }
    }
    if (lane < nk) lp[kw + lane] = lse_mine;
    load_rows(vr, vp, w0 + kWindow);
    // The carry of the next window is warp 7's running state after its
    // rescan: the carry in (+) every key of this window.
    if (warp == 7) {
      if (lane == 0) {
        car_m = m;
        car_d = d;
      }
#pragma unroll
      for (int j = 0; j < VPL; ++j) car_o[lane * VPL + j] = o[j];
    }
    __syncthreads();  // the totals are rewritten by the next window
    cm = car_m;
    cd = car_d;
#pragma unroll
    for (int j = 0; j < VPL; ++j) co[j] = car_o[lane * VPL + j];
  }
}

}  // namespace

cudaError_t launch_prefix_scan(const ScanArgs& a, int D, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>(static_cast<long long>(a.B) * a.H * a.S);
  if (D == 128)
    fa_prefix_scan_kernel<128><<<blocks, 256, 0, stream>>>(a);
  else
    fa_prefix_scan_kernel<64><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
