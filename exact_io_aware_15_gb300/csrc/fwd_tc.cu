// Exact attention forward on the sm_103a tensor cores (bf16 in, fp32 state).
//
// One CTA owns one 128-row query tile of one (sequence, head) and folds the
// key/value tiles of that sequence into the per-row state (m, d, o) of
// "Learning FlashAttention the Hard Way - Part 1", sections "The State" and
// "The Merge, and the Twist", in the base-2 coordinates of "Alternative Twist:
// Base 2" (sigma = s * scale * log2 e, every exponential an ex2).  Each KV tile
// is one merge: the tile's own (max, sum, P V) is folded into the running
// state by rescaling the side with the smaller maximum.  Keys outside the
// sequence or above the causal diagonal get sigma = -inf, the identity's m,
// so they add nothing ("Associativity is All You Need": a neutral element
// pads the ragged tail).  The output division o / d and the log-sum-exp are
// deferred to the epilogue.  S and P live only in tensor memory.
//
// Reference maximum.  A state (m, d, o) stands for the same element of the
// monoid for any reference m (d 2^m and o 2^m do not change; "The Merge, and
// the Twist"), so a row moves its reference only when a tile's maximum
// exceeds it by more than kRescaleLog2 = 32 (base 2).  The reference never
// exceeds the running maximum, so d >= 1 as with the exact maximum
// ("Numerical Analysis of the FlashAttention Kernel"), and every weight p =
// 2^(sigma - m) is at most 2^32: fp32 d and o and bf16 P hold that as long
// as N * 2^32 * max|V| stays below fp32's range (|V| < 2^82 at N = 2^14).
// The O rescale between two P V products, which waits for the earlier one,
// is then needed almost never after a row's first tile, even for scores
// with a spread of many units (a warp rescales if any of its 32 rows moved).
// P is rounded to bf16 for the product; a weight that is not 1 then loses up
// to 2^-9 of itself, which for a row whose weight sits on one key would bias
// O by that much.  So O is divided by d less, per tile, what rounding took
// from the tile's largest weight (that weight is recomputed exactly as the
// tile loop computes it); the log-sum-exp uses d itself.
//
// Roles (224 threads):
//   warp 0      TMA producer: Q once, then K and V tiles into two rings of
//               stages, in the order the MMA issuers consume them
//               (K_0 .. K_{KS-1}, then V_j, K_{j+KS} for each j).
//   warp 1      QK issuer (one thread): S_j = Q K_j^T into TMEM S buffer
//               j % 3 (SS form), once K_j has landed and P_{j-3} V_{j-3} has
//               finished with that buffer.  With three S buffers the
//               products run up to two tiles ahead of the softmax, so the
//               softmax warps never wait for S.
//   warp 6      PV issuer (one thread): O += P_j V_j with P_j read from TMEM
//               (TS form, P_j over the second half of S buffer j % 3) once
//               the softmax has written P_j (and, on the rare tiles that
//               need it, rescaled O).  Two issuing threads keep the tensor
//               pipe fed: one thread issues an M=128 K=16 product about
//               every 80-90 cycles at best, while two threads together reach
//               one per ~65 cycles at N = 128, the pipe's own rate.
//   warps 2..5  softmax: thread t owns row 32*(warp%4) + lane; per tile it
//               loads its raw S row, masks, takes the row max (3-input max
//               instructions, sixteen independent chains), moves its
//               reference maximum if the tile's exceeds it by more than
//               kRescaleLog2, computes p = 2^(s c - m) with one packed fused
//               multiply-add per pair of columns, rounds P to bf16 over the
//               second half of the tile's S buffer (those scores are in
//               registers by then), sums p with packed adds (four chains),
//               and, on the
//               rare tiles where a row of the warp moved its reference,
//               waits for P_{j-1} V_{j-1} and rescales its O row in TMEM by
//               alpha_j = 2^(m_old - m_new) (the rescale half of the merge);
//               then it signals P_j.
//               Epilogue: O / d' in fp32 (d' = d less the largest weights'
//               rounding), LSE = ln2 (m + log2 d), stores (bf16 O at
//               D = 128: staged in Q's buffer, one TMA store per warp and
//               64-column half).
//
// Shared memory (1024-byte aligned): Q tile, KS K tiles, VS V tiles, the
// mbarriers.  A 128 x D bf16 tile is stored as D/64 column halves of
// 128 rows x 128 bytes, 128-byte swizzled (the TMA box layout and the
// canonical K-major / MN-major tcgen05 operand layouts).
// Tensor memory (512 columns): S buffers at [128 b, 128 b + 128) for b < 3
// (P_j, bf16 pairs, over columns [64, 128) of its buffer) and O at
// [384, 384 + D).

#include <cuda.h>
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {

// A row's reference maximum moves only when a tile's maximum exceeds it by
// more than this (base-2 units).
constexpr float kRescaleLog2 = 32.f;

template <int D>
struct TcCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int HALVES = D / 64;
  static constexpr uint32_t HALF_BYTES = 128u * 128u;
  static constexpr uint32_t TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int KS = 2;  // K ring stages
  static constexpr int VS = 3;  // V ring stages
  static constexpr int NS = 3;  // S buffers in TMEM (P_j is written over S_j)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KS * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VS * TILE_BYTES;
  // barrier indices, one per stage or buffer.  V_EMPTY(s) completes when the
  // P V product that read V stage s has finished; S_FULL(b) when Q K_j^T is
  // in S buffer b = j % NS, P_FULL(b) when the softmax warps have written
  // P_j over it, PV_DONE(b) when P_j V_j has finished (O holds it and S
  // buffer b is free for Q K_{j+NS}^T).
  static constexpr int B_Q_FULL = 0;
  static constexpr int B_K_FULL = 1;
  static constexpr int B_V_FULL = B_K_FULL + KS;
  static constexpr int B_K_EMPTY = B_V_FULL + VS;
  static constexpr int B_V_EMPTY = B_K_EMPTY + KS;
  static constexpr int B_S_FULL = B_V_EMPTY + VS;
  static constexpr int B_P_FULL = B_S_FULL + NS;
  static constexpr int B_PV_DONE = B_P_FULL + NS;
  static constexpr int B_DRAIN = B_PV_DONE + NS;  // one per issuing thread
  static constexpr int NUM_BARS = B_DRAIN + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TMEM_S = 0;    // buffer b at TMEM_S + 128 b
  static constexpr uint32_t TMEM_O = 384;
  static constexpr int THREADS = 224;
  static constexpr int WARP_PV = 6;
  static constexpr int SOFTMAX_THREADS = 128;
};

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Bounded wait used only while unwinding after an abort: ignores the abort
// flag (the copies or MMAs it waits for are already in flight) but still
// gives up after a short time.
__device__ __forceinline__ void mbar_wait_unwind(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;  // 200 ms
  }
}

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::THREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o, const TcFwdArgs args) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];

  // ---- which tile ----
  // A 1-D grid of (heads x query tiles).  Heads are taken in groups of four;
  // inside a group the heaviest query tiles (the longest causal KV ranges)
  // come first.  A group's K/V (4 heads x 8 MB at N = 16384, D = 128) stays
  // in L2 while its tiles run, and the light tiles fill the tail.
  const int nmb = args.num_mblocks;
  const int BHt = static_cast<int>(gridDim.x) / nmb;
  const long long lin = blockIdx.x;
  const long long per_group = 4LL * nmb;
  const int g = static_cast<int>(lin / per_group);
  const int gsize = min(4, BHt - g * 4);
  const int rr = static_cast<int>(lin - g * per_group);
  const int mb = nmb - 1 - rr / gsize;
  const int bh = g * 4 + rr % gsize;
  const int h = bh % args.H;
  const int seq = bh / args.H;
  const bool varlen = args.cu_seqlens != nullptr;
  int L, tok0;
  if (varlen) {
    const int a = __ldg(args.cu_seqlens + seq);
    const int e = __ldg(args.cu_seqlens + seq + 1);
    if (a < 0 || e < a || e > args.total_tokens || e - a > args.max_seqlen) {
      if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(args.status, kStatusBounds);
      return;
    }
    L = e - a;
    tok0 = a;
  } else {
    L = args.N;
    tok0 = 0;
  }
  if (mb * C::BM >= L) return;  // no query row of this sequence in the tile
  int n_kv = (L + C::BN - 1) / C::BN;
  if (args.causal) n_kv = min(n_kv, mb + 1);
  // With a sliding window the tile's rows see no key below
  // mb*BM - window + 1, so the KV tiles start at j0 (all later tile indices
  // j run from 0 and stand for KV tile j0 + j).
  int j0 = 0;
  if (args.window > 0) {
    const int lo = mb * C::BM - args.window + 1;
    j0 = lo > 0 ? lo / C::BN : 0;
  }
  n_kv -= j0;

  // ---- shared memory carve-up ----
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const unsigned long long wlim = args.wait_limit_ns ? args.wait_limit_ns : kWaitLimitNs;

  // TMA box origin of a 128-row tile starting at sequence position `row0`,
  // column half `c`.  Dense maps are (D, N, B*H); varlen maps are (D, H, T).
  auto tile_coords = [&](int c, int row0, int& c0, int& c1, int& c2) {
    c0 = c * 64;
    if (varlen) {
      c1 = h;
      c2 = tok0 + row0;
    } else {
      c1 = row0;
      c2 = bh;
    }
  };
  // One tile of K (is_v false) or V into its ring, after the product that
  // read the stage's previous tile has finished (issued by thread 0 only).
  auto load = [&](bool is_v, int j) -> bool {
    const int S = is_v ? C::VS : C::KS;
    const int st = j % S;
    if (j >= S && !mbar_wait(bar((is_v ? C::B_V_EMPTY : C::B_K_EMPTY) + st), ((j / S) - 1) & 1,
                             abort_flag, args.status, wlim))
      return false;
    // Fault injection (tests of the timeout path only): this key tile is
    // never requested, so its full barrier never completes.
    if (!is_v && j == args.skip_k_tile) return true;
    const uint32_t fb = bar((is_v ? C::B_V_FULL : C::B_K_FULL) + st);
    const uint32_t dst = sbase + (is_v ? C::OFF_V : C::OFF_K) + st * C::TILE_BYTES;
    mbar_arrive_expect_tx(fb, C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::HALVES; ++c) {
      int c0, c1, c2;
      tile_coords(c, (j0 + j) * C::BN, c0, c1, c2);
      tma_load_3d(dst + c * C::HALF_BYTES, is_v ? &tm_v : &tm_k, fb, c0, c1, c2);
    }
    return true;
  };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    mbar_init(bar(C::B_Q_FULL), 1);
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_K_FULL + s), 1);
      mbar_init(bar(C::B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_V_FULL + s), 1);
      mbar_init(bar(C::B_V_EMPTY + s), 1);
    }
    for (int b = 0; b < C::NS; ++b) {
      mbar_init(bar(C::B_S_FULL + b), 1);
      mbar_init(bar(C::B_P_FULL + b), C::SOFTMAX_THREADS);
      mbar_init(bar(C::B_PV_DONE + b), 1);
    }
    mbar_init(bar(C::B_DRAIN), 1);
    mbar_init(bar(C::B_DRAIN + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // The first copies need no free stage: start them before the CTA-wide
    // setup (TMEM allocation, barrier), so their latency overlaps it.
    const uint32_t qb = bar(C::B_Q_FULL);
    mbar_arrive_expect_tx(qb, C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::HALVES; ++c) {
      int c0, c1, c2;
      tile_coords(c, mb * C::BM, c0, c1, c2);
      tma_load_3d(sbase + C::OFF_Q + c * C::HALF_BYTES, &tm_q, qb, c0, c1, c2);
    }
    for (int jk = 0; jk < C::KS && jk < n_kv; ++jk) load(false, jk);
    load(true, 0);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      // Q, K_0 .. K_{KS-1} and V_0 were issued before the CTA barrier.
      int k_issued = min(n_kv, C::KS), v_issued = 1;
      for (int j = 0; j < n_kv; ++j) {
        if (j > 0) {
          if (!load(true, j)) break;
          v_issued = j + 1;
        }
        if (j + C::KS < n_kv) {
          if (!load(false, j + C::KS)) break;
          k_issued = j + C::KS + 1;
        }
      }
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        // Tiles before the last KS (VS) were waited for by the products
        // that freed their stages for the later tiles.
        mbar_wait_unwind(bar(C::B_Q_FULL), 0);
        for (int j = max(0, k_issued - C::KS); j < k_issued; ++j)
          if (j != args.skip_k_tile)  // never requested: nothing in flight
            mbar_wait_unwind(bar(C::B_K_FULL + j % C::KS), (j / C::KS) & 1);
        for (int j = max(0, v_issued - C::VS); j < v_issued; ++j)
          mbar_wait_unwind(bar(C::B_V_FULL + j % C::VS), (j / C::VS) & 1);
      }
    }
  } else if (warp == 1) {
    // ======================= QK issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
      const uint32_t q_s = sbase + C::OFF_Q;
      bool ok = mbar_wait(bar(C::B_Q_FULL), 0, abort_flag, args.status, wlim);
      for (int j = 0; ok && j < n_kv; ++j) {
        // S buffer j % NS is free once P_{j-NS} V_{j-NS}, which read the P
        // written over it, has finished (the softmax warps loaded S_{j-NS}
        // before writing that P).
        if (!mbar_wait(bar(C::B_K_FULL + j % C::KS), (j / C::KS) & 1, abort_flag,
                       args.status, wlim) ||
            (j >= C::NS && !mbar_wait(bar(C::B_PV_DONE + j % C::NS), ((j - C::NS) / C::NS) & 1,
                                      abort_flag, args.status, wlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_s = sbase + C::OFF_K + (j % C::KS) * C::TILE_BYTES;
        const uint32_t s_t = tmem + C::TMEM_S + 128u * (j % C::NS);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // 16-column slice kk of the head dimension: half kk/4, 32 bytes
          // per slice inside the 128-byte swizzled row.
          const uint32_t off = (kk >> 2) * C::HALF_BYTES + (kk & 3) * 32u;
          tc_mma_ss(s_t, sdesc_sw128(q_s + off, 16u, 1024u), sdesc_sw128(k_s + off, 16u, 1024u),
                    idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_S_FULL + j % C::NS));
        tc_commit(bar(C::B_K_EMPTY + j % C::KS));
      }
      // Every MMA this thread issued completes before TMEM is released.
      tc_commit(bar(C::B_DRAIN));
      mbar_wait_unwind(bar(C::B_DRAIN), 0);
    }
  } else if (warp == C::WARP_PV) {
    // ======================= PV issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      for (int j = 0; j < n_kv; ++j) {
        const int sv = j % C::VS;
        if (!mbar_wait(bar(C::B_P_FULL + j % C::NS), (j / C::NS) & 1, abort_flag, args.status, wlim) ||
            !mbar_wait(bar(C::B_V_FULL + sv), (j / C::VS) & 1, abort_flag, args.status, wlim))
          break;
        tc_fence_after();
        const uint32_t v_s = sbase + C::OFF_V + sv * C::TILE_BYTES;
        // P_j lies over the second half of S_j's buffer
        const uint32_t p_t = tmem + C::TMEM_S + 128u * (j % C::NS) + 64u;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          // B = V_j as an MN-major operand: N = D (64-column halves
          // HALF_BYTES apart), K = 16 keys starting at key 16*kk.
          const uint64_t bdesc = sdesc_sw128(v_s + kk * 16u * 128u, C::HALF_BYTES, 1024u);
          tc_mma_ts(tmem + C::TMEM_O, p_t + kk * 8u, bdesc, idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(C::B_V_EMPTY + sv));
        tc_commit(bar(C::B_PV_DONE + j % C::NS));
      }
      tc_commit(bar(C::B_DRAIN + 1));
      mbar_wait_unwind(bar(C::B_DRAIN + 1), 0);
    }
  } else {
    // ======================= softmax / epilogue =======================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qpos = mb * C::BM + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // sigma = s * c; with c = 0 every visible score is 0 and the masked ones
    // -inf, which c = 1 applied to (0 | -inf) reproduces without 0 * inf.
    const bool zero_scale = args.scale_log2 == 0.f;
    const float c = zero_scale ? 1.f : args.scale_log2;
    float m = -INFINITY;  // reference maximum (base 2)
    float dsum = 0.f;     // sum of the weights (for the log-sum-exp)
    float dnorm = 0.f;    // the same less the largest weights' rounding (divides O)
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      const int sb = j % C::NS;
      const uint32_t s_t = tmem + lane_off + C::TMEM_S + 128u * sb;
      const bool w = mbar_wait(bar(C::B_S_FULL + sb), (j / C::NS) & 1, abort_flag, args.status,
                               wlim);
      if (__any_sync(0xffffffffu, !w)) {
        ok = false;
        break;
      }
      tc_fence_after();

      float t[128];
      {
        uint32_t raw[64];
        tmem_ld64(s_t, raw);
#pragma unroll
        for (int i = 0; i < 64; ++i) t[i] = __uint_as_float(raw[i]);
        tmem_ld64(s_t + 64, raw);
#pragma unroll
        for (int i = 0; i < 64; ++i) t[64 + i] = __uint_as_float(raw[i]);
      }
      const int kbase = (j0 + j) * C::BN;
      const bool win_edge = args.window > 0 && kbase < mb * C::BM + C::BM - args.window;
      const bool masked = (args.causal && j0 + j == mb) || kbase + C::BN > L || win_edge;
      if (masked) {
        int lim = L - kbase;  // keys [lo, lim) of the tile are visible
        if (args.causal) lim = min(lim, qpos - kbase + 1);
        if (args.window > 0) {
          const int lo = qpos - args.window + 1 - kbase;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= lim || i < lo) t[i] = -INFINITY;
        } else {
          // Without a window the visible keys are a prefix: one compare.
#pragma unroll
          for (int i = 0; i < 128; ++i) t[i] = i < lim ? t[i] : -INFINITY;
        }
      }
      if (zero_scale) {
#pragma unroll
        for (int i = 0; i < 128; ++i) t[i] = (t[i] == -INFINITY) ? -INFINITY : 0.f;
      }
      // Row max over 128 values in 16 independent chains of 3-input maxima.
      float q[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = fmax3(t[8 * k], t[8 * k + 1], t[8 * k + 2]);
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = fmax3(q[k], t[8 * k + 3], t[8 * k + 4]);
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = fmax3(q[k], t[8 * k + 5], t[8 * k + 6]);
#pragma unroll
      for (int k = 0; k < 16; ++k) q[k] = fmaxf(q[k], t[8 * k + 7]);
      const float r0 = fmax3(q[0], q[1], q[2]), r1 = fmax3(q[3], q[4], q[5]);
      const float r2 = fmax3(q[6], q[7], q[8]), r3 = fmax3(q[9], q[10], q[11]);
      const float r4 = fmax3(q[12], q[13], q[14]);
      const float tmax = fmaxf(fmax3(r0, r1, r2), fmax3(r3, r4, q[15]));
      const float mx = tmax * c;
      const float m_new = (mx > m + kRescaleLog2) ? mx : m;  // also moves off -inf
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      // p = 2^(sigma - m_use), rounded to bf16 over the second half of S's
      // buffer (its scores are in registers), from where P_j V_j reads it.
      const uint32_t p_t = s_t + 64u;
      const float2 cc = make_float2(c, c), nm = make_float2(-m_use, -m_use);
      // Four packed sum chains keep the additions off each other's latency.
      float2 a[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) a[k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 x = __ffma2_rn(make_float2(t[64 * h + 2 * i], t[64 * h + 2 * i + 1]), cc, nm);
          const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          a[i & 3] = __fadd2_rn(a[i & 3], p);
          pk[i] = pack_bf16x2(p.x, p.y);
        }
        tmem_st32(p_t + 32u * h, pk);
      }
      const float alpha = (m_new == m) ? 1.f : ex2_approx(m - m_use);
      const float2 aa = __fadd2_rn(__fadd2_rn(a[0], a[1]), __fadd2_rn(a[2], a[3]));
      // The tile's largest weight as the loop computed it (same fused
      // multiply-add, same ex2) and what bf16 rounding took from it.
      const float pm = ex2_approx(fmaf(tmax, c, -m_use));
      const float pm_dropped = pm - __uint_as_float(pack_bf16x2(pm, 0.f) << 16);
      dnorm = dnorm * alpha + ((aa.x + aa.y) - pm_dropped);
      dsum = dsum * alpha + (aa.x + aa.y);
      m = m_new;

      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // o <- alpha * o between P_{j-1} V_{j-1} and P_j V_j (rare: only
        // when a row of this warp moved its reference maximum).
        const bool w2 = mbar_wait(bar(C::B_PV_DONE + (j - 1) % C::NS), ((j - 1) / C::NS) & 1,
                                  abort_flag, args.status, wlim);
        if (__any_sync(0xffffffffu, !w2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t o_t = tmem + lane_off + C::TMEM_O;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld32(o_t + c0, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(o_t + c0, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_P_FULL + sb));
    }

    if (ok) {
      const bool w = mbar_wait(bar(C::B_PV_DONE + (n_kv - 1) % C::NS),
                               ((n_kv - 1) / C::NS) & 1, abort_flag, args.status, wlim);
      if (!__any_sync(0xffffffffu, !w)) {
        tc_fence_after();
        const float inv = dnorm > 0.f ? 1.f / dnorm : 0.f;
        const float lse = dsum > 0.f ? (m + log2f(dsum)) * 0.69314718055994530942f : -INFINITY;
        const bool store = qpos < L;
        size_t orow, lidx;
        if (varlen) {
          const size_t t = static_cast<size_t>(tok0) + qpos;
          orow = t * args.H + h;
          lidx = static_cast<size_t>(h) * args.total_tokens + t;
        } else {
          orow = static_cast<size_t>(bh) * args.N + qpos;
          lidx = orow;
        }
        const uint32_t o_t = tmem + lane_off + C::TMEM_O;
        const int wrow0 = mb * C::BM + quarter * 32;  // this warp's first row
        if (D == 128 && args.o_tma && (varlen ? wrow0 + 32 <= L : wrow0 < L)) {
          // bf16 O through shared memory and one TMA store per 64-column half
          // and warp: the rows are staged in Q's buffer (no product reads Q
          // any more) in the 128-byte-swizzled box layout, and the tensor
          // map clips rows past the end of a dense sequence.  (A packed
          // sequence's last rows are followed by the next sequence's, so a
          // warp with rows past its end stores row by row below.)  At
          // D = 64 a row is 128 bytes and the row-by-row stores are faster.
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t ov[64];
            tmem_ld64(o_t + c0, ov);
            uint8_t* row = smem + C::OFF_Q + (c0 / 64) * C::HALF_BYTES + r * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              uint4 u;
              u.x = pack_bf16x2(__uint_as_float(ov[8 * ch + 0]) * inv,
                                __uint_as_float(ov[8 * ch + 1]) * inv);
              u.y = pack_bf16x2(__uint_as_float(ov[8 * ch + 2]) * inv,
                                __uint_as_float(ov[8 * ch + 3]) * inv);
              u.z = pack_bf16x2(__uint_as_float(ov[8 * ch + 4]) * inv,
                                __uint_as_float(ov[8 * ch + 5]) * inv);
              u.w = pack_bf16x2(__uint_as_float(ov[8 * ch + 6]) * inv,
                                __uint_as_float(ov[8 * ch + 7]) * inv);
              *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) << 4)) = u;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < C::HALVES; ++c) {
              const uint32_t src = sbase + C::OFF_Q + c * C::HALF_BYTES + quarter * 32 * 128;
              if (varlen)
                tma_store_3d(&tm_o, src, c * 64, h, tok0 + wrow0);
              else
                tma_store_3d(&tm_o, src, c * 64, wrow0, bh);
            }
            tma_store_commit_and_wait_read();
          }
          __syncwarp();
        } else {
          // 64 columns per TMEM load (one wait each), then the stores.
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 64) {
            uint32_t ov[64];
            tmem_ld64(o_t + c0, ov);
            if (store) {
              if (args.o_f32) {
                float4* dst =
                    reinterpret_cast<float4*>(static_cast<float*>(args.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv,
                                       __uint_as_float(ov[4 * i + 1]) * inv,
                                       __uint_as_float(ov[4 * i + 2]) * inv,
                                       __uint_as_float(ov[4 * i + 3]) * inv);
              } else {
                uint4* dst =
                    reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  uint4 u;
                  u.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv,
                                    __uint_as_float(ov[8 * i + 1]) * inv);
                  u.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv,
                                    __uint_as_float(ov[8 * i + 3]) * inv);
                  u.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv,
                                    __uint_as_float(ov[8 * i + 5]) * inv);
                  u.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv,
                                    __uint_as_float(ov[8 * i + 7]) * inv);
                  dst[i] = u;
                }
              }
            }
          }
        }
        if (store) args.lse[lidx] = lse;
      }
    }
    tc_fence_before();
  }

  // Role warps ran their loops in lane 0 alone: reconverge each warp before
  // the CTA barrier, which counts whole warps.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
static cudaError_t launch_tc_impl(const TcMaps& maps, const TcFwdArgs& a, int grid_x,
                                  cudaStream_t stream) {
  using C = TcCfg<D>;
  // The shared-memory opt-in is a per-device attribute of the function.
  static std::atomic<bool> attr_set[64];  // per device: attribute already set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(fa_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  dim3 grid(static_cast<unsigned>(grid_x * a.num_mblocks));
  fa_fwd_tc_kernel<D><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(maps.q, maps.k, maps.v, maps.o,
                                                                   a);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const TcMaps& maps, const TcFwdArgs& a, int D, int grid_x,
                          cudaStream_t stream) {
  if (D == 128) return launch_tc_impl<128>(maps, a, grid_x, stream);
  return launch_tc_impl<64>(maps, a, grid_x, stream);
}

}  // namespace fa
