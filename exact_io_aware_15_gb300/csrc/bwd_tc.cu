// Exact attention backward on the sm_103a tensor cores, by recomputation.
//
// "Understanding FlashAttention Pt 1: Personal Notes" (Introduction) sums the
// method up as tiling + online softmax + recomputation, and the review of
// "Learning FlashAttention the Hard Way - Part 1" names the backward pass
// that recomputes the attention weights instead of storing them.  Neither
// page prints the gradient formulas; they follow from the forward
// O = P V, P = softmax(S), S = scale Q K^T:
//     P_ij = 2^(sigma_ij - LSE2_i)      (sigma = s log2 e, LSE2 = LSE log2 e),
//     dV = P^T dO,   dP = dO V^T,   Delta_i = sum_d dO_id O_id,
//     dS = P * (dP - Delta),   dQ = scale dS K,   dK = scale dS^T Q.
// P is rebuilt tile by tile from the forward's log-sum-exp and never written
// to memory, like S in the forward.
//
// Three kernels, in stream order:
//   fa_bwd_delta_kernel  Delta = rowsum(dO * O) in fp32 (one warp per row).
//   fa_bwd_dkdv_kernel   one CTA per 128-key tile, streaming the query tiles
//                        that see it.  Thread = key row.
//   fa_bwd_dq_kernel     one CTA per 128-query tile, streaming the key tiles
//                        it sees.  Thread = query row.
// No atomics: every gradient row is owned by one CTA, so results are
// deterministic.  dK/dV and dQ each recompute S and dP (seven tile products
// per (query tile, key tile) pair instead of five) to keep it so.
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 MMA issuer (one
// thread), warps 2..5 elementwise and epilogue (TMEM lanes 32*(warp%4)..+31).
// The elementwise work of a tile is split in two phases with their own
// barriers -- P from S, then dS from dP -- and the MMA issue order lets the
// tensor cores run the next tile's products while the warps are busy:
//   dK/dV:  SS_S(0) SS_dP(0) | TS_dV(t) SS_S(t+1) TS_dK(t) SS_dP(t+1) | ...
//           TS_dV(t) waits for P(t), TS_dK(t) for dS(t).
//   dQ:     warp 1 issues SS_S(0) SS_dP(0) SS_S(1) | SS_dP(t+1) SS_S(t+2) | ...,
//           warp 6 TS_dQ(t) | ...; S is double-buffered in TMEM and dS(t)
//           is written over S(t).  TS_dQ(t) and SS_dP(t+1) both wait for
//           dS(t) (the warps have read dP(t) by then) and run at once, on two
//           issuing threads; SS_S(t+2) waits until TS_dQ(t) has read dS(t)
//           out of the buffer it overwrites.
// tcgen05.mma instructions of one thread execute in issue order, so a
// product that overwrites a TMEM region never overtakes an earlier one that
// reads it.  Every wait is bounded: on expiry the kernel records
// FA_ERR_DEVICE_TIMEOUT, lets in-flight copies and MMAs land, frees TMEM and
// returns.

#include <cuda.h>
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBM = 128;
constexpr uint32_t kHalfBytes = 128u * 128u;  // 128 rows x 64 bf16 columns
constexpr int kThreads = 192;     // dK/dV kernel
constexpr int kDqThreads = 224;   // dQ kernel: + the warp that issues TS_dQ
constexpr int kWarpAcc = 6;       // dQ: issues TS_dQ
constexpr int kElemThreads = 128;

__device__ __forceinline__ void mbar_wait_unwind_b(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;  // 200 ms
  }
}

// 32 lanes x 16 columns store (no wait).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Product over the head dimension: D(tmem) = A . B^T with both 128-row tiles
// K-major in shared memory (slice kk of 16 columns: half kk/4, 32 bytes per
// slice inside the 128-byte swizzled row).
template <int D>
__device__ __forceinline__ void mma_rows(uint32_t d_tmem, uint32_t a_s, uint32_t b_s) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32u;
    tc_mma_ss(d_tmem, sdesc_sw128(a_s + off, 16u, 1024u), sdesc_sw128(b_s + off, 16u, 1024u),
              idesc, kk > 0 ? 1u : 0u);
  }
}

// Accumulating product over the 128 rows of a streamed tile: D(tmem) (+)=
// A(tmem, bf16 pairs, 16 rows = 8 columns per step) . B, with B the tile as
// an MN-major operand (N = D, 64-column halves kHalfBytes apart, 16 rows =
// 2048 bytes per step).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_s,
                                        bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int kk = 0; kk < kBM / 16; ++kk)
    tc_mma_ts(d_tmem, a_tmem + kk * 8u, sdesc_sw128(b_s + kk * 2048u, kHalfBytes, 1024u),
              idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// Stores this thread's TMEM row of D fp32 columns, times `mult`, as one bf16
// row of dst (when `store`).
template <int D>
__device__ __forceinline__ void store_row(uint32_t tmem_row, void* dst, size_t row, bool store,
                                          float mult) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t ov[32];
    tmem_ld32(tmem_row + c0, ov);
    if (store) {
      uint4* out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + row * D + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 u;
        u.x = pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * mult,
                          __uint_as_float(ov[8 * i + 1]) * mult);
        u.y = pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * mult,
                          __uint_as_float(ov[8 * i + 3]) * mult);
        u.z = pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * mult,
                          __uint_as_float(ov[8 * i + 5]) * mult);
        u.w = pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * mult,
                          __uint_as_float(ov[8 * i + 7]) * mult);
        out[i] = u;
      }
    }
  }
}

// Which tile a CTA of the 1-D grid (heads x 128-row tiles) takes.  Heads go
// in groups of four and, inside a group, the heaviest tiles (under causal
// masking) first: the tensors the tiles stream (Q and dO, or K and V: 4
// heads x 8 MB at N = 16384, D = 128) stay in L2 while the group runs.
// Returns the head and the tile's rank by weight (0 = heaviest).
// (32-bit unsigned divisions: the grid has fewer than 2^31 CTAs, and a 64-bit
// division costs several hundred cycles.)
__device__ __forceinline__ void tile_of(int nt, int BH, int& bh, int& rank) {
  const unsigned lin = blockIdx.x;
  const unsigned per_group = 4u * static_cast<unsigned>(nt);
  const unsigned g = lin / per_group;
  const unsigned gsize = static_cast<unsigned>(min(4, BH - static_cast<int>(g) * 4));
  const unsigned rr = lin - g * per_group;
  const unsigned q = rr / gsize;
  rank = static_cast<int>(q);
  bh = static_cast<int>(g * 4u + (rr - q * gsize));
}

// Packed sequences: sequence s owns the tile slots [st(s), st(s+1)) with
// st(s) = cu[s] / 128 + s, at least its number of 128-row tiles, so the grid
// (H CTAs per slot) holds every tile of every sequence and one or two empty
// slots per sequence; inside a sequence the order is tile_of's.  Returns
// the (sequence, head) pair and the tile's rank by weight; a rank past the
// sequence's tiles marks an empty slot.  Offsets that fail the bounds check
// leave the CTA to seq_of's check.
__device__ __forceinline__ void slot_of(const BwdArgs& a, int& bh, int& rank) {
  constexpr int BM = 128;
  const unsigned Hu = static_cast<unsigned>(a.H);
  const unsigned lin = blockIdx.x;
  int lo = 0, hi = a.BH / a.H;  // the last sequence with st(s) * H <= lin
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    const long long st = __ldg(a.cu_seqlens + mid) / BM + mid;
    if (st * static_cast<long long>(Hu) <= static_cast<long long>(lin))
      lo = mid;
    else
      hi = mid;
  }
  const int seq = lo;
  const int b0 = __ldg(a.cu_seqlens + seq), b1 = __ldg(a.cu_seqlens + seq + 1);
  bh = seq * a.H;
  rank = 0x7fffffff;
  if (b0 < 0 || b1 < b0) return;  // seq_of reports it
  const unsigned st0 = static_cast<unsigned>(b0 / BM + seq);
  const unsigned slots = static_cast<unsigned>(b1 / BM + seq + 1) - st0;
  if (lin < st0 * Hu || lin - st0 * Hu >= slots * Hu) return;
  const unsigned local = lin - st0 * Hu;
  const unsigned g = local / (4u * slots);
  const unsigned gsize = static_cast<unsigned>(min(4, a.H - static_cast<int>(g) * 4));
  const unsigned rr = local - g * 4u * slots;
  const unsigned q = rr / gsize;
  rank = static_cast<int>(q);
  bh = seq * a.H + static_cast<int>(g * 4u + (rr - q * gsize));
}

// Where one (sequence, head) of the problem lives.  Dense: [B, H, N, D]
// tensors, LSE / Delta [B, H, N].  Varlen: packed [T, H, D] tensors,
// LSE / Delta [H, T], sequence s owning tokens [cu[s], cu[s+1]).
struct SeqView {
  bool ok;        // offsets passed the bounds check
  int L;          // positions of the sequence
  int h, tok0;    // varlen: head and first token
  size_t lse0;    // index of position 0 in LSE / Delta
  size_t row0;    // row of position 0 in the [., D] tensors
  size_t rstep;   // rows between consecutive positions
};

template <bool VAR>
__device__ __forceinline__ SeqView seq_of(const BwdArgs& a, int bh) {
  SeqView v;
  if constexpr (VAR) {
    const int seq = bh / a.H;
    v.h = bh % a.H;
    const int b0 = __ldg(a.cu_seqlens + seq), b1 = __ldg(a.cu_seqlens + seq + 1);
    v.ok = b0 >= 0 && b1 >= b0 && b1 <= a.total_tokens && b1 - b0 <= a.max_seqlen;
    v.L = v.ok ? b1 - b0 : 0;
    v.tok0 = v.ok ? b0 : 0;
    v.lse0 = static_cast<size_t>(v.h) * a.total_tokens + v.tok0;
    v.row0 = static_cast<size_t>(v.tok0) * a.H + v.h;
    v.rstep = static_cast<size_t>(a.H);
  } else {
    v.ok = true;
    v.L = a.N;
    v.h = 0;
    v.tok0 = 0;
    v.lse0 = static_cast<size_t>(bh) * a.N;
    v.row0 = v.lse0;
    v.rstep = 1;
  }
  return v;
}

// TMA box origin of 128 rows from sequence position `pos`, column half c:
// dense maps are (D, N, B*H), varlen maps (D, H, T).
template <bool VAR>
__device__ __forceinline__ void tile_load(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                          int halves, const SeqView& v, int bh, int pos) {
  for (int c = 0; c < halves; ++c) {
    if constexpr (VAR)
      tma_load_3d(dst + c * kHalfBytes, map, bar, c * 64, v.h, v.tok0 + pos);
    else
      tma_load_3d(dst + c * kHalfBytes, map, bar, c * 64, pos, bh);
  }
}

// ============================================================ dK / dV

template <int D>
struct DkdvCfg {
  static constexpr uint32_t TILE = (D / 64) * kHalfBytes;
  static constexpr int STAGES = (D == 128) ? 2 : 4;  // ring of (Q, dO) tile pairs
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = TILE;
  static constexpr uint32_t OFF_RING = 2 * TILE;  // stage s: Q at +2s*TILE, dO at +(2s+1)*TILE
  static constexpr uint32_t OFF_VEC = OFF_RING + STAGES * 2 * TILE;  // 4 warps x 256 floats
  static constexpr uint32_t OFF_BAR = OFF_VEC + 4 * 256 * 4;
  static constexpr int B_A_FULL = 0;
  static constexpr int B_FULL = 1;
  static constexpr int B_EMPTY = B_FULL + STAGES;
  static constexpr int B_S_FULL = B_EMPTY + STAGES;
  static constexpr int B_DP_FULL = B_S_FULL + 1;
  static constexpr int B_P_DONE = B_DP_FULL + 1;
  static constexpr int B_DS_DONE = B_P_DONE + 1;
  static constexpr int B_ACC_DONE = B_DS_DONE + 1;
  static constexpr int B_DRAIN = B_ACC_DONE + 1;
  static constexpr int NUM_BARS = B_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  // TMEM columns: S^T (then P^T in its first 64), dP^T (then dS^T), dV, dK
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384;
};

// One CTA per (head, 128-key tile n), in tile_of's order.
// Problem modes of the tile kernels: dense tensors zero-fill rows past N,
// whose contributions vanish without a mask; packed sequences mask the rows
// of the next sequence in a tail tile; the causal sliding window skips the
// tiles outside every row's window and masks the edge tiles.
constexpr int kDense = 0, kVarlen = 1, kWindow = 2;

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = args.num_tiles;
  constexpr bool VAR = MODE == kVarlen, WIN = MODE == kWindow;
  int bh, n;  // key tile n sees query tiles n..ntl-1 under causal masking
  if constexpr (VAR)
    slot_of(args, bh, n);
  else
    tile_of(nt, args.BH, bh, n);
  const SeqView sv = seq_of<VAR>(args, bh);
  if (!sv.ok) {
    if (threadIdx.x == 0) atomicOr(args.status, kStatusBounds);
    return;
  }
  const int ntl = (sv.L + kBM - 1) / kBM;  // tiles of this sequence
  if (n >= ntl) return;
  const int t_begin = args.causal ? n : 0;  // first query tile that sees key tile n
  // last query tile that sees key tile n: query i sees key j iff
  // j <= i < j + window under the window
  const int t_last =
      WIN ? min(ntl - 1, (n * kBM + kBM - 1 + args.window - 1) / kBM) : ntl - 1;
  const int count = t_last - t_begin + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_A_FULL), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    mbar_init(bar(C::B_P_DONE), kElemThreads);
    mbar_init(bar(C::B_DS_DONE), kElemThreads);
    mbar_init(bar(C::B_ACC_DONE), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      auto load = [&](const CUtensorMap* map, uint32_t dst, uint32_t fb, int row0) {
        tile_load<VAR>(map, dst, fb, D / 64, sv, bh, row0);
      };
      const uint32_t ab = bar(C::B_A_FULL);
      mbar_arrive_expect_tx(ab, 2 * C::TILE);
      load(&tm_k, sbase + C::OFF_K, ab, n * kBM);
      load(&tm_v, sbase + C::OFF_V, ab, n * kBM);
      int issued = 0;
      for (int t = 0; t < count; ++t) {
        const int s = t % C::STAGES;
        if (t >= C::STAGES &&
            !mbar_wait(bar(C::B_EMPTY + s), ((t / C::STAGES) - 1) & 1, abort_flag, args.status))
          break;
        const uint32_t fb = bar(C::B_FULL + s);
        mbar_arrive_expect_tx(fb, 2 * C::TILE);
        const uint32_t st = sbase + C::OFF_RING + 2u * s * C::TILE;
        load(&tm_q, st, fb, (t_begin + t) * kBM);
        load(&tm_do, st + C::TILE, fb, (t_begin + t) * kBM);
        issued = t + 1;
      }
      if (*abort_flag) {
        mbar_wait_unwind_b(bar(C::B_A_FULL), 0);
        for (int t = max(0, issued - C::STAGES); t < issued; ++t)
          mbar_wait_unwind_b(bar(C::B_FULL + t % C::STAGES), (t / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      const uint32_t k_s = sbase + C::OFF_K, v_s = sbase + C::OFF_V;
      auto q_of = [&](int t) { return sbase + C::OFF_RING + 2u * (t % C::STAGES) * C::TILE; };
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait(bar(b), parity, abort_flag, args.status);
      };
      bool ok = wait(C::B_A_FULL, 0) && wait(C::B_FULL, 0);
      if (ok) {
        tc_fence_after();
        mma_rows<D>(tmem + C::TM_S, k_s, q_of(0));             // S^T(0) = K Q_0^T
        tc_commit(bar(C::B_S_FULL));
        mma_rows<D>(tmem + C::TM_DP, v_s, q_of(0) + C::TILE);  // dP^T(0) = V dO_0^T
        tc_commit(bar(C::B_DP_FULL));
      }
      for (int t = 0; ok && t < count; ++t) {
        const uint32_t q_t = q_of(t);
        if (!wait(C::B_P_DONE, t & 1)) break;
        tc_fence_after();
        mma_acc<D>(tmem + C::TM_DV, tmem + C::TM_S, q_t + C::TILE, t > 0);  // dV += P^T dO_t
        if (t + 1 < count) {
          if (!wait(C::B_FULL + (t + 1) % C::STAGES, ((t + 1) / C::STAGES) & 1)) break;
          tc_fence_after();
          mma_rows<D>(tmem + C::TM_S, k_s, q_of(t + 1));
          tc_commit(bar(C::B_S_FULL));
        }
        if (!wait(C::B_DS_DONE, t & 1)) break;
        tc_fence_after();
        mma_acc<D>(tmem + C::TM_DK, tmem + C::TM_DP, q_t, t > 0);  // dK += dS^T Q_t
        tc_commit(bar(C::B_EMPTY + t % C::STAGES));
        if (t + 1 < count) {
          mma_rows<D>(tmem + C::TM_DP, v_s, q_of(t + 1) + C::TILE);
          tc_commit(bar(C::B_DP_FULL));
        }
      }
      tc_commit(bar(C::B_ACC_DONE));
      tc_commit(bar(C::B_DRAIN));
      mbar_wait_unwind_b(bar(C::B_DRAIN), 0);
    }
  } else {
    // ======================= elementwise / epilogue =======================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane = key row of the tile
    const int kj = n * kBM + r;         // key position
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // this warp's copy of the query tile's -LSE2 and -Delta
    float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC) + (warp - 2) * 256;
    const uint32_t s_t = tmem + lane_off + C::TM_S;
    const uint32_t dp_t = tmem + lane_off + C::TM_DP;
    const float2 cc = make_float2(args.scale_log2, args.scale_log2);
    bool ok = true;
    for (int t = 0; t < count; ++t) {
      const int tg = t_begin + t;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = lane + 32 * u;
        const int ig = tg * kBM + i;
        vec[i] = ig < sv.L ? -args.lse[sv.lse0 + ig] * kLog2e : 0.f;
        vec[128 + i] = ig < sv.L ? -args.delta[sv.lse0 + ig] : 0.f;
      }
      __syncwarp();
      // Masked: the causal diagonal tile, and query columns past the
      // sequence end (next sequence's rows when packed; key rows past the
      // end are not stored).
      const bool diag = args.causal && tg == n;
      // visible query columns: clo <= col < qlim (window: i - j < window,
      // i = tg*128 + col, j = n*128 + r)
      const int qlim = VAR ? sv.L - tg * kBM
                           : (WIN ? min(kBM, r + args.window - (tg - n) * kBM) : kBM);
      const bool masked =
          diag || (VAR && qlim < kBM) || (WIN && (tg - n) * kBM + kBM - 1 >= args.window);
      const int clo = diag ? r : 0;
      const bool w1 = mbar_wait(bar(C::B_S_FULL), t & 1, abort_flag, args.status);
      if (__any_sync(0xffffffffu, !w1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float p[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sr[32];
        tmem_ld32(s_t + 32u * ch, sr);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int col = 32 * ch + i;
          const float2 nl = *reinterpret_cast<const float2*>(vec + col);
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), cc, nl);
          float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          if constexpr (VAR || WIN) {
            if (masked) {
              if (col < clo || col >= qlim) p0 = 0.f;
              if (col + 1 < clo || col + 1 >= qlim) p1 = 0.f;
            }
          } else if (diag) {  // query tg*128+col sees key n*128+r iff col >= r
            if (col < r) p0 = 0.f;
            if (col + 1 < r) p1 = 0.f;
          }
          p[col] = p0;
          p[col + 1] = p1;
          pk[i / 2] = pack_bf16x2(p0, p1);
        }
        tmem_st16(s_t + 16u * ch, pk);  // P^T over the first 64 columns of S^T
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_P_DONE));

      const bool w2 = mbar_wait(bar(C::B_DP_FULL), t & 1, abort_flag, args.status);
      if (__any_sync(0xffffffffu, !w2)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t dr[32];
        tmem_ld32(dp_t + 32u * ch, dr);
        uint32_t dsk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int col = 32 * ch + i;
          const float2 nd = *reinterpret_cast<const float2*>(vec + 128 + col);
          const float2 g = __fadd2_rn(
              make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])), nd);
          const float2 ds = __fmul2_rn(make_float2(p[col], p[col + 1]), g);
          dsk[i / 2] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st16(dp_t + 16u * ch, dsk);  // dS^T over the first 64 columns of dP^T
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DS_DONE));
      __syncwarp();  // vec is rewritten for the next tile
    }

    if (ok) {
      const bool w3 = mbar_wait(bar(C::B_ACC_DONE), 0, abort_flag, args.status);
      if (!__any_sync(0xffffffffu, !w3)) {
        tc_fence_after();
        const bool store = kj < sv.L;
        const size_t row = sv.row0 + static_cast<size_t>(kj) * sv.rstep;
        store_row<D>(tmem + lane_off + C::TM_DV, args.dv, row, store, 1.f);
        store_row<D>(tmem + lane_off + C::TM_DK, args.dk, row, store, args.scale);
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
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================= dQ

template <int D>
struct DqCfg {
  static constexpr uint32_t TILE = (D / 64) * kHalfBytes;
  static constexpr int KS = (D == 128) ? 3 : 4;  // K ring (live from S(t) to dQ(t))
  static constexpr int VS = (D == 128) ? 2 : 4;  // V ring (live for dP(t) only)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + KS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + VS * TILE;
  static constexpr int B_A_FULL = 0;
  static constexpr int B_K_FULL = 1;
  static constexpr int B_K_EMPTY = B_K_FULL + KS;
  static constexpr int B_V_FULL = B_K_EMPTY + KS;
  static constexpr int B_V_EMPTY = B_V_FULL + VS;
  static constexpr int B_S_FULL = B_V_EMPTY + VS;  // two, one per S buffer
  static constexpr int B_DP_FULL = B_S_FULL + 2;
  static constexpr int B_DS_DONE = B_DP_FULL + 1;  // two: dS(t) in slot t % 2
  static constexpr int B_DQ_DONE = B_DS_DONE + 2;  // two: TS_dQ(t) finished, slot t % 2
  static constexpr int B_ACC_DONE = B_DQ_DONE + 2;
  static constexpr int B_DRAIN = B_ACC_DONE + 1;   // one per issuing thread
  static constexpr int NUM_BARS = B_DRAIN + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  // TMEM columns: S0, S1 (dS over the first 64 of the tile's buffer), dP, dQ
  static constexpr uint32_t TM_S0 = 0, TM_DP = 256, TM_DQ = 384;
};

// One CTA per (head, 128-query tile m), in tile_of's order.
template <int D, int MODE>
__global__ void __launch_bounds__(kDqThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = args.num_tiles;
  constexpr bool VAR = MODE == kVarlen, WIN = MODE == kWindow;
  int bh, rank;  // query tile m sees key tiles 0..m under causal masking
  if constexpr (VAR)
    slot_of(args, bh, rank);
  else
    tile_of(nt, args.BH, bh, rank);
  const SeqView sv = seq_of<VAR>(args, bh);
  if (!sv.ok) {
    if (threadIdx.x == 0) atomicOr(args.status, kStatusBounds);
    return;
  }
  const int ntl = (sv.L + kBM - 1) / kBM;  // tiles of this sequence
  // heaviest first: the last query tile of the sequence (of the longest one
  // for dense tensors, where every sequence has nt tiles)
  if (rank >= (VAR ? ntl : nt)) return;
  const int m = (VAR ? ntl : nt) - 1 - rank;
  if (m >= ntl) return;
  // key tiles j0 .. j0 + count - 1: under the window, query rows
  // m*128 .. m*128+127 see no key below m*128 - window + 1
  const int wlo = m * kBM - args.window + 1;
  const int j0 = (WIN && wlo > 0) ? wlo / kBM : 0;
  const int count = (args.causal ? m + 1 : ntl) - j0;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_A_FULL), 1);
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(bar(C::B_K_FULL + s), 1);
      mbar_init(bar(C::B_K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(bar(C::B_V_FULL + s), 1);
      mbar_init(bar(C::B_V_EMPTY + s), 1);
    }
    mbar_init(bar(C::B_S_FULL), 1);
    mbar_init(bar(C::B_S_FULL + 1), 1);
    mbar_init(bar(C::B_DP_FULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_DS_DONE + i), kElemThreads);
      mbar_init(bar(C::B_DQ_DONE + i), 1);
    }
    mbar_init(bar(C::B_ACC_DONE), 1);
    mbar_init(bar(C::B_DRAIN), 1);
    mbar_init(bar(C::B_DRAIN + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      auto load = [&](const CUtensorMap* map, uint32_t dst, uint32_t fb, int row0) {
        tile_load<VAR>(map, dst, fb, D / 64, sv, bh, row0);
      };
      const uint32_t ab = bar(C::B_A_FULL);
      mbar_arrive_expect_tx(ab, 2 * C::TILE);
      load(&tm_q, sbase + C::OFF_Q, ab, m * kBM);
      load(&tm_do, sbase + C::OFF_DO, ab, m * kBM);
      int k_issued = 0, v_issued = 0;
      for (int t = 0; t < count; ++t) {
        const int ks = t % C::KS;
        if (t >= C::KS &&
            !mbar_wait(bar(C::B_K_EMPTY + ks), ((t / C::KS) - 1) & 1, abort_flag, args.status))
          break;
        mbar_arrive_expect_tx(bar(C::B_K_FULL + ks), C::TILE);
        load(&tm_k, sbase + C::OFF_K + ks * C::TILE, bar(C::B_K_FULL + ks), (j0 + t) * kBM);
        k_issued = t + 1;
        const int vs = t % C::VS;
        if (t >= C::VS &&
            !mbar_wait(bar(C::B_V_EMPTY + vs), ((t / C::VS) - 1) & 1, abort_flag, args.status))
          break;
        mbar_arrive_expect_tx(bar(C::B_V_FULL + vs), C::TILE);
        load(&tm_v, sbase + C::OFF_V + vs * C::TILE, bar(C::B_V_FULL + vs), (j0 + t) * kBM);
        v_issued = t + 1;
      }
      if (*abort_flag) {
        mbar_wait_unwind_b(bar(C::B_A_FULL), 0);
        for (int t = max(0, k_issued - C::KS); t < k_issued; ++t)
          mbar_wait_unwind_b(bar(C::B_K_FULL + t % C::KS), (t / C::KS) & 1);
        for (int t = max(0, v_issued - C::VS); t < v_issued; ++t)
          mbar_wait_unwind_b(bar(C::B_V_FULL + t % C::VS), (t / C::VS) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      const uint32_t q_s = sbase + C::OFF_Q, do_s = sbase + C::OFF_DO;
      auto k_of = [&](int t) { return sbase + C::OFF_K + (t % C::KS) * C::TILE; };
      auto v_of = [&](int t) { return sbase + C::OFF_V + (t % C::VS) * C::TILE; };
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait(bar(b), parity, abort_flag, args.status);
      };
      auto issue_s = [&](int t) -> bool {  // S(t) = Q K_t^T into buffer t & 1
        if (!wait(C::B_K_FULL + t % C::KS, (t / C::KS) & 1)) return false;
        tc_fence_after();
        mma_rows<D>(tmem + C::TM_S0 + 128u * (t & 1), q_s, k_of(t));
        tc_commit(bar(C::B_S_FULL + (t & 1)));
        return true;
      };
      auto issue_dp = [&](int t) -> bool {  // dP(t) = dO V_t^T
        if (!wait(C::B_V_FULL + t % C::VS, (t / C::VS) & 1)) return false;
        tc_fence_after();
        mma_rows<D>(tmem + C::TM_DP, do_s, v_of(t));
        tc_commit(bar(C::B_DP_FULL));
        tc_commit(bar(C::B_V_EMPTY + t % C::VS));
        return true;
      };
      bool ok = wait(C::B_A_FULL, 0) && issue_s(0) && issue_dp(0) && (count < 2 || issue_s(1));
      for (int t = 0; ok && t + 1 < count; ++t) {
        // dP(t+1) once the warps have turned dP(t) into dS(t); S(t+2) once
        // TS_dQ(t) has read dS(t) out of S buffer t % 2.
        if (!wait(C::B_DS_DONE + (t & 1), (t >> 1) & 1) || !issue_dp(t + 1)) break;
        if (t + 2 < count &&
            (!wait(C::B_DQ_DONE + (t & 1), (t >> 1) & 1) || !issue_s(t + 2)))
          break;
      }
      tc_commit(bar(C::B_DRAIN));
      mbar_wait_unwind_b(bar(C::B_DRAIN), 0);
    }
  } else if (warp == kWarpAcc) {
    // ======================= accumulating product =======================
    if (lane == 0) {
      auto k_of = [&](int t) { return sbase + C::OFF_K + (t % C::KS) * C::TILE; };
      for (int t = 0; t < count; ++t) {
        if (!mbar_wait(bar(C::B_DS_DONE + (t & 1)), (t >> 1) & 1, abort_flag, args.status)) break;
        tc_fence_after();
        mma_acc<D>(tmem + C::TM_DQ, tmem + C::TM_S0 + 128u * (t & 1), k_of(t), t > 0);
        tc_commit(bar(C::B_DQ_DONE + (t & 1)));
        tc_commit(bar(C::B_K_EMPTY + t % C::KS));
      }
      tc_commit(bar(C::B_ACC_DONE));
      tc_commit(bar(C::B_DRAIN + 1));
      mbar_wait_unwind_b(bar(C::B_DRAIN + 1), 0);
    }
  } else {
    // ======================= elementwise / epilogue =======================
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane = query row of the tile
    const int qi = m * kBM + r;         // query position
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float nl2 = qi < sv.L ? -args.lse[sv.lse0 + qi] * kLog2e : 0.f;
    const float ndl = qi < sv.L ? -args.delta[sv.lse0 + qi] : 0.f;
    const float2 cc = make_float2(args.scale_log2, args.scale_log2);
    const float2 nl = make_float2(nl2, nl2), nd = make_float2(ndl, ndl);
    const uint32_t dp_t = tmem + lane_off + C::TM_DP;
    bool ok = true;
    for (int t = 0; t < count; ++t) {
      const uint32_t s_t = tmem + lane_off + C::TM_S0 + 128u * (t & 1);
      // Masked: the causal diagonal tile, and key columns past the sequence
      // end (next sequence's rows when packed).
      const int kt = j0 + t;  // key tile
      const bool diag = args.causal && kt == m;
      const int klim = VAR ? sv.L - kt * kBM : kBM;
      // visible key columns: klo <= col < khi (window: i - j < window,
      // i = m*128 + r, j = kt*128 + col)
      const int khi = diag ? min(klim, r + 1) : klim;
      const int klo = WIN ? (m - kt) * kBM + r - args.window + 1 : 0;
      const bool masked =
          diag || (VAR && klim < kBM) || (WIN && (m - kt) * kBM + kBM - 1 >= args.window);
      const bool w1 =
          mbar_wait(bar(C::B_S_FULL + (t & 1)), (t >> 1) & 1, abort_flag, args.status);
      if (__any_sync(0xffffffffu, !w1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float p[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sr[32];
        tmem_ld32(s_t + 32u * ch, sr);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int col = 32 * ch + i;
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), cc, nl);
          float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          if constexpr (VAR || WIN) {
            if (masked) {
              if (col < klo || col >= khi) p0 = 0.f;
              if (col + 1 < klo || col + 1 >= khi) p1 = 0.f;
            }
          } else if (diag) {  // key t*128+col is visible iff col <= r
            if (col > r) p0 = 0.f;
            if (col + 1 > r) p1 = 0.f;
          }
          p[col] = p0;
          p[col + 1] = p1;
        }
      }
      const bool w2 = mbar_wait(bar(C::B_DP_FULL), t & 1, abort_flag, args.status);
      if (__any_sync(0xffffffffu, !w2)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t dr[32];
        tmem_ld32(dp_t + 32u * ch, dr);
        uint32_t dsk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int col = 32 * ch + i;
          const float2 g = __fadd2_rn(
              make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])), nd);
          const float2 ds = __fmul2_rn(make_float2(p[col], p[col + 1]), g);
          dsk[i / 2] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st16(s_t + 16u * ch, dsk);  // dS over the first 64 columns of S(t)
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(C::B_DS_DONE + (t & 1)));
    }

    if (ok) {
      const bool w3 = mbar_wait(bar(C::B_ACC_DONE), 0, abort_flag, args.status);
      if (!__any_sync(0xffffffffu, !w3)) {
        tc_fence_after();
        store_row<D>(tmem + lane_off + C::TM_DQ, args.dq,
                     sv.row0 + static_cast<size_t>(qi) * sv.rstep, qi < sv.L, args.scale);
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
    tmem_dealloc(tmem, 512);
  }
}

// Delta_r = sum_d dO[r, d] O[r, d] in fp32; one warp per row.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_delta_kernel(const BwdArgs a) {
  constexpr int VPL = D / 32;  // bf16 values per lane (4 or 2)
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const uint16_t* o = static_cast<const uint16_t*>(a.o) + row * D + lane * VPL;
  const uint16_t* g = static_cast<const uint16_t*>(a.dout) + row * D + lane * VPL;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    s = fmaf(__uint_as_float(static_cast<uint32_t>(o[i]) << 16),
             __uint_as_float(static_cast<uint32_t>(g[i]) << 16), s);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    // dense: Delta [B, H, N] in row order; packed: row = t * H + h -> [H, T]
    const long long idx =
        a.cu_seqlens ? (row % a.H) * a.total_tokens + row / a.H : row;
    a.delta[idx] = s;
  }
}

static_assert(DkdvCfg<128>::SMEM_BYTES <= 232448, "dK/dV shared memory");
static_assert(DkdvCfg<64>::SMEM_BYTES <= 232448, "dK/dV shared memory");
static_assert(DqCfg<128>::SMEM_BYTES <= 232448, "dQ shared memory");
static_assert(DqCfg<64>::SMEM_BYTES <= 232448, "dQ shared memory");

template <int D, int MODE>
cudaError_t launch_impl(const BwdMaps& m, const BwdArgs& a, cudaStream_t stream) {
  static std::atomic<bool> attr_set[64];  // per device: attribute already set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(fa_bwd_dkdv_kernel<D, MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(DkdvCfg<D>::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fa_bwd_dq_kernel<D, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(DqCfg<D>::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  fa_bwd_delta_kernel<D><<<static_cast<unsigned>((a.rows + 7) / 8), 256, 0, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned blocks =
      MODE == kVarlen
          ? static_cast<unsigned>(a.H * (a.total_tokens / 128 + a.BH / a.H))
          : static_cast<unsigned>(static_cast<long long>(a.BH) * a.num_tiles);
  fa_bwd_dkdv_kernel<D, MODE>
      <<<blocks, kThreads, DkdvCfg<D>::SMEM_BYTES, stream>>>(m.q, m.k, m.v, m.dout, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_dq_kernel<D, MODE>
      <<<blocks, kDqThreads, DqCfg<D>::SMEM_BYTES, stream>>>(m.q, m.k, m.v, m.dout, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdMaps& maps, const BwdArgs& a, int D, cudaStream_t stream) {
  const int mode = a.cu_seqlens != nullptr ? kVarlen : (a.window > 0 ? kWindow : kDense);
  if (D == 128) {
    if (mode == kVarlen) return launch_impl<128, kVarlen>(maps, a, stream);
    if (mode == kWindow) return launch_impl<128, kWindow>(maps, a, stream);
    return launch_impl<128, kDense>(maps, a, stream);
  }
  if (mode == kVarlen) return launch_impl<64, kVarlen>(maps, a, stream);
  if (mode == kWindow) return launch_impl<64, kWindow>(maps, a, stream);
  return launch_impl<64, kDense>(maps, a, stream);
}

}  // namespace fa
