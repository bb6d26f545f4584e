// Exact attention forward on the sm_103a tensor cores (bf16 in, fp32 state).
//
// A work item is one 128-row query tile of one (sequence, head); a CTA takes
// one item (or, on persistent CTAs for short dense sequences, a sequence of
// them) and folds the key/value tiles of that sequence into the per-row
// state (m, d, o) of
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
// Roles at D = 128 (224 threads; at D = 64, 384 threads: two softmax groups
// of four warps split the key tiles between them, and each group has its own
// P V issuing thread, see TcCfg and the softmax section):
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
//               registers by then), sums p with packed adds (four chains).
//               (Dense one-item launches without a window compute the
//               weights against the current reference while the maximum is
//               reduced, and redo them in the rare tile where a row moves.)
//               On the rare tiles where a row of the warp moved its reference,
//               waits for P_{j-1} V_{j-1} and rescales its O row in TMEM by
//               alpha_j = 2^(m_old - m_new) (the rescale half of the merge);
//               then it signals P_j.
//               Epilogue: O / d' in fp32 (d' = d less the largest weights'
//               rounding), LSE = ln2 (m + log2 d), stores (bf16 O at
//               D = 128: staged in Q's buffer, one TMA store per warp and
//               64-column half).
//
// Shared memory (1024-byte aligned): two Q tiles (consecutive items), KS K
// tiles, VS V tiles, the mbarriers.  A 128 x D bf16 tile is stored as D/64 column halves of
// 128 rows x 128 bytes, 128-byte swizzled (the TMA box layout and the
// canonical K-major / MN-major tcgen05 operand layouts).
// Tensor memory (512 columns): S buffers at [128 b, 128 b + 128) for b < 3
// (P_j, bf16 pairs, over columns [64, 128) of its buffer) and O at
// [384, 384 + D); at D = 64 two S buffers at [0, 256), two P buffers at
// [256, 384) and the two groups' O at [384, 512).

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

// Sequences of at most this many 128-row query tiles run on persistent CTAs
// (measured crossovers: at D = 128 the one-item kernel, which computes weights
// before the maximum, wins from 24 tiles on; at D = 64, where its groups
// start P V on half of P and have one issuing thread each, from 20 tiles on).
constexpr int persistent_max_tiles(int D) { return D == 128 ? 20 : 16; }

// Softmax warpgroups per CTA at D = 64 (at D = 128 tensor memory holds one O).
constexpr int kSoftmaxGroups64 = 2;

// NG softmax warpgroups per CTA.  With two (D = 64), group g folds the key
// tiles j with j % 2 == g into its own state and O accumulator, and the
// epilogue merges the two states (split-K inside the CTA, "Associativity is
// All You Need"): each scheduler then runs two softmax warps on different
// tiles.  At D = 64 tensor memory then holds two S buffers, two separate P
// buffers and the two O accumulators: a group frees its S buffer for the
// product Q K_{j+2}^T as soon as it has read the scores, instead of when
// P_j V_j has finished.
template <int D, int NG = 1>
struct TcCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int HALVES = D / 64;
  static constexpr uint32_t HALF_BYTES = 128u * 128u;
  static constexpr uint32_t TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int KS = 2;  // K ring stages
  // V ring stages; with two groups, each group has two of them (its c-th
  // tile takes stage 2 g + c % 2), so a stage serves one group (and its P V
  // issuer) alone.
  static constexpr int VS = NG == 1 ? 3 : 4;
  // S buffers in TMEM: with one group P_j is written over S_j; with two,
  // group g has S buffer g and P buffer g (separate) for its tiles.
  static constexpr int NS = NG == 1 ? 3 : 2;
  static constexpr uint32_t OFF_Q = 0;  // two Q buffers (consecutive items)
  static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KS * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VS * TILE_BYTES;
  // barrier indices, one per stage or buffer.  V_EMPTY(s) completes when the
  // P V product that read V stage s has finished; S_FULL(b) when Q K_j^T is
  // in S buffer b (j % NS; with two groups the tile's group), P_FULL(b) when
  // the softmax warps have written P_j (over it, or into P buffer b),
  // PV_DONE(b) (one group) when P_j V_j has finished: O holds it and S
  // buffer b is free for Q K_{j+NS}^T.
  static constexpr int B_Q_FULL = 0;   // two: one per Q buffer
  static constexpr int B_Q_EMPTY = 2;  // two: the item's epilogue is done with it
  static constexpr int B_K_FULL = 4;
  static constexpr int B_V_FULL = B_K_FULL + KS;
  static constexpr int B_K_EMPTY = B_V_FULL + VS;
  static constexpr int B_V_EMPTY = B_K_EMPTY + KS;
  static constexpr int B_S_FULL = B_V_EMPTY + VS;
  static constexpr int B_P_FULL = B_S_FULL + NS;
  static constexpr int B_PV_DONE = B_P_FULL + NS;
  // PV_GRP(g): a P V product of softmax group g has finished (one phase per
  // product of that group; two groups only); XCH_FULL / XCH_DONE: the two
  // groups' epilogue
  // exchange (group 1's state is in shared memory and its O is final; group
  // 0 has read group 1's O).
  static constexpr int B_PV_GRP = B_PV_DONE + NS;
  static constexpr int B_XCH_FULL = B_PV_GRP + NG;
  static constexpr int B_XCH_DONE = B_XCH_FULL + 1;
  static constexpr int B_DRAIN = B_XCH_DONE + 1;  // one per issuing thread (three)
  // PH_FULL(b) (two groups, one item per CTA): P's second half (keys
  // 64..127) is in S buffer b, so P_j V_j may start on those keys while the
  // first half is computed.
  static constexpr int B_PH_FULL = B_DRAIN + 3;
  // S_FREE(b) (two groups): the softmax warps have read S_j out of S buffer
  // b, so Q K_{j+2}^T may overwrite it.
  static constexpr int B_S_FREE = B_PH_FULL + NS;
  static constexpr int NUM_BARS = B_S_FREE + NS;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_XCH = (OFF_MISC + 16 + 15) & ~15u;  // [128 rows][4] floats
  static constexpr uint32_t SMEM_BYTES = OFF_XCH + (NG > 1 ? 128 * 16 : 0) + 1024;  // + slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TMEM_S = 0;    // buffer b at TMEM_S + 128 b
  static constexpr uint32_t TMEM_P = 256;  // two groups: P buffer b at TMEM_P + 64 b
  static constexpr uint32_t TMEM_O = 384;  // group g's O at TMEM_O + g D
  static_assert(TMEM_O + NG * D <= TMEM_COLS, "S buffers and O accumulators exceed TMEM");
  static_assert(NG == 1 || (TMEM_S + 128 * NS <= TMEM_P && TMEM_P + 64 * NS <= TMEM_O),
                "S and P buffers overlap");
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory per CTA exceeded");
  static constexpr int WARP_PV = NG == 1 ? 6 : 2;
  static constexpr int WARP_SM0 = NG == 1 ? 2 : 4;  // first softmax warp
  // two groups: the P V issuer of group 1 (WARP_PV issues group 0's)
  static constexpr int WARP_PV1 = NG == 1 ? -1 : 3;
  static constexpr int THREADS = 32 * (NG == 1 ? 7 : 12);
  // Two groups: the issuing warps 0..3 form one warpgroup, the softmax groups
  // the other two.  A thread starts with REGS_LAUNCH registers (the most 384
  // threads can have); the issuing warpgroup then gives registers to the
  // softmax warpgroups, which hold a tile's 128 scores at once.  The split
  // may not exceed the CTA's pool, or the raise would wait forever; the
  // launcher checks that the compiled kernel starts with REGS_LAUNCH.
  static constexpr int REGS_LAUNCH = 168, REGS_ISSUE = 88, REGS_SOFTMAX = 200;
  static_assert(NG == 1 || (65536 / THREADS) / 8 * 8 == REGS_LAUNCH, "registers at launch");
  static_assert(NG == 1 || 128 * REGS_ISSUE + 256 * REGS_SOFTMAX <= THREADS * REGS_LAUNCH,
                "register split exceeds the CTA's pool");
  static constexpr int SOFTMAX_THREADS = 128;  // one group
};

// The item of CTA `lin` of a packed-sequence launch (one item per CTA).
// Sequence s owns the query-tile slots [st(s), st(s+1)) with st(s) =
// cu[s] / 128 + s, at least its number of query tiles, so the grid (H CTAs
// per slot) holds every tile of every sequence and one or two empty slots
// per sequence.  Inside a sequence the order is the dense one: groups of four
// heads, heaviest tile first.  n_kv = 0 marks an empty slot or offsets that
// fail the bounds check (reported once, by thread 0).
struct VarlenItem {
  int mb, bh, h, L, tok0, n_kv;
};
__device__ __forceinline__ VarlenItem varlen_item(const TcFwdArgs& args, unsigned lin) {
  constexpr int BM = 128;
  VarlenItem it{0, 0, 0, 0, 0, 0};
  const unsigned Hu = static_cast<unsigned>(args.H);
  int lo = 0, hi = args.num_seqs;  // the last sequence with st(s) * H <= lin
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    const long long st = __ldg(args.cu_seqlens + mid) / BM + mid;
    if (st * static_cast<long long>(Hu) <= static_cast<long long>(lin))
      lo = mid;
    else
      hi = mid;
  }
  const int seq = lo;
  const int a = __ldg(args.cu_seqlens + seq);
  const int e = __ldg(args.cu_seqlens + seq + 1);
  it.bh = seq * args.H;
  if (a < 0 || e < a || e > args.total_tokens || e - a > args.max_seqlen) {
    if (threadIdx.x == 0) atomicOr(args.status, kStatusBounds);
    return it;
  }
  const unsigned st0 = static_cast<unsigned>(a / BM + seq);
  const unsigned slots = static_cast<unsigned>(e / BM + seq + 1) - st0;
  if (lin < st0 * Hu || lin - st0 * Hu >= slots * Hu) return it;  // (inconsistent offsets)
  const unsigned local = lin - st0 * Hu;
  const unsigned g = local / (4u * slots);
  const unsigned gsize = static_cast<unsigned>(min(4, args.H - static_cast<int>(g) * 4));
  const unsigned rr = local - g * 4u * slots;
  const unsigned i = rr / gsize;  // rank by weight, 0 = heaviest
  const int h = static_cast<int>(g * 4u + (rr - i * gsize));
  const int L = e - a;
  const int tiles = (L + BM - 1) / BM;
  it.h = h;
  it.bh = seq * args.H + h;
  it.L = L;
  it.tok0 = a;
  if (static_cast<int>(i) >= tiles) return it;  // an empty slot
  it.mb = tiles - 1 - static_cast<int>(i);
  int n_kv = tiles;  // 128-key tiles (BN = BM)
  if (args.causal) n_kv = min(n_kv, it.mb + 1);
  it.n_kv = n_kv;
  return it;
}

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

// SPEC (one group, one item per CTA, no window): weights computed against
// the current reference while the tile maximum is reduced (see below).
// VL: packed sequences (cu_seqlens), one item per CTA.  WIN: the launch may
// have a sliding window (without it the window code folds away).
template <int D, bool PERSIST, int NG, bool SPEC, bool VL, bool WIN>
__global__ void __launch_bounds__(TcCfg<D, NG>::THREADS, 1)
    fa_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o, const TcFwdArgs args) {
  using C = TcCfg<D, NG>;
  extern __shared__ uint8_t smem_raw[];
  // Two groups, one item per CTA: P V products start on P's second half
  // (PH_FULL).  (The persistent instantiation keeps one signal per P: the
  // early rescale's registers cost it more than the split gains.)
  constexpr bool kHalfP = NG > 1 && !PERSIST;

  const int nmb = args.num_mblocks;
  const int BHt = args.num_items / nmb;  // (sequence, head) pairs
  constexpr bool varlen = VL;
  const int window = WIN ? args.window : 0;

  // ---- work items ----
  // An item is one 128-row query tile of one (sequence, head).  With one CTA
  // per item, CTA i takes item i of a head-grouped order: heads in groups of
  // four, inside a group the heaviest query tiles (the longest causal KV
  // ranges) first, so a group's K/V (4 heads x 8 MB at N = 16384, D = 128)
  // stays in L2 while its tiles run and the light tiles fill the tail.
  // Launched persistently (one CTA per SM, for short sequences), CTA c of P
  // takes the items at positions c, 2P-1-c, 2P+c, 4P-1-c, ... of a
  // heavy-first list (every head's last query tile first; the direction of
  // each round alternates, which evens out the causal loads), and the next
  // item's loads and first products overlap the current item's last tiles
  // and epilogue.
  struct Item {
    int mb, bh, h, L, tok0, n_kv, j0;
  };
  // The k-th item of this CTA; false when there is none.  An item whose
  // query tile holds no row of its sequence, or whose sequence offsets fail
  // the bounds check (reported once, by thread 0), gets n_kv = 0 and is
  // skipped by every role.
  auto item_at = [&](int k, Item& it) -> bool {
    // (32-bit unsigned divisions: num_items fits in an int, and the 64-bit
    // ones cost several hundred cycles at every item change)
    int mb = 0, bh = 0;
    if constexpr (PERSIST) {
      const unsigned P = gridDim.x;
      const unsigned c = blockIdx.x;
      if (static_cast<long long>(k) * P >= args.num_items) return false;
      const unsigned idx = static_cast<unsigned>(k) * P + ((k & 1) ? P - 1u - c : c);
      if (idx >= static_cast<unsigned>(args.num_items)) return false;
      const unsigned hq = idx / static_cast<unsigned>(BHt);
      mb = nmb - 1 - static_cast<int>(hq);
      bh = static_cast<int>(idx - hq * static_cast<unsigned>(BHt));
    } else if constexpr (VL) {
      if (k > 0) return false;
      const VarlenItem v = varlen_item(args, blockIdx.x);
      it.mb = v.mb;
      it.bh = v.bh;
      it.h = v.h;
      it.L = v.L;
      it.tok0 = v.tok0;
      it.n_kv = v.n_kv;
      it.j0 = 0;
      return true;
    } else {
      if (k > 0) return false;
      const unsigned lin = blockIdx.x;
      const unsigned per_group = 4u * static_cast<unsigned>(nmb);
      const unsigned g = lin / per_group;
      const unsigned gsize = static_cast<unsigned>(min(4, BHt - static_cast<int>(g) * 4));
      const unsigned rr = lin - g * per_group;
      const unsigned q = rr / gsize;
      mb = nmb - 1 - static_cast<int>(q);
      bh = static_cast<int>(g * 4u + (rr - q * gsize));
    }
    it.mb = mb;
    it.bh = bh;
    it.h = bh % args.H;
    it.n_kv = 0;
    it.j0 = 0;
    if (varlen) {
      const int seq = bh / args.H;
      const int a = __ldg(args.cu_seqlens + seq);
      const int e = __ldg(args.cu_seqlens + seq + 1);
      if (a < 0 || e < a || e > args.total_tokens || e - a > args.max_seqlen) {
        if (threadIdx.x == 0) atomicOr(args.status, kStatusBounds);
        return true;
      }
      it.L = e - a;
      it.tok0 = a;
    } else {
      it.L = args.N;
      it.tok0 = 0;
    }
    if (mb * C::BM >= it.L) return true;  // no query row of this sequence in the tile
    int n_kv = (it.L + C::BN - 1) / C::BN;
    if (args.causal) n_kv = min(n_kv, mb + 1);
    // With a sliding window the tile's rows see no key below
    // mb*BM - window + 1, so the KV tiles start at j0 (all later tile indices
    // j run from 0 and stand for KV tile j0 + j).
    if (window > 0) {
      const int lo = mb * C::BM - window + 1;
      it.j0 = lo > 0 ? lo / C::BN : 0;
    }
    it.n_kv = n_kv - it.j0;
    return true;
  };
  // Advances k to this CTA's next item with work; false when none is left.
  // (A CTA of the one-item launch has exactly one item: the loops below then
  // run once, with their counters known at compile time.)
  auto next_item = [&](int& k, Item& it) -> bool {
    if constexpr (!PERSIST) {
      if (k >= 0) return false;
    }
    while (item_at(++k, it))
      if (it.n_kv > 0) return true;
    return false;
  };
  // A CTA without any item leaves at once.
  int first_k = -1;
  Item first{};
  if (!next_item(first_k, first)) return;

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
  // Debug-build checks (fa_dbg_ok): a shared-memory range must lie in this
  // CTA's dynamic shared memory above the aligned base.
  const uint32_t smem_end = raw_addr + C::SMEM_BYTES;
  auto smem_ok = [&](uint32_t addr, uint32_t bytes) -> bool {
    return fa_dbg_ok(addr >= sbase && addr + bytes <= smem_end, args.status);
  };

  // TMA box origin of a 128-row tile of item `it` starting at sequence
  // position `row0`, column half `c`.  Dense maps are (D, N, B*H); varlen
  // maps are (D, H, T).
  auto tile_coords = [&](const Item& it, int c, int row0, int& c0, int& c1, int& c2) {
    c0 = c * 64;
    if (varlen) {
      c1 = it.h;
      c2 = it.tok0 + row0;
    } else {
      c1 = row0;
      c2 = it.bh;
    }
  };

  // ---- producer state (thread 0) ----
  // Loads are numbered per CTA across items: the K and V tiles of the g-th
  // KV step of the CTA go to ring stages g % KS and g % VS (with two groups
  // the c-th V tile of group gr to stage 2 gr + c % 2), the Q tile of the
  // t-th item to buffer t % 2.
  int k_issued = 0, q_issued = 0;
  int v_cnt0 = 0, v_cnt1 = 0;  // V tiles loaded for group 0 / 1 (two groups)
  uint32_t v_used = 0, v_par = 0;  // bit s: V stage s loaded; the parity of its last load
  uint32_t k_skipped = 0;  // bit s: stage s's last request was left out (fault injection)
  // The tile of KV step j of item `it` (global step g) into its ring, once
  // the product that read the stage's previous tile has finished.
  auto load_kv = [&](bool is_v, const Item& it, int j, int g) -> bool {
    const int S = is_v ? C::VS : C::KS;
    int st = g % S, n = g / S;  // stage, and this load's index among the stage's loads
    if (NG == 2 && is_v) {
      const int gr = j & 1;
      const int c = gr ? v_cnt1++ : v_cnt0++;
      st = 2 * gr + (c & 1);
      n = c >> 1;
    }
    if (n >= 1 && !mbar_wait(bar((is_v ? C::B_V_EMPTY : C::B_K_EMPTY) + st), (n - 1) & 1,
                             abort_flag, args.status, wlim))
      return false;
    if (is_v) {
      v_used |= 1u << st;
      v_par = (v_par & ~(1u << st)) | (static_cast<uint32_t>(n & 1) << st);
    } else {
      k_issued = g + 1;
      // Fault injection (tests of the timeout path only): this key tile is
      // never requested, so its full barrier never completes.
      if (j == args.skip_k_tile) {
        k_skipped |= 1u << st;
        return true;
      }
      k_skipped &= ~(1u << st);
    }
    const uint32_t fb = bar((is_v ? C::B_V_FULL : C::B_K_FULL) + st);
    const uint32_t dst = sbase + (is_v ? C::OFF_V : C::OFF_K) + st * C::TILE_BYTES;
    if (!smem_ok(dst, C::TILE_BYTES) || !smem_ok(fb, 8)) return true;
    mbar_arrive_expect_tx(fb, C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::HALVES; ++c) {
      int c0, c1, c2;
      tile_coords(it, c, (it.j0 + j) * C::BN, c0, c1, c2);
      tma_load_3d(dst + c * C::HALF_BYTES, is_v ? &tm_v : &tm_k, fb, c0, c1, c2);
    }
    return true;
  };
  // The Q tile of the t-th item, once the epilogue of item t-2 has released
  // its buffer.
  auto load_q = [&](const Item& it, int t) -> bool {
    const int qb = t & 1;
    if (t >= 2 && !mbar_wait(bar(C::B_Q_EMPTY + qb), ((t >> 1) - 1) & 1, abort_flag,
                             args.status, wlim))
      return false;
    q_issued = t + 1;
    const uint32_t fb = bar(C::B_Q_FULL + qb);
    if (!smem_ok(sbase + C::OFF_Q + qb * C::TILE_BYTES, C::TILE_BYTES) || !smem_ok(fb, 8))
      return true;
    mbar_arrive_expect_tx(fb, C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::HALVES; ++c) {
      int c0, c1, c2;
      tile_coords(it, c, it.mb * C::BM, c0, c1, c2);
      tma_load_3d(sbase + C::OFF_Q + qb * C::TILE_BYTES + c * C::HALF_BYTES, &tm_q, fb, c0, c1,
                  c2);
    }
    return true;
  };
  // An item's first copies: Q, K_0 .. K_{KS-1}, V_0 (global step g0).
  auto load_prologue = [&](const Item& it, int t, int g0) -> bool {
    if (!load_q(it, t)) return false;
    for (int jk = 0; jk < C::KS && jk < it.n_kv; ++jk)
      if (!load_kv(false, it, jk, g0 + jk)) return false;
    return load_kv(true, it, 0, g0);
  };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_Q_FULL + b), 1);
      mbar_init(bar(C::B_Q_EMPTY + b), C::SOFTMAX_THREADS);
    }
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
    for (int gr = 0; gr < NG; ++gr) mbar_init(bar(C::B_PV_GRP + gr), 1);
    mbar_init(bar(C::B_XCH_FULL), C::SOFTMAX_THREADS);
    mbar_init(bar(C::B_XCH_DONE), C::SOFTMAX_THREADS);
    for (int i = 0; i < 3; ++i) mbar_init(bar(C::B_DRAIN + i), 1);
    for (int b = 0; b < C::NS; ++b) {
      mbar_init(bar(C::B_PH_FULL + b), C::SOFTMAX_THREADS);
      mbar_init(bar(C::B_S_FREE + b), C::SOFTMAX_THREADS);
    }
    *abort_flag = 0;
    fence_mbar_init();
    // The first item's copies need no free stage: start them before the
    // CTA-wide setup (TMEM allocation, barrier), so their latency overlaps it.
    load_prologue(first, 0, 0);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // Debug-build check: a tensor-memory range (lanes x columns starting at
  // taddr = lane << 16 | column) must lie in this CTA's allocation.
  auto tmem_ok = [&](uint32_t taddr, uint32_t lanes, uint32_t cols) -> bool {
    const uint32_t col = taddr & 0xFFFFu, col0 = tmem & 0xFFFFu;
    return fa_dbg_ok((taddr >> 16) + lanes <= 128u && col >= col0 &&
                         col + cols <= col0 + C::TMEM_COLS,
                     args.status);
  };

  // The issuing warps (producer, QK issuer, P V issuers) and the softmax
  // warps; with two groups the former are one warpgroup, which gives
  // registers to the latter.
  const bool issuing = NG == 1 ? (warp < C::WARP_SM0 || warp == C::WARP_PV) : warp < 4;
  if (issuing) {
  if constexpr (NG == 2) regs_release<C::REGS_ISSUE>();
  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      int g0 = 0, ti = 0, k = first_k;
      bool ok = true;
      Item it = first;
      do {
        if (ti > 0 && !load_prologue(it, ti, g0)) break;
        for (int j = 0; j < it.n_kv; ++j) {
          if ((j > 0 && !load_kv(true, it, j, g0 + j)) ||
              (j + C::KS < it.n_kv && !load_kv(false, it, j + C::KS, g0 + j + C::KS))) {
            ok = false;
            break;
          }
        }
        g0 += it.n_kv;
        ++ti;
      } while (ok && next_item(k, it));
      if (*abort_flag) {
        // Let every copy this thread started land before the CTA exits.
        // Copies before the last two Q tiles, the last KS K tiles and the
        // last V tile of each stage were waited for by the products that
        // freed their buffers for the later ones.
        for (int i = max(0, q_issued - 2); i < q_issued; ++i)
          mbar_wait_unwind(bar(C::B_Q_FULL + (i & 1)), (i >> 1) & 1);
        for (int g = max(0, k_issued - C::KS); g < k_issued; ++g)
          if (!((k_skipped >> (g % C::KS)) & 1u))  // never requested: nothing in flight
            mbar_wait_unwind(bar(C::B_K_FULL + g % C::KS), (g / C::KS) & 1);
        for (int st = 0; st < C::VS; ++st)
          if ((v_used >> st) & 1u) mbar_wait_unwind(bar(C::B_V_FULL + st), (v_par >> st) & 1u);
      }
    }
  } else if (warp == 1) {
    // ======================= QK issuer =======================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
      int g0 = 0, ti = 0, k = first_k;
      int qc0 = 0, qc1 = 0;  // S products issued for group 0 / 1 (two groups)
      bool ok = true;
      Item it = first;
      do {
        const int qb = ti & 1;
        if (!mbar_wait(bar(C::B_Q_FULL + qb), (ti >> 1) & 1, abort_flag, args.status, wlim)) break;
        const uint32_t q_s = sbase + C::OFF_Q + qb * C::TILE_BYTES;
        for (int j = 0; j < it.n_kv; ++j) {
          const int g = g0 + j;
          // S buffer g % NS is free once P_{g-NS} V_{g-NS}, which read the P
          // written over it, has finished (the softmax warps loaded S_{g-NS}
          // before writing that P).  Two groups: the tile's group's buffer,
          // once that group has read its previous S.
          int sb = g % C::NS, sn = g / C::NS;  // buffer; this product's index among its products
          if constexpr (NG == 2) {
            sb = j & 1;
            sn = sb ? qc1++ : qc0++;
          }
          if (!mbar_wait(bar(C::B_K_FULL + g % C::KS), (g / C::KS) & 1, abort_flag,
                         args.status, wlim) ||
              (sn >= 1 && !mbar_wait(bar((NG == 1 ? C::B_PV_DONE : C::B_S_FREE) + sb),
                                     (sn - 1) & 1, abort_flag, args.status, wlim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_s = sbase + C::OFF_K + (g % C::KS) * C::TILE_BYTES;
          const uint32_t s_t = tmem + C::TMEM_S + 128u * sb;
          const bool in_range = smem_ok(q_s, C::TILE_BYTES) && smem_ok(k_s, C::TILE_BYTES) &&
                                tmem_ok(s_t, 128u, 128u);
#pragma unroll
          for (int kk = 0; kk < D / 16 && in_range; ++kk) {
            // 16-column slice kk of the head dimension: half kk/4, 32 bytes
            // per slice inside the 128-byte swizzled row.
            const uint32_t off = (kk >> 2) * C::HALF_BYTES + (kk & 3) * 32u;
            tc_mma_ss(s_t, sdesc_sw128(q_s + off, 16u, 1024u),
                      sdesc_sw128(k_s + off, 16u, 1024u), idesc_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(C::B_S_FULL + sb));
          tc_commit(bar(C::B_K_EMPTY + g % C::KS));
        }
        g0 += it.n_kv;
        ++ti;
      } while (ok && next_item(k, it));
      // Every MMA this thread issued completes before TMEM is released.
      tc_commit(bar(C::B_DRAIN));
      mbar_wait_unwind(bar(C::B_DRAIN), 0);
    }
  } else if (warp == C::WARP_PV || warp == C::WARP_PV1) {
    // ======================= PV issuer(s) =======================
    // Two groups: one issuing thread per group, each for the tiles j % 2 ==
    // pv of its group (its own P buffer, V stages and accumulator).  One
    // group: warp WARP_PV issues every product.
    constexpr int NPV = NG;
    const int pv = warp == C::WARP_PV ? 0 : 1;
    if (lane == 0 && pv < NPV) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      int g0 = 0, k = first_k;
      int pc = 0;  // products of this issuer so far (two groups)
      bool ok = true;
      Item it = first;
      do {
        for (int j = pv; j < it.n_kv; j += NPV) {
          const int g = g0 + j;
          // P buffer and V stage, and this tile's index among their tiles
          int pb = g % C::NS, pn = g / C::NS, sv = g % C::VS, vn = g / C::VS;
          if constexpr (NG == 2) {
            pb = pv;
            pn = pc;
            sv = 2 * pv + (pc & 1);
            vn = pc >> 1;
            ++pc;
          }
          // (split P: the products on P's second half wait only for it)
          if (!mbar_wait(bar((kHalfP ? C::B_PH_FULL : C::B_P_FULL) + pb), pn & 1, abort_flag,
                         args.status, wlim) ||
              !mbar_wait(bar(C::B_V_FULL + sv), vn & 1, abort_flag, args.status, wlim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_s = sbase + C::OFF_V + sv * C::TILE_BYTES;
          // P_j lies over the second half of S_j's buffer (one group) or in the
          // group's P buffer (two)
          const uint32_t p_t = NG == 1 ? tmem + C::TMEM_S + 128u * pb + 64u
                                       : tmem + C::TMEM_P + 64u * pb;
          // group j % NG's accumulator; its first product of the item
          // overwrites it (the previous item's epilogue has read it).
          const int grp = j % NG;
          const uint32_t o_acc = tmem + C::TMEM_O + grp * D;
          const bool in_range = smem_ok(v_s, C::TILE_BYTES) && tmem_ok(p_t, 128u, 64u) &&
                                tmem_ok(o_acc, 128u, D);
          // B = V_j as an MN-major operand: N = D (64-column halves
          // HALF_BYTES apart), K = 16 keys starting at key 16*kk.  The
          // item's first product overwrites O (the previous item's epilogue
          // has read it: its softmax warps wrote P_0 after).  With two
          // groups keys 64..127 go first, then 0..63 (with P split, once the
          // whole of P is in; both instantiations then add in one order).
          auto pv_steps = [&](int k0, int k1, bool first) {
#pragma unroll
            for (int kk = k0; kk < k1; ++kk) {
              if (!in_range) break;
              const uint64_t bdesc = sdesc_sw128(v_s + kk * 16u * 128u, C::HALF_BYTES, 1024u);
              tc_mma_ts(o_acc, p_t + kk * 8u, bdesc, idesc_pv,
                        (j >= NG || !first || kk > k0) ? 1u : 0u);
            }
          };
          if constexpr (NG == 1) {
            pv_steps(0, C::BN / 16, true);
          } else if constexpr (!kHalfP) {
            pv_steps(C::BN / 32, C::BN / 16, true);
            pv_steps(0, C::BN / 32, false);
          } else {
            pv_steps(C::BN / 32, C::BN / 16, true);
            if (!mbar_wait(bar(C::B_P_FULL + pb), pn & 1, abort_flag, args.status, wlim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv_steps(0, C::BN / 32, false);
          }
          tc_commit(bar(C::B_V_EMPTY + sv));
          // (two groups: nothing waits for PV_DONE; PV_GRP tells each group)
          if constexpr (NG == 1) tc_commit(bar(C::B_PV_DONE + pb));
          if constexpr (NG > 1) tc_commit(bar(C::B_PV_GRP + grp));
        }
        g0 += it.n_kv;
      } while (ok && next_item(k, it));
      tc_commit(bar(C::B_DRAIN + 1 + pv));
      mbar_wait_unwind(bar(C::B_DRAIN + 1 + pv), 0);
    }
  }
  } else {
    if constexpr (NG == 2) regs_acquire<C::REGS_SOFTMAX>();
    // ======================= softmax / epilogue =======================
    // Group grp of NG folds the key tiles j with j % NG == grp; warp w reads
    // TMEM lanes 32 (w % 4) ... + 31 (every group covers all 128 rows).
    const int grp = (warp - C::WARP_SM0) >> 2;
    int pvn = 0;  // P V products of this group so far (phases of PV_GRP(grp))
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // sigma = s * c; with c = 0 every visible score is 0 and the masked ones
    // -inf, which c = 1 applied to (0 | -inf) reproduces without 0 * inf.
    const bool zero_scale = args.scale_log2 == 0.f;
    const float c = zero_scale ? 1.f : args.scale_log2;
    bool ok = true;
    int g0 = 0, ti = 0, k = first_k;
    Item it = first;
    // Persistent CTAs: the Q buffer holding an item's O for TMA stores whose
    // read of it has not been waited for yet (-1: none).  Lane 0 of the warp
    // issued the stores; the buffer is released (Q_EMPTY) after the wait.
    int q_release = -1;
    auto release_q = [&]() {
      if (lane == 0) tma_store_wait_read();
      __syncwarp();
      tc_fence_before();
      mbar_arrive(bar(C::B_Q_EMPTY + q_release));
      q_release = -1;
    };
    do {
      const int mb = it.mb, L = it.L, j0 = it.j0, n_kv = it.n_kv;
      const int qpos = mb * C::BM + r;
      float m = -INFINITY;  // reference maximum (base 2)
      float dsum = 0.f;     // sum of the weights (for the log-sum-exp)
      float dnorm = 0.f;    // the same less the largest weights' rounding (divides O)

      for (int j = grp; j < n_kv; j += NG) {
        const int g = g0 + j;
        // S buffer (two groups: the group's own, its pvn-th S)
        const int sb = NG == 1 ? g % C::NS : grp;
        const uint32_t s_t = tmem + lane_off + C::TMEM_S + 128u * sb;
        const bool w = mbar_wait(bar(C::B_S_FULL + sb), (NG == 1 ? g / C::NS : pvn) & 1,
                                 abort_flag, args.status, wlim);
        if (__any_sync(0xffffffffu, !w)) {
          ok = false;
          break;
        }
        tc_fence_after();

        const int kbase = (j0 + j) * C::BN;
        const bool win_edge = window > 0 && kbase < mb * C::BM + C::BM - window;
        const bool masked = (args.causal && j0 + j == mb) || kbase + C::BN > L || win_edge;
        float tmax, m_new, m_use;
        // p = 2^(sigma - m_use), rounded to bf16 over the second half of S's
        // buffer (its scores are in registers) or, with two groups, into P
        // buffer sb, from where P_j V_j reads it.
        const uint32_t p_t =
            NG == 1 ? s_t + 64u : tmem + lane_off + C::TMEM_P + 64u * static_cast<uint32_t>(sb);
        const bool p_ok = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(p_t, 32u, 64u));
        // Four packed sum chains keep the additions off each other's latency.
        float2 a[4];
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) a[kq] = make_float2(0.f, 0.f);
        if constexpr (NG == 1) {
          float t[128];
          if (!kDebugChecks || __all_sync(0xffffffffu, tmem_ok(s_t, 32u, 128u))) {
            uint32_t raw[64];
            tmem_ld64(s_t, raw);
  #pragma unroll
            for (int i = 0; i < 64; ++i) t[i] = __uint_as_float(raw[i]);
            tmem_ld64(s_t + 64, raw);
  #pragma unroll
            for (int i = 0; i < 64; ++i) t[64 + i] = __uint_as_float(raw[i]);
          } else {
  #pragma unroll
            for (int i = 0; i < 128; ++i) t[i] = 0.f;
          }
          if (masked) {
            int lim = L - kbase;  // keys [lo, lim) of the tile are visible
            if (args.causal) lim = min(lim, qpos - kbase + 1);
            if (window > 0) {
              const int lo = qpos - window + 1 - kbase;
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
          auto tile_max = [&]() -> float {
            float q[16];
  #pragma unroll
            for (int kq = 0; kq < 16; ++kq) q[kq] = fmax3(t[8 * kq], t[8 * kq + 1], t[8 * kq + 2]);
  #pragma unroll
            for (int kq = 0; kq < 16; ++kq) q[kq] = fmax3(q[kq], t[8 * kq + 3], t[8 * kq + 4]);
  #pragma unroll
            for (int kq = 0; kq < 16; ++kq) q[kq] = fmax3(q[kq], t[8 * kq + 5], t[8 * kq + 6]);
  #pragma unroll
            for (int kq = 0; kq < 16; ++kq) q[kq] = fmaxf(q[kq], t[8 * kq + 7]);
            const float r0 = fmax3(q[0], q[1], q[2]), r1 = fmax3(q[3], q[4], q[5]);
            const float r2 = fmax3(q[6], q[7], q[8]), r3 = fmax3(q[9], q[10], q[11]);
            const float r4 = fmax3(q[12], q[13], q[14]);
            return fmaxf(fmax3(r0, r1, r2), fmax3(r3, r4, q[15]));
          };
          // p = 2^(sigma - mu) for the tile, summed into a[] and stored as P.
          auto tile_exp = [&](float mu) {
            const float2 cc = make_float2(c, c), nm = make_float2(-mu, -mu);
  #pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t pk[32];
  #pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float2 x =
                    __ffma2_rn(make_float2(t[64 * hh + 2 * i], t[64 * hh + 2 * i + 1]), cc, nm);
                const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                a[i & 3] = __fadd2_rn(a[i & 3], p);
                pk[i] = pack_bf16x2(p.x, p.y);
              }
              if (p_ok) tmem_st32(p_t + 32u * hh, pk);
            }
          };
          // Once every row of the warp has a reference, the reference moves
          // only when the tile's maximum exceeds it by kRescaleLog2: the
          // weights are computed against the current reference while the
          // maximum is reduced, and recomputed in the rare tile where a row
          // moves (all lanes store P, so the warp redoes it together).  (One
          // item per CTA without a window only: in the persistent and the
          // window instantiations the second copy of the exponential loop
          // costs more registers and code than it gains.)
          if (SPEC && __all_sync(0xffffffffu, m != -INFINITY)) {
            m_use = m;
            tile_exp(m_use);
            tmax = tile_max();
            const float mx = tmax * c;
            m_new = (mx > m + kRescaleLog2) ? mx : m;
            if (__any_sync(0xffffffffu, m_new != m)) {
              m_use = m_new;
  #pragma unroll
              for (int kq = 0; kq < 4; ++kq) a[kq] = make_float2(0.f, 0.f);
              tile_exp(m_use);
            }
          } else {
            tmax = tile_max();
            const float mx = tmax * c;
            m_new = (mx > m + kRescaleLog2) ? mx : m;  // also moves off -inf
            m_use = (m_new == -INFINITY) ? 0.f : m_new;
            tile_exp(m_use);
          }
        } else {
          // The issuing warpgroup gave the softmax warps the registers to
          // hold a tile's 128 scores: one read of S, after which S buffer sb
          // is released for Q K_{j+2}^T, then the row maximum, then the
          // weights of keys 64..127 (into columns 32..63 of P buffer sb) and
          // of keys 0..63.
          const bool s_in = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(s_t, 32u, 128u));
          float t[128];
          if (s_in) {
            uint32_t raw[64];
            tmem_ld64(s_t, raw);
#pragma unroll
            for (int i = 0; i < 64; ++i) t[i] = __uint_as_float(raw[i]);
            tmem_ld64(s_t + 64u, raw);
#pragma unroll
            for (int i = 0; i < 64; ++i) t[64 + i] = __uint_as_float(raw[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 128; ++i) t[i] = 0.f;
          }
          // S_j has been read (the loads waited for their data).
          tc_fence_before();
          mbar_arrive(bar(C::B_S_FREE + sb));
          if (masked) {
            int lim = L - kbase;  // the row's visible keys of the tile: [lo, lim)
            if (args.causal) lim = min(lim, qpos - kbase + 1);
            const int lo = window > 0 ? qpos - window + 1 - kbase : -1;
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i >= lim || i < lo) t[i] = -INFINITY;
          }
          if (zero_scale) {
#pragma unroll
            for (int i = 0; i < 128; ++i) t[i] = (t[i] == -INFINITY) ? -INFINITY : 0.f;
          }
          float q[16];
#pragma unroll
          for (int kq = 0; kq < 16; ++kq) {
            q[kq] = fmax3(t[8 * kq], t[8 * kq + 1], t[8 * kq + 2]);
            q[kq] = fmax3(q[kq], t[8 * kq + 3], t[8 * kq + 4]);
            q[kq] = fmax3(q[kq], t[8 * kq + 5], t[8 * kq + 6]);
            q[kq] = fmaxf(q[kq], t[8 * kq + 7]);
          }
          const float r0 = fmax3(q[0], q[1], q[2]), r1 = fmax3(q[3], q[4], q[5]);
          const float r2 = fmax3(q[6], q[7], q[8]), r3 = fmax3(q[9], q[10], q[11]);
          const float r4 = fmax3(q[12], q[13], q[14]);
          tmax = fmaxf(fmax3(r0, r1, r2), fmax3(r3, r4, q[15]));
          const float mx = tmax * c;
          m_new = (mx > m + kRescaleLog2) ? mx : m;  // also moves off -inf
          m_use = (m_new == -INFINITY) ? 0.f : m_new;
          const float2 cc = make_float2(c, c), nm = make_float2(-m_use, -m_use);
          // keys base .. base + 63 (pair i into a[i % 4])
          auto exp_half = [&](int base, uint32_t (&pk)[32]) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 xv =
                  __ffma2_rn(make_float2(t[base + 2 * i], t[base + 2 * i + 1]), cc, nm);
              const float2 p = make_float2(ex2_approx(xv.x), ex2_approx(xv.y));
              a[i & 3] = __fadd2_rn(a[i & 3], p);
              pk[i] = pack_bf16x2(p.x, p.y);
            }
          };
          uint32_t pk[32];
          exp_half(64, pk);
          // The group's P buffer holds its previous P, whose product must
          // have read it: that product is confirmed here (within the item;
          // the item's epilogue confirmed the last one of the previous item),
          // and with P split O is rescaled now, before P_j V_j can start on
          // P's second half.
          if (kHalfP && j >= NG) {
            const bool w2 = mbar_wait(bar(C::B_PV_GRP + grp), (pvn - 1) & 1, abort_flag,
                                      args.status, wlim);
            if (__any_sync(0xffffffffu, !w2)) {
              ok = false;
              break;
            }
            const float alpha_g = (m_new == m) ? 1.f : ex2_approx(m - m_use);
            if (__any_sync(0xffffffffu, alpha_g != 1.f)) {
              tc_fence_after();
              const uint32_t o_t = tmem + lane_off + C::TMEM_O + grp * D;
              const bool o_ok = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(o_t, 32u, D));
#pragma unroll
              for (int c0 = 0; c0 < D && o_ok; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32(o_t + c0, ov);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha_g);
                tmem_st32(o_t + c0, ov);
              }
            }
          } else if (!kHalfP && j >= NG) {
            const bool w2 = mbar_wait(bar(C::B_PV_GRP + grp), (pvn - 1) & 1, abort_flag,
                                      args.status, wlim);
            if (__any_sync(0xffffffffu, !w2)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          if (p_ok) tmem_st32(p_t + 32u, pk);
          if constexpr (kHalfP) {
            tmem_st_wait();  // (also the rescaled O)
            tc_fence_before();
            mbar_arrive(bar(C::B_PH_FULL + sb));
          }
          exp_half(0, pk);
          if (p_ok) tmem_st32(p_t, pk);
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

        if (!kHalfP && j >= NG && __any_sync(0xffffffffu, alpha != 1.f)) {
          // o <- alpha * o between the group's previous P V product and
          // P_j V_j (rare: only when a row of this warp moved its reference
          // maximum; with P split this happened before the exponentials).
          // With one group that product's S buffer barrier is waited for
          // (its next phase needs this warp's P, so it cannot run ahead of
          // the wait); with two, the product was confirmed above.
          if constexpr (NG == 1) {
            const bool w2 = mbar_wait(bar(C::B_PV_DONE + (g - 1) % C::NS),
                                      ((g - 1) / C::NS) & 1, abort_flag, args.status, wlim);
            if (__any_sync(0xffffffffu, !w2)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t o_t = tmem + lane_off + C::TMEM_O + grp * D;
          const bool o_ok = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(o_t, 32u, D));
#pragma unroll
          for (int c0 = 0; c0 < D && o_ok; c0 += 32) {
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
        ++pvn;
        if constexpr (PERSIST && NG == 1) {
          // the previous item's staged O: its TMA stores have read it by now
          if (q_release >= 0) release_q();
        }
      }
      if (!ok) break;

      // ---- epilogue of the item ----
      // (the row's scalars first: they need only the state, and overlap the
      // wait for the last product)
      const int qb = ti & 1;
      const float inv = dnorm > 0.f ? 1.f / dnorm : 0.f;
      const float lse = dsum > 0.f ? (m + log2f(dsum)) * 0.69314718055994530942f : -INFINITY;
      const bool store = qpos < L;
      size_t orow, lidx;
      if (varlen) {
        const size_t tk = static_cast<size_t>(it.tok0) + qpos;
        orow = tk * args.H + it.h;
        lidx = static_cast<size_t>(it.h) * args.total_tokens + tk;
      } else {
        orow = static_cast<size_t>(it.bh) * args.N + qpos;
        lidx = orow;
      }
      // The group's last P V product of the item (none for a group beyond
      // the item's tile count): with one group, through the S buffer
      // barrier of the item's last step; with two, through the group's
      // barrier (its earlier products were confirmed tile by tile).
      if (n_kv > grp) {
        bool w;
        if constexpr (NG == 1) {
          const int gl = g0 + n_kv - 1;
          w = mbar_wait(bar(C::B_PV_DONE + gl % C::NS), (gl / C::NS) & 1, abort_flag,
                        args.status, wlim);
        } else {
          w = mbar_wait(bar(C::B_PV_GRP + grp), (pvn - 1) & 1, abort_flag, args.status, wlim);
        }
        if (__any_sync(0xffffffffu, !w)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      if constexpr (NG == 2) {
        // Two partial states per row: group 0 (here) and group 1, whose
        // (m, dsum, dnorm) come through shared memory and whose O is read
        // from its TMEM accumulator once final.  They merge by the rule of
        // "The Merge, and the Twist": both sides rescaled to the larger
        // reference.  Rows are stored one by one (D = 64).
        float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
        if (grp == 1) {
          xch[4 * r + 0] = m;
          xch[4 * r + 1] = dsum;
          xch[4 * r + 2] = dnorm;
          tc_fence_before();
          mbar_arrive(bar(C::B_XCH_FULL));
          // Group 0 reads this group's O before its next item overwrites it.
          const bool w3 = mbar_wait(bar(C::B_XCH_DONE), ti & 1, abort_flag, args.status, wlim);
          if (__any_sync(0xffffffffu, !w3)) {
            ok = false;
            break;
          }
        } else {
          const bool w3 = mbar_wait(bar(C::B_XCH_FULL), ti & 1, abort_flag, args.status, wlim);
          if (__any_sync(0xffffffffu, !w3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool has1 = n_kv > 1;  // group 1 folded a tile of this item
          const float m1 = has1 ? xch[4 * r + 0] : -INFINITY;
          const float ds1 = xch[4 * r + 1], dn1 = xch[4 * r + 2];
          const uint32_t o_t0 = tmem + lane_off + C::TMEM_O;
          const bool o_in = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(o_t0, 32u, 2u * D));
          const float M = fmaxf(m, m1);
          const float f0 = (m == -INFINITY) ? 0.f : ex2_approx(m - M);
          const float f1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - M);
          const float dn = dnorm * f0 + (has1 ? dn1 * f1 : 0.f);
          const float ds = dsum * f0 + (has1 ? ds1 * f1 : 0.f);
          const float inv = dn > 0.f ? 1.f / dn : 0.f;
          const float lse2 = ds > 0.f ? (M + log2f(ds)) * 0.69314718055994530942f : -INFINITY;
          const bool store2 = qpos < L;
          const size_t rows_total = varlen ? static_cast<size_t>(args.total_tokens) * args.H
                                           : static_cast<size_t>(BHt) * args.N;
          const bool out_in =
              !store2 || fa_dbg_ok(orow < rows_total && lidx < rows_total, args.status);
          const float s0 = f0 * inv, s1 = f1 * inv;
          // 32 columns of each accumulator at a time, merged and stored.
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o0[32], o1[32];
            if (o_in) tmem_ld32(o_t0 + c0, o0);
            if (o_in && has1) tmem_ld32(o_t0 + D + c0, o1);
            if (store2 && out_in && o_in) {
              float ov[32];
#pragma unroll
              for (int i = 0; i < 32; ++i)
                ov[i] = __uint_as_float(o0[i]) * s0 + (has1 ? __uint_as_float(o1[i]) * s1 : 0.f);
              if (args.o_f32) {
                float4* dst =
                    reinterpret_cast<float4*>(static_cast<float*>(args.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
              } else {
                uint4* dst =
                    reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.o) + orow * D + c0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint4 u;
                  u.x = pack_bf16x2(ov[8 * i + 0], ov[8 * i + 1]);
                  u.y = pack_bf16x2(ov[8 * i + 2], ov[8 * i + 3]);
                  u.z = pack_bf16x2(ov[8 * i + 4], ov[8 * i + 5]);
                  u.w = pack_bf16x2(ov[8 * i + 6], ov[8 * i + 7]);
                  dst[i] = u;
                }
              }
            }
          }
          // Group 1's accumulator has been read: its next item may overwrite it.
          tc_fence_before();
          mbar_arrive(bar(C::B_XCH_DONE));
          if (store2 && out_in) args.lse[lidx] = lse2;
          tc_fence_before();
          mbar_arrive(bar(C::B_Q_EMPTY + qb));
        }
        g0 += n_kv;
        ++ti;
        continue;
      }
      const uint32_t o_t = tmem + lane_off + C::TMEM_O;
      const int wrow0 = mb * C::BM + quarter * 32;  // this warp's first row
      // Debug-build checks of the epilogue: O's TMEM range, the staging
      // rows, and the output indices against the tensors' sizes.
      const bool o_in = !kDebugChecks || __all_sync(0xffffffffu, tmem_ok(o_t, 32u, D));
      const size_t rows_total = varlen ? static_cast<size_t>(args.total_tokens) * args.H
                                       : static_cast<size_t>(BHt) * args.N;
      const bool out_in = !store || fa_dbg_ok(orow < rows_total && lidx < rows_total, args.status);
      if (!o_in) {
        // (debug build only) nothing to read: skip the item's stores
      } else if (D == 128 && args.o_tma && (varlen ? wrow0 + 32 <= L : wrow0 < L)) {
        // bf16 O through shared memory and one TMA store per 64-column half
        // and warp: the rows are staged in the item's Q buffer (no product
        // reads it any more) in the 128-byte-swizzled box layout, and the
        // tensor map clips rows past the end of a dense sequence.  (A packed
        // sequence's last rows are followed by the next sequence's, so a
        // warp with rows past its end stores row by row below.)  At D = 64 a
        // row is 128 bytes and the row-by-row stores are faster.
        uint8_t* qbuf = smem + C::OFF_Q + qb * C::TILE_BYTES;
        uint32_t ov[128];  // the row's 128 columns in one TMEM load and wait
        tmem_ld128(o_t, ov);
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 64) {
          uint8_t* row = qbuf + (c0 / 64) * C::HALF_BYTES + r * 128;
          if (!smem_ok(sbase + static_cast<uint32_t>(row - smem), 128u)) continue;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t* v8 = ov + c0 + 8 * ch;
            const float2 ii = make_float2(inv, inv);
            auto scaled = [&](int e) {  // (packed multiply, the same rounding per element)
              const float2 pr = __fmul2_rn(
                  make_float2(__uint_as_float(v8[e]), __uint_as_float(v8[e + 1])), ii);
              return pack_bf16x2(pr.x, pr.y);
            };
            uint4 u;
            u.x = scaled(0);
            u.y = scaled(2);
            u.z = scaled(4);
            u.w = scaled(6);
            *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) << 4)) = u;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int cc = 0; cc < C::HALVES; ++cc) {
            const uint32_t src =
                sbase + C::OFF_Q + qb * C::TILE_BYTES + cc * C::HALF_BYTES + quarter * 32 * 128;
            if (!smem_ok(src, 32u * 128u)) continue;
            if (varlen)
              tma_store_3d(&tm_o, src, cc * 64, it.h, it.tok0 + wrow0);
            else
              tma_store_3d(&tm_o, src, cc * 64, wrow0, it.bh);
          }
          tma_store_commit();
          // One item per CTA: the staging buffer must be read before the CTA
          // exits.  Persistent: the wait and the buffer's release follow the
          // next item's first tile (the stores read it meanwhile).
          if constexpr (!PERSIST) tma_store_wait_read();
        }
        __syncwarp();
        if constexpr (PERSIST) q_release = qb;
      } else {
        // 64 columns per TMEM load (one wait each), then the stores.
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t ov[64];
          tmem_ld64(o_t + c0, ov);
          if (store && out_in) {
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
      if (store && out_in) args.lse[lidx] = lse;
      // The item's Q buffer may take the Q tile of item ti + 2: its products
      // have finished (P_last V_last has) and the staged O has been read
      // (or, for deferred TMA stores, will have been once q_release runs).
      if (q_release != qb) {
        tc_fence_before();
        mbar_arrive(bar(C::B_Q_EMPTY + qb));
      }
      g0 += n_kv;
      ++ti;
    } while (ok && next_item(k, it));
    // Outstanding stores read shared memory until this wait; the CTA may not
    // exit before.
    if (q_release >= 0) {
      if (lane == 0) tma_store_wait_read();
      __syncwarp();
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

template <int D, int NG>
static cudaError_t launch_tc_impl(const TcMaps& maps, const TcFwdArgs& a, int grid_x,
                                  cudaStream_t stream) {
  using C = TcCfg<D, NG>;
  // The shared-memory opt-in is a per-device attribute of each function.
  static std::atomic<bool> attr_set[64];  // per device: attributes already set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    // every instantiation launch_tc_impl may launch (see the choice below)
    for (const void* f : {reinterpret_cast<const void*>(fa_fwd_tc_kernel<D, true, NG, false, false, true>),
                          reinterpret_cast<const void*>(fa_fwd_tc_kernel<D, true, NG, false, false, false>),
                          reinterpret_cast<const void*>(fa_fwd_tc_kernel<D, false, NG, NG == 1, true, false>),
                          reinterpret_cast<const void*>(fa_fwd_tc_kernel<D, false, NG, NG == 1, false, false>),
                          reinterpret_cast<const void*>(fa_fwd_tc_kernel<D, false, NG, false, false, true>)}) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(C::SMEM_BYTES));
      if (e != cudaSuccess) return e;
      if constexpr (NG == 2) {
        // The warpgroups' register split adds up only if a thread starts
        // with REGS_LAUNCH registers: refuse any other build of the kernel.
        cudaFuncAttributes fattr{};
        e = cudaFuncGetAttributes(&fattr, f);
        if (e != cudaSuccess) return e;
        if (fattr.numRegs != C::REGS_LAUNCH) return cudaErrorInvalidKernelImage;
      }
    }
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  static std::atomic<int> sm_count[64];  // per device: multiprocessors (0 = not read yet)
  int nsm = (dev >= 0 && dev < 64) ? sm_count[dev].load(std::memory_order_acquire) : 0;
  if (nsm == 0) {
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) sm_count[dev].store(nsm, std::memory_order_release);
  }
  TcFwdArgs args = a;
  // Packed sequences: H slots per query-tile slot (see the kernel's item
  // mapping); dense: every (sequence, head) pair's query tiles.
  args.num_items = a.cu_seqlens != nullptr ? a.H * (a.total_tokens / 128 + a.num_seqs)
                                           : grid_x * a.num_mblocks;
  // Persistent CTAs (one per SM) for short dense sequences, where the fixed
  // cost of a CTA (setup, first product, epilogue) is a large share of its
  // work; one CTA per item otherwise (the hardware scheduler balances the
  // long causal ranges, the head-grouped order keeps K/V in L2, and most
  // items of a packed batch are empty, which a one-item CTA skips at once).
  args.persistent = (a.cu_seqlens == nullptr && a.num_mblocks <= persistent_max_tiles(D) &&
                     args.num_items > nsm)
                        ? 1
                        : 0;
  const dim3 one_item(static_cast<unsigned>(args.num_items));
  const dim3 per_sm(static_cast<unsigned>(nsm));
  const unsigned T = C::THREADS, SM = C::SMEM_BYTES;
  if (args.persistent && args.window > 0)
    fa_fwd_tc_kernel<D, true, NG, false, false, true><<<per_sm, T, SM, stream>>>(
        maps.q, maps.k, maps.v, maps.o, args);
  else if (args.persistent)
    fa_fwd_tc_kernel<D, true, NG, false, false, false><<<per_sm, T, SM, stream>>>(
        maps.q, maps.k, maps.v, maps.o, args);
  else if (a.cu_seqlens != nullptr)  // (packed launches have no window)
    fa_fwd_tc_kernel<D, false, NG, NG == 1, true, false><<<one_item, T, SM, stream>>>(
        maps.q, maps.k, maps.v, maps.o, args);
  else if (args.window == 0)
    fa_fwd_tc_kernel<D, false, NG, NG == 1, false, false><<<one_item, T, SM, stream>>>(
        maps.q, maps.k, maps.v, maps.o, args);
  else
    fa_fwd_tc_kernel<D, false, NG, false, false, true><<<one_item, T, SM, stream>>>(
        maps.q, maps.k, maps.v, maps.o, args);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const TcMaps& maps, const TcFwdArgs& a, int D, int grid_x,
                          cudaStream_t stream) {
  if (D == 128) return launch_tc_impl<128, 1>(maps, a, grid_x, stream);
  return launch_tc_impl<64, kSoftmaxGroups64>(maps, a, grid_x, stream);
}

}  // namespace fa
