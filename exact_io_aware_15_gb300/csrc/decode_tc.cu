// Split-KV decode over a paged KV cache with grouped query heads, on the
// tensor cores: the G = H / H_kv query heads that share a KV head are packed
// into the N dimension of one tcgen05 product, so every key row read from
// HBM is used by all G heads in one instruction stream.
//
// Pages: the review of "Learning FlashAttention the Hard Way - Part 1" names
// PagedAttention and grouped decoding among the descendants of the same
// algebra; the fold is the online-softmax state (m, d, o) of "The Merge, and
// the Twist" in the base-2 coordinates of "Alternative Twist: Base 2", and
// the chunk states are merged afterwards by the split-K combine of
// "Associativity is All You Need".
//
// fa_decode_paged_tc_kernel: one CTA per (sequence b, KV head hk, chunk c),
// 192 threads: warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 softmax.
// Per tile of 128 keys (tiles aligned to multiples of 128 in the sequence,
// chunks made of whole tiles, keys past the sequence end masked):
//   S^T[key, head] = K_tile . Q_g^T      M = 128 keys, N = 16 (the G heads,
//                                         padded), A = K (smem), B = Q (smem)
//   softmax, thread = key: per-head maximum over the tile through one
//   bounded exchange between the 4 warps, P = 2^(sigma - m) in bf16 to smem
//   O^T[d, head] += V_tile^T . P          M = D = 128, N = 16, A = V as an
//                                         MN-major operand, B = P (smem)
// S^T is double-buffered in TMEM (16 columns each), O^T takes 16 more.  The
// tile's keys are fetched page by page with 3-D TMA boxes (one box per page
// piece and 64-column half); pieces past the sequence end or whose page
// index is out of range are fetched from a row past the pool, which TMA
// fills with zeros (an out-of-range index also sets FA_ERR_DEVICE_BOUNDS).
// Value rows past the sequence end inside its last page are zeroed in
// shared memory before the P.V product, so stale page contents never reach
// it.  Every wait is bounded.

#include <cuda.h>
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kKeys = 128;                    // keys per tile
constexpr int kN = 16;                        // heads per product (G <= 16, padded)
constexpr uint32_t kHalf = 128u * 128u;       // 128 rows x 64 bf16 columns
constexpr uint32_t kQHalf = 16u * 128u;       // 16 rows x 64 bf16 columns
constexpr int kStages = 3;
constexpr uint32_t kTile = 2 * kHalf;         // K or V tile, D = 128
constexpr uint32_t OFF_Q = 0;                 // 2 halves x 2 KB
constexpr uint32_t OFF_P = 2 * kQHalf;        // 2 buffers x (2 key halves x 2 KB)
constexpr uint32_t OFF_KV = 4096 + 8192;      // stage s: K at +2s*kTile, V at +(2s+1)*kTile
constexpr uint32_t OFF_XCH = OFF_KV + kStages * 2 * kTile;  // [2][4][16] floats
constexpr uint32_t OFF_BAR = OFF_XCH + 2 * 4 * kN * 4;
constexpr int B_Q_FULL = 0;
constexpr int B_KV_FULL = 1;
constexpr int B_KV_EMPTY = B_KV_FULL + kStages;
constexpr int B_S_FULL = B_KV_EMPTY + kStages;  // two
constexpr int B_P_FULL = B_S_FULL + 2;
constexpr int B_O_DONE = B_P_FULL + 1;
constexpr int B_XCH = B_O_DONE + 1;
constexpr int B_DRAIN = B_XCH + 1;
constexpr int kNumBars = B_DRAIN + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t kSmemBytes = OFF_MISC + 16 + 1024;
constexpr uint32_t TM_S = 0, TM_O = 32, kTmemCols = 64;
static_assert(kSmemBytes <= 232448, "shared memory");

// kind::f16 instruction descriptor, bf16 A and B, fp32 D, with the major-ness
// of both operands: bit 15 A (1 = MN-major), bit 16 B.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void wait_unwind(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(192, 1)
    fa_decode_paged_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const PagedDecodeArgs a, int G, int page_shift) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  auto bar = [&](int i) -> uint32_t { return sbase + OFF_BAR + 8u * i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int S = a.S, H = a.H;
  const int P = 1 << page_shift;

  int L = __ldg(a.seqlens + b);
  if (L < 0 || static_cast<long long>(L) > static_cast<long long>(a.max_blocks) * P) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBounds);
    L = 0;
  }
  // Chunks are whole 128-key tiles (ceil(L / S) rounded up), so no tile is
  // read by two chunks.
  const int size = ((L + S - 1) / S + kKeys - 1) / kKeys * kKeys;
  const int k0 = min(L, c * size), k1 = min(L, (c + 1) * size);
  if (k0 >= k1) {  // empty chunk: the identity (-inf, 0, 0) for every head of the group
    for (int i = threadIdx.x; i < G * 128; i += blockDim.x) {
      const size_t row = (static_cast<size_t>(b) * H + hk * G + i / 128) * S + c;
      a.part_o[row * 128 + (i % 128)] = 0.f;
      if (i % 128 == 0) {
        a.part_m[row] = -INFINITY;
        a.part_d[row] = 0.f;
      }
    }
    return;
  }
  const int t0 = k0 / kKeys;
  const int nt = (k1 + kKeys - 1) / kKeys - t0;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KV_FULL + s), 1);
      mbar_init(bar(B_KV_EMPTY + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_P_FULL), 128);
    mbar_init(bar(B_O_DONE), 1);
    mbar_init(bar(B_XCH), 128);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // P rows of the padding heads stay zero
  for (int i = threadIdx.x; i < 8192 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_Q_FULL), 2 * kQHalf);
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sbase + OFF_Q + h * kQHalf, &tm_q, bar(B_Q_FULL), h * 64, hk * G, b);
      const int R = min(P, kKeys);  // rows per page piece
      const int pool_rows = a.num_pages * P;
      const int* table = a.block_table + static_cast<size_t>(b) * a.max_blocks;
      int issued = 0;
      bool bad = false;
      for (int t = 0; t < nt; ++t) {
        const int s = t % kStages;
        if (t >= kStages &&
            !mbar_wait(bar(B_KV_EMPTY + s), ((t / kStages) - 1) & 1, abort_flag, a.status))
          break;
        const uint32_t fb = bar(B_KV_FULL + s);
        mbar_arrive_expect_tx(fb, 2 * kTile);
        const uint32_t ks = sbase + OFF_KV + 2u * s * kTile, vs = ks + kTile;
        const int kbase = (t0 + t) * kKeys;
        for (int i = 0; i < kKeys / R; ++i) {
          const int key = kbase + i * R;
          int row = pool_rows;  // past the pool: zero fill
          if (key < L) {
            const int pg = __ldg(table + (key >> page_shift));
            if (pg >= 0 && pg < a.num_pages)
              row = pg * P + (key & (P - 1));
            else
              bad = true;
          }
          for (int h = 0; h < 2; ++h) {
            const uint32_t off = h * kHalf + i * R * 128u;
            tma_load_3d(ks + off, &tm_k, fb, h * 64, hk, row);
            tma_load_3d(vs + off, &tm_v, fb, h * 64, hk, row);
          }
        }
        issued = t + 1;
      }
      if (bad) atomicOr(a.status, kStatusBounds);
      if (*abort_flag) {
        wait_unwind(bar(B_Q_FULL), 0);
        for (int t = max(0, issued - kStages); t < issued; ++t)
          wait_unwind(bar(B_KV_FULL + t % kStages), (t / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kN, false, false);
      constexpr uint32_t id_pv = idesc(128, kN, true, false);
      auto wait = [&](int bb, uint32_t parity) {
        return mbar_wait(bar(bb), parity, abort_flag, a.status);
      };
      auto kv_of = [&](int t) { return sbase + OFF_KV + 2u * (t % kStages) * kTile; };
      auto issue_qk = [&](int t) -> bool {
        if (!wait(B_KV_FULL + t % kStages, (t / kStages) & 1)) return false;
        tc_fence_after();
        const uint32_t ks = kv_of(t);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off_k = (kk >> 2) * kHalf + (kk & 3) * 32u;
          const uint32_t off_q = (kk >> 2) * kQHalf + (kk & 3) * 32u;
          tc_mma_ss(tmem + TM_S + 16u * (t & 1), sdesc_sw128(ks + off_k, 16u, 1024u),
                    sdesc_sw128(sbase + OFF_Q + off_q, 16u, 1024u), id_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_S_FULL + (t & 1)));
        return true;
      };
      bool ok = wait(B_Q_FULL, 0) && issue_qk(0) && (nt < 2 || issue_qk(1));
      for (int t = 0; ok && t < nt; ++t) {
        if (!wait(B_P_FULL, t & 1)) break;
        tc_fence_after();
        const uint32_t vs = kv_of(t) + kTile;
        const uint32_t pb = sbase + OFF_P + (t & 1) * 4096u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // A = V^T: M = D (64-column halves kHalf apart), K = 16 keys = 2048 B
          // B = P: N = 16 heads, K = 16 keys (key half kk/4, 32 B per slice)
          const uint32_t off_p = (kk >> 2) * 2048u + (kk & 3) * 32u;
          tc_mma_ss(tmem + TM_O, sdesc_sw128(vs + kk * 2048u, kHalf, 1024u),
                    sdesc_sw128(pb + off_p, 16u, 1024u), id_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_O_DONE));
        tc_commit(bar(B_KV_EMPTY + t % kStages));
        if (t + 2 < nt && !issue_qk(t + 2)) break;
      }
      tc_commit(bar(B_DRAIN));
      wait_unwind(bar(B_DRAIN), 0);
    }
  } else {
    // ========================= softmax / epilogue =========================
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // TMEM lane: key of the tile, and column d of O^T
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);  // [2][4][16]
    const float c2 = a.scale_log2;
    float m[kN], dpart[kN];
#pragma unroll
    for (int h = 0; h < kN; ++h) {
      m[h] = -INFINITY;
      dpart[h] = 0.f;
    }
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int key = (t0 + t) * kKeys + r;
      const bool vis = key >= k0 && key < k1;
      const bool w1 =
          mbar_wait(bar(B_S_FULL + (t & 1)), (t >> 1) & 1, abort_flag, a.status);
      if (__any_sync(0xffffffffu, !w1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[16];
      tmem_ld16(tmem + lane_off + TM_S + 16u * (t & 1), sr);
      float sg[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        sg[h] = (vis && h < G) ? __uint_as_float(sr[h]) * c2 : -INFINITY;
        float mx = sg[h];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) xch[((t & 1) * 4 + q4) * kN + h] = mx;
      }
      mbar_arrive(bar(B_XCH));
      const bool w2 = mbar_wait(bar(B_XCH), t & 1, abort_flag, a.status);
      if (__any_sync(0xffffffffu, !w2)) {
        ok = false;
        break;
      }
      float alpha[kN];
      bool moved = false;
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        const float* x = xch + (t & 1) * 4 * kN + h;
        const float tm = fmaxf(fmaxf(x[0], x[kN]), fmaxf(x[2 * kN], x[3 * kN]));
        const float mn = fmaxf(m[h], tm);
        alpha[h] = (mn == m[h]) ? 1.f : ex2_approx(m[h] - mn);  // m = -inf: 0
        moved |= alpha[h] != 1.f;
        m[h] = mn;
      }
      // P (bf16) of this key for every head, into the tile's P buffer:
      // row h, key r -> key half r/64, 16-byte chunk (r%64)/8 swizzled by h%8
      uint8_t* pbuf = smem + OFF_P + (t & 1) * 4096u + (r >> 6) * 2048u;
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        if (h < G) {
          const float p = vis ? ex2_approx(sg[h] - m[h]) : 0.f;
          dpart[h] = dpart[h] * alpha[h] + p;
          const uint32_t chunk = ((r & 63) >> 3) ^ (h & 7);
          *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + chunk * 16 + (r & 7) * 2) =
              __float2bfloat16_rn(p);
        }
      }
      // value rows past the sequence end may hold stale page contents
      if (key >= L) {
        uint4* vrow = reinterpret_cast<uint4*>(smem + OFF_KV + (2 * (t % kStages) + 1) * kTile +
                                               r * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          vrow[j] = make_uint4(0u, 0u, 0u, 0u);
          vrow[kHalf / 16 + j] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (t > 0 && moved) {  // o <- alpha o needs P.V of the previous tile in TMEM
        const bool w3 = mbar_wait(bar(B_O_DONE), (t - 1) & 1, abort_flag, a.status);
        if (__any_sync(0xffffffffu, !w3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t ov[16];
        tmem_ld16(tmem + lane_off + TM_O, ov);
#pragma unroll
        for (int h = 0; h < kN; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
        tmem_st16(tmem + lane_off + TM_O, ov);
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_P_FULL));
    }

    if (ok) {
      // d of every head: sum of the 128 threads' partial sums (exchange
      // slots reused after the last tile's maxima were read)
      __syncwarp();
      const bool w4 = mbar_wait(bar(B_O_DONE), (nt - 1) & 1, abort_flag, a.status);
      if (!__any_sync(0xffffffffu, !w4)) {
        tc_fence_after();
        uint32_t ov[16];
        tmem_ld16(tmem + lane_off + TM_O, ov);
        float* dx = xch + (nt & 1) * 4 * kN;  // slot of the next (unused) exchange
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          float s = dpart[h];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
          if (lane == 0) dx[q4 * kN + h] = s;
        }
        mbar_arrive(bar(B_XCH));
        const bool w5 = mbar_wait(bar(B_XCH), nt & 1, abort_flag, a.status);
        if (!__any_sync(0xffffffffu, !w5)) {
#pragma unroll
          for (int h = 0; h < kN; ++h) {
            if (h < G) {
              const size_t row = (static_cast<size_t>(b) * H + hk * G + h) * S + c;
              a.part_o[row * 128 + r] = __uint_as_float(ov[h]);
              if (r == 0) {
                a.part_m[row] = m[h];
                a.part_d[row] = (dx[h] + dx[kN + h]) + (dx[2 * kN + h] + dx[3 * kN + h]);
              }
            }
          }
        }
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool decode_paged_tc_supported(int D, int G, int page_size) {
  return D == 128 && G >= 2 && G <= kN && page_size >= 8;
}

cudaError_t launch_decode_paged_tc(const PagedTcMaps& maps, const PagedDecodeArgs& a, int G,
                                   cudaStream_t stream) {
  static std::atomic<bool> attr_set[64];  // per device: attribute already set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(fa_decode_paged_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int page_shift = __builtin_ctz(static_cast<unsigned>(a.page_size));
  dim3 grid(static_cast<unsigned>(a.S), static_cast<unsigned>(a.Hkv),
            static_cast<unsigned>(a.B));
  fa_decode_paged_tc_kernel<<<grid, 192, kSmemBytes, stream>>>(maps.q, maps.k, maps.v, a, G,
                                                                page_shift);
  return cudaGetLastError();
}

}  // namespace fa
