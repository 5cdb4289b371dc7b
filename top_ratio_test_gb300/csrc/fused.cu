// Fused similarity contraction + row/column top-2 for exhaustive SIFT matching.
//
// The "SERAC" page ("What changed": DP4A, fused row reduction, wider tiles) keeps
// the best two scores of each row in registers while the dot products are formed,
// so the num1 x num2 matrix is never written, and emits per-block column partials
// for the cross check.  This kernel keeps that dataflow but forms the dot products
// on the sm_103a tensor cores instead of DP4A:
//
//   * a persistent CTA per SM walks a contiguous range of work items; an item is one
//     128-row tile of A (resident in shared memory) against a run of 256-row tiles of
//     B streamed by TMA (128-byte swizzle, two stages);
//   * one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> f32, M=128, N=256,
//     K=16 x 8) into one of two TMEM accumulators (2 x 256 columns), so the epilogue
//     of tile t overlaps the MMAs of tile t+1.  u8 values are exact in bf16 and every
//     partial sum is an integer below 2^24, so the f32 accumulator holds the exact
//     integer score ("Exactness": 128 * 255^2 = 8,323,200 cannot overflow);
//   * eight epilogue warps read the accumulator (thread = row, 128 columns each) and
//       - add 2^23, which turns the f32 score s into the integer bits 0x4B000000 | s,
//       - build packed keys (s << 8 | 255 - column) for the row and
//         (s << 8 | 127 - row) for the column, so a plain unsigned max orders by score
//         then lower index -- the order-independent tie rule of "Real-Time Dense
//         Stereo at 34 Hz on a Jetson TX2 (MASDA, Part 3)", section 6, which packs
//         (value, k) into one integer for its fused warp top-2,
//       - keep the row top-2 in registers across the item's tiles,
//       - transpose each 32 x 32 block of column keys through shared memory, take the
//         top-2 of every column over the warp's 32 rows, then merge the four row
//         quadrants into one (k1, k2) per column per row tile: the column partials a
//         second kernel reduces ("Wider tiles": the column-partial table).
//
// Zero-padded rows and columns score 0 and fall to the zero floor, so ragged tails
// need no masking.  Every wait is bounded; a timeout sets an error bit that the
// match kernel reports through the count.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "ptx.cuh"
#include "serac_internal.h"

namespace serac {

namespace {

constexpr int A_BYTES = BM * KDIM * 2;   // 32 KB: one A tile, both K halves
constexpr int A_HALF = BM * 64 * 2;      // 16 KB: 128 rows x 64 bf16 (128 B)
constexpr int B_BYTES = BN * KDIM * 2;   // 64 KB
constexpr int B_HALF = BN * 64 * 2;      // 32 KB
constexpr int BOX_BYTES = 128 * 64 * 2;  // 16 KB: one TMA box (64 x 128)
constexpr int NUM_EPI_WARPS = 8;
constexpr int T_STRIDE = 36;             // transpose block: 32 columns x 36 words (padded)
constexpr int T_WARP_WORDS = 32 * T_STRIDE;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + A_BYTES;
constexpr int OFF_T = OFF_B + 2 * B_BYTES;
constexpr int OFF_M = OFF_T + NUM_EPI_WARPS * T_WARP_WORDS * 4;
constexpr int M_BYTES = 2 * 4 * BN * 8;  // [parity][quadrant][column] (k1, k2)
constexpr int OFF_BAR = OFF_M + M_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_TOTAL = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

struct Item {
  int p, rt, ct0, ct1;
};

__device__ __forceinline__ Item decode_item(const FusedParams& P, int item) {
  int lo = 0, hi = P.n_pairs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.pairs[mid].item_base <= item) lo = mid; else hi = mid - 1;
  }
  const FusedPair& fp = P.pairs[lo];
  const int local = item - fp.item_base;
  const int rt = local / fp.nsplit, s = local - rt * fp.nsplit;
  const int ct_total = (fp.n_b + BN - 1) / BN;
  return Item{lo, rt, s * ct_total / fp.nsplit, (s + 1) * ct_total / fp.nsplit};
}

// Insert a key into a top-2 of distinct keys (k1 > k2).
__device__ __forceinline__ void ins2(uint32_t& k1, uint32_t& k2, uint32_t x) {
  const uint32_t t = min(k1, x);
  k1 = max(k1, x);
  k2 = max(k2, t);
}
__device__ __forceinline__ void ins2_64(uint64_t& k1, uint64_t& k2, uint64_t x) {
  if (x > k1) { k2 = k1; k1 = x; } else if (x > k2) { k2 = x; }
}

// Tile-local row key (s << 8 | 255 - column) -> 64-bit (s << 32 | ~j); 0 if s == 0.
__device__ __forceinline__ uint64_t row_key64(uint32_t k, int col0) {
  const uint32_t s = k >> 8;
  if (s == 0) return 0;
  const uint32_t j = static_cast<uint32_t>(col0) + (255u - (k & 255u));
  return (static_cast<uint64_t>(s) << 32) | (0xFFFFFFFFu - j);
}

// Bounded wait by lane 0, result broadcast to the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          int code) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, err, code, WAIT_LIMIT_NS) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <bool DUMP>
__global__ void __launch_bounds__(FUSED_THREADS, 1)
    fused_top2_kernel(const __grid_constant__ FusedParams P, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + OFF_A;
  uint8_t* sB = smem + OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* a_full = bars + 0;
  uint64_t* a_empty = bars + 1;
  uint64_t* b_full = bars + 2;    // [2]
  uint64_t* b_empty = bars + 4;   // [2]
  uint64_t* t_full = bars + 6;    // [2]
  uint64_t* t_empty = bars + 8;   // [2]
  uint64_t* merged = bars + 10;   // [parity 2][half 2]
  uint64_t* drain = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], NUM_EPI_WARPS);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&merged[i], 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int it0 = P.cta_first[blockIdx.x], it1 = P.cta_first[blockIdx.x + 1];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t bcount = 0;
      for (int it = it0; it < it1; ++it) {
        const Item I = decode_item(P, it);
        const FusedPair& fp = P.pairs[I.p];
        const uint32_t n_local = static_cast<uint32_t>(it - it0);
        if (!mbar_wait(a_empty, (n_local & 1u) ^ 1u, abort_flag, P.err, ERR_TIMEOUT_PRODUCER, WAIT_LIMIT_NS)) break;
        mbar_arrive_expect_tx(a_full, A_BYTES);
        const int ay = fp.a_row0 + I.rt * BM;
        tma_load_2d(sA, &tmap, a_full, 0, ay);
        tma_load_2d(sA + A_HALF, &tmap, a_full, 64, ay);
        bool ok = true;
        for (int ct = I.ct0; ct < I.ct1; ++ct, ++bcount) {
          const uint32_t st = bcount & 1u, ph = (bcount >> 1) & 1u;
          if (!mbar_wait(&b_empty[st], ph ^ 1u, abort_flag, P.err, ERR_TIMEOUT_PRODUCER, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[st], B_BYTES);
          const int by = fp.b_row0 + ct * BN;
          uint8_t* dst = sB + st * B_BYTES;
          tma_load_2d(dst, &tmap, &b_full[st], 0, by);
          tma_load_2d(dst + BOX_BYTES, &tmap, &b_full[st], 0, by + 128);
          tma_load_2d(dst + B_HALF, &tmap, &b_full[st], 64, by);
          tma_load_2d(dst + B_HALF + BOX_BYTES, &tmap, &b_full[st], 64, by + 128);
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // let any copy still in flight land before shared memory is released
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 20000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t bcount = 0, tcount = 0;
      const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const Item I = decode_item(P, it);
        const uint32_t n_local = static_cast<uint32_t>(it - it0);
        if (!mbar_wait(a_full, n_local & 1u, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS)) break;
        tc_fence_after();
        for (int ct = I.ct0; ct < I.ct1; ++ct, ++bcount, ++tcount) {
          const uint32_t st = bcount & 1u, ph = (bcount >> 1) & 1u;
          const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&b_full[st], ph, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS) ||
              !mbar_wait(&t_empty[acc], aph ^ 1u, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * BN;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk >> 2) * A_HALF + (kk & 3) * 32);
            const uint32_t kboff = static_cast<uint32_t>((kk >> 2) * B_HALF + (kk & 3) * 32);
            mma_bf16(d, sw128_kmajor_desc(a_addr + koff), sw128_kmajor_desc(b_addr + st * B_BYTES + kboff), IDESC,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(&b_empty[st]);
          mma_commit(&t_full[acc]);
        }
        if (ok) mma_commit(a_empty);
      }
      // every MMA this thread issued must finish before TMEM is released
      mma_commit(drain);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(drain, 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;       // 0..7
    const int q = warp & 3;       // TMEM lane quadrant this warp may read
    const int h = e >> 2;         // which 128-column half of the tile
    const uint32_t rl = static_cast<uint32_t>(q * 32 + lane);  // row within the tile
    const uint32_t rowbits = 127u - rl;
    const uint32_t hbits = static_cast<uint32_t>(1 - h) << 7;
    uint32_t* tb = reinterpret_cast<uint32_t*>(smem + OFF_T) + e * T_WARP_WORDS;
    uint2* sm = reinterpret_cast<uint2*>(smem + OFF_M);
    uint32_t tcount = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const Item I = decode_item(P, it);
      const FusedPair& fp = P.pairs[I.p];
      const int64_t nb_pad = round_up(fp.n_b, PAD_ROWS);
      uint64_t K1 = 0, K2 = 0;
      for (int ct = I.ct0; ct < I.ct1; ++ct, ++tcount) {
        const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
        if (!warp_wait(&t_full[acc], aph, abort_flag, P.err, ERR_TIMEOUT_EPILOGUE)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t par = tcount & 1u;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + h * 128;
        uint32_t k1 = 0, k2 = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + c * 32, v);
          tmem_wait_ld();
          if (c == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&t_empty[acc]);
          }
          if constexpr (DUMP) {
            const int row = I.rt * BM + static_cast<int>(rl);
            if (row < fp.n_a) {
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int col = ct * BN + h * 128 + c * 32 + k;
                if (col < fp.n_b) P.dump[static_cast<int64_t>(row) * P.dump_ld + col] = __float2int_rn(__uint_as_float(v[k]));
              }
            }
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const uint32_t u = __float_as_uint(__fadd_rn(__uint_as_float(v[k]), 8388608.0f)) << 8;
              ins2(k1, k2, u | hbits | static_cast<uint32_t>(127 - c * 32 - k));
              tb[k * T_STRIDE + lane] = u | rowbits;
            }
            __syncwarp();
            uint32_t c1 = 0, c2 = 0;
#pragma unroll
            for (int r4 = 0; r4 < 8; ++r4) {
              const uint4 x = *reinterpret_cast<const uint4*>(tb + lane * T_STRIDE + r4 * 4);
              ins2(c1, c2, x.x);
              ins2(c1, c2, x.y);
              ins2(c1, c2, x.z);
              ins2(c1, c2, x.w);
            }
            __syncwarp();
            sm[(par * 4 + q) * BN + h * 128 + c * 32 + lane] = make_uint2(c1, c2);
          }
        }
        if constexpr (!DUMP) {
          // row: fold this tile's top-2 into the item's running top-2
          const int col0 = ct * BN;
          ins2_64(K1, K2, row_key64(k1, col0));
          ins2_64(K1, K2, row_key64(k2, col0));
          // columns: merge the four row quadrants once all four have written
          __syncwarp();
          if (lane == 0) mbar_arrive(&merged[par * 2 + h]);
          if (!warp_wait(&merged[par * 2 + h], (tcount >> 1) & 1u, abort_flag, P.err, ERR_TIMEOUT_EPILOGUE)) {
            ok = false;
            break;
          }
          const int col = h * 128 + q * 32 + lane;
          uint32_t m1 = 0, m2 = 0;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint2 x = sm[(par * 4 + qq) * BN + col];
            ins2(m1, m2, x.x);
            ins2(m1, m2, x.y);
          }
          P.colpart[fp.colpart_base + static_cast<int64_t>(I.rt) * nb_pad + ct * BN + col] = make_uint2(m1, m2);
        }
      }
      if constexpr (!DUMP) {
        if (ok) P.rowpart[(static_cast<int64_t>(it) * 2 + h) * BM + rl] = make_ulonglong2(K1, K2);
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

int fused_smem_bytes() { return SMEM_TOTAL; }

int launch_fused(const FusedParams& p, const void* tmap, bool dump, void* stream) {
  static bool configured[2] = {false, false};
  const int idx = dump ? 1 : 0;
  cudaError_t e;
  if (!configured[idx]) {
    e = dump ? cudaFuncSetAttribute(fused_top2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL)
             : cudaFuncSetAttribute(fused_top2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
    if (e != cudaSuccess) return static_cast<int>(e);
    configured[idx] = true;
  }
  CUtensorMap map;
  memcpy(&map, tmap, sizeof(map));
  const dim3 grid(p.grid), block(FUSED_THREADS);
  if (dump)
    fused_top2_kernel<true><<<grid, block, SMEM_TOTAL, static_cast<cudaStream_t>(stream)>>>(p, map);
  else
    fused_top2_kernel<false><<<grid, block, SMEM_TOTAL, static_cast<cudaStream_t>(stream)>>>(p, map);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace serac
