// Fused similarity contraction + row top-2 for exhaustive SIFT matching.
//
// The "SERAC" page ("What changed": DP4A, fused row reduction, wider tiles) keeps
// the best two scores of each row in registers while the dot products are formed,
// so the num1 x num2 matrix is never written.  This kernel keeps that dataflow but
// forms the dot products on the sm_103a tensor cores instead of DP4A, and it does so
// for row problems only: the column top-2 of a pair (A, B) is the row top-2 of
// (B, A), so the host hands every pair over as two problems, and both directions of
// the match come out of the same in-thread reduction:
//
//   * a persistent CTA per SM takes one contiguous piece (a row-major run of
//     128 x 256 tiles) of every problem of the launch; the tiles of a piece on one
//     row tile form a segment: one 128-row tile resident in shared memory against a
//     run of 256-row column tiles streamed by TMA (128-byte swizzle, two stages);
//   * one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> f32, M=128, N=256,
//     K=16 x 8) into one of two TMEM accumulators (2 x 256 columns), so the epilogue
//     of tile t overlaps the MMAs of tile t+1.  u8 values are exact in bf16 and every
//     partial sum is an integer below 2^24, so the f32 accumulator holds the exact
//     integer score ("Exactness": 128 * 255^2 = 8,323,200 cannot overflow);
//   * sixteen epilogue warps (four per SM sub-partition) read the accumulator
//     (thread = row, 64 columns each, one 64-column TMEM load per tile) and
//       - read 2^23 + s (each tile's first MMA writes 2^23 from two small bias
//         operands), whose f32 bits are the integer 0x4B000000 | s,
//       - build packed keys s << 8 | index with one integer multiply-add each (the
//         multiply by 256 drops the exponent bits), so a plain max orders by score
//         then lower index -- the order-independent tie rule of "Real-Time Dense
//         Stereo at 34 Hz on a Jetson TX2 (MASDA, Part 3)", section 6, which packs
//         (value, k) into one integer for its fused warp top-2.  Every key is below
//         0x7F800000, so keys also compare correctly as finite floats and the 3-input
//         float max can merge them;
//       - reduce each 32-key half with a min/max tree and keep each row's top-2 in
//         registers across the segment;
//     no epilogue warp waits for another: they share only the accumulator barriers.
//
// Global top-2 by atomics at the end of a segment: old = max(best, x1);
// second = max(second, min(old, x1)); second = max(second, x2).  Every candidate other
// than the final best reaches `second`, the final best never does (keys are unique),
// whatever the order.
//
// The same template serves two more epilogues (MODE): the score dump (the matrix
// written out, for the exactness and fused == unfused checks) and the row top-k of
// guided matching (each row's k <= 8 best keys per segment, sorting networks in place
// of the trees, written to per-segment lists that topk.cu merges).
//
// Zero-padded rows and columns score 0 and fall to the zero floor, so ragged tails
// need no masking.  Every wait is bounded; a timeout sets an error bit that the
// match kernel (or the top-k merge) reports.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "ptx.cuh"
#include "serac_internal.h"
#include "topk_net.cuh"

namespace serac {

namespace {

constexpr int A_BYTES = BM * KDIM * 2;   // 32 KB: one A tile, both K halves
constexpr int A_HALF = BM * 64 * 2;      // 16 KB: 128 rows x 64 bf16 (128 B)
constexpr int B_BYTES = BN * KDIM * 2;   // 64 KB
constexpr int B_HALF = BN * 64 * 2;      // 32 KB
constexpr int BOX_BYTES = 128 * 64 * 2;  // 16 KB: one TMA box (64 x 128)
constexpr int NUM_EPI_WARPS = 16;

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + A_BYTES;
constexpr int OFF_BAR = OFF_B + 2 * B_BYTES;
constexpr int BAR_BYTES = 256;
// bias operands of the first MMA of every tile (no swizzle, one 8-row group read by
// every group): A_bias rows [1, 0, ..., 0], B_bias rows [2^23, 0, ..., 0], each two K
// core matrices of 128 bytes
constexpr int OFF_BIAS = OFF_BAR + BAR_BYTES;
constexpr int BIAS_BYTES = 512;
constexpr int SMEM_TOTAL = OFF_BIAS + BIAS_BYTES + 1024;  // + alignment slack
static_assert(SMEM_TOTAL <= 232448, "shared memory budget");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

// Where a CTA stands in its work: problem p, its piece k of that problem, the next
// tile t of the piece and the piece's end (tiles numbered row-major within the problem).
struct Cursor {
  int p, k, t, tend;
};

// One segment: row tile rt of problem p against the column tiles [ct0, ct1), part of
// piece k.
struct Segment {
  int p, k, rt, ct0, ct1;
};

// Advances `cur` by one segment; false once the CTA has no work left.  Piece k of a
// problem belongs to CTA (offset + k) mod grid: the problem's T tiles are dealt to its
// n pieces as q = T / n tiles per piece plus one more for the first r = T mod n, so
// piece k starts at tile k q + min(k, r).
__device__ __forceinline__ bool next_segment(const FusedParams& P, Cursor& cur, Segment& g) {
  while (cur.t >= cur.tend) {
    if (++cur.p >= P.n_pairs) return false;
    const FusedPair& fp = P.pairs[cur.p];
    int k = static_cast<int>(blockIdx.x) - fp.offset;
    if (k < 0) k += P.grid;
    if (k >= fp.npieces) continue;
    const int tiles = ((fp.n_a + BM - 1) / BM) * ((fp.n_b + BN - 1) / BN);
    const int q = tiles / fp.npieces, r = tiles - q * fp.npieces;
    cur.k = k;
    cur.t = k * q + min(k, r);
    cur.tend = cur.t + q + (k < r ? 1 : 0);
  }
  const int ct_total = (P.pairs[cur.p].n_b + BN - 1) / BN;
  g.p = cur.p;
  g.k = cur.k;
  g.rt = cur.t / ct_total;
  g.ct0 = cur.t - g.rt * ct_total;
  g.ct1 = min(ct_total, g.ct0 + (cur.tend - cur.t));
  cur.t += g.ct1 - g.ct0;
  return true;
}

// ---- key arithmetic
__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Merge top-2 (b1, b2) into top-2 (a1, a2).
__device__ __forceinline__ void merge2(float& a1, float& a2, float b1, float b2) {
  const float m = fminf(a1, b1);
  a1 = fmaxf(a1, b1);
  a2 = fmax3(a2, m, b2);
}
// Top-2 of N distinct keys as a tree (pairwise, then pairwise merges): the same
// number of min/max as a sequential scan, but log2(N) deep instead of N.
template <int N>
__device__ __forceinline__ void tree_top2(const float (&x)[N], float& k1, float& k2) {
  float hi[N / 2], lo[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    hi[i] = fmaxf(x[2 * i], x[2 * i + 1]);
    lo[i] = fminf(x[2 * i], x[2 * i + 1]);
  }
#pragma unroll
  for (int w = N / 4; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) {
      float a1 = hi[2 * i], a2 = lo[2 * i];
      merge2(a1, a2, hi[2 * i + 1], lo[2 * i + 1]);
      hi[i] = a1;
      lo[i] = a2;
    }
  }
  k1 = hi[0];
  k2 = lo[0];
}
// 32-bit key s << 8 | (255 - local) -> 64-bit s << 32 | ~(base + local); 0 if s == 0.
__device__ __forceinline__ unsigned long long key64(uint32_t k, uint32_t base) {
  const uint32_t s = k >> 8;
  if (s == 0) return 0ull;
  const uint32_t idx = base + (255u - (k & 255u));
  return (static_cast<unsigned long long>(s) << 32) | (0xFFFFFFFFu - idx);
}

// The K largest tile keys (s << 8 | 255 - column in the tile) of one 32-column half,
// sorted descending: keys by one multiply-add each, sorted groups of K, then merges.
template <int K>
__device__ __forceinline__ void half_topk(const uint32_t (&v)[32], uint32_t key_mult, uint32_t chb, float (&t)[K]) {
  float x[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(mad_lo(v[k], key_mult, 31u - k));
#pragma unroll
  for (int gi = 0; gi < 32 / K; ++gi) sort_net<K>(x + gi * K);
#pragma unroll
  for (int gi = 1; gi < 32 / K; ++gi) merge_top<K>(x, x + gi * K);
#pragma unroll
  for (int i = 0; i < K; ++i) t[i] = __uint_as_float(__float_as_uint(x[i]) | chb);
}

// The epilogue of the row top-k modes: per segment, each row's K largest 64-bit keys
// over this warp's quarter of the columns, kept sorted in registers across the tiles
// and written to the segment's list (topk_list_index) at the segment's end.
template <int K>
__device__ __forceinline__ void topk_epilogue(const FusedParams& P, uint32_t tmem_base, uint64_t* t_full,
                                              uint64_t* t_empty, volatile int* abort_flag, int warp, int lane) {
  const int e = warp - 2;    // 0..15
  const int q = warp & 3;    // TMEM lane quadrant this warp may read
  const int qt = e >> 2;     // which 64-column quarter of the tile
  const uint32_t rl = static_cast<uint32_t>(q * 32 + lane);
  const uint32_t key_mult = P.key_mult;
  uint32_t tcount = 0;
  bool ok = true;
  Cursor cur{-1, 0, 0, 0};
  Segment g;
  while (next_segment(P, cur, g)) {
    const FusedPair& fp = P.pairs[g.p];
    unsigned long long R[K];  // the row's K best keys of the segment, descending; 0 = empty
#pragma unroll
    for (int j = 0; j < K; ++j) R[j] = 0ull;
    for (int ct = g.ct0; ct < g.ct1; ++ct, ++tcount) {
      const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
      {
        const bool w = mbar_wait(&t_full[acc], aph, abort_flag, P.err, ERR_TIMEOUT_EPILOGUE, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, w)) ok = false;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + qt * 64;
      // the two 32-column halves one after the other (32 values live at a time); the
      // buffer goes back to the MMA once the second is in registers.  Half index
      // (31 - k) -> tile-local 255 - (64 qt + 32 c + k).
      float t[K], u[K];
      {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr, v);
        tmem_wait_ld();
        half_topk<K>(v, key_mult, static_cast<uint32_t>(7 - 2 * qt) << 5, t);
      }
      {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + 32, v);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&t_empty[acc]);
        half_topk<K>(v, key_mult, static_cast<uint32_t>(6 - 2 * qt) << 5, u);
      }
      merge_top<K>(t, u);  // the tile's K largest
      unsigned long long y[K];
#pragma unroll
      for (int j = 0; j < K; ++j) y[j] = key64(__float_as_uint(t[j]), static_cast<uint32_t>(ct * BN));
      merge_top<K>(R, y);
    }
    const int i = g.rt * BM + static_cast<int>(rl);
    if (ok && i < fp.n_a) {
      const int ct_total = (fp.n_b + BN - 1) / BN;
      const int64_t tiles = static_cast<int64_t>((fp.n_a + BM - 1) / BM) * ct_total;
      const int slot = g.k - piece_of(static_cast<int64_t>(g.rt) * ct_total, tiles, fp.npieces);
#pragma unroll
      for (int j = 0; j < K; ++j) fp.keys[topk_list_index(slot, qt, j, K, fp.ldl, i)] = R[j];
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(FUSED_THREADS, 1)
    fused_top2_kernel(const __grid_constant__ FusedParams P, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ uint8_t smem_raw[];
  // align to 1024 B by pointer arithmetic on the shared array (keeps the address space)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem + OFF_A;
  uint8_t* sB = smem + OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* a_full = bars + 0;
  uint64_t* a_empty = bars + 1;
  uint64_t* b_full = bars + 2;    // [2]
  uint64_t* b_empty = bars + 4;   // [2]
  uint64_t* t_full = bars + 6;    // [2]
  uint64_t* t_empty = bars + 8;   // [2]
  uint64_t* drain = bars + 18;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 20);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], NUM_EPI_WARPS * 32);
    }
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
  // Every tile starts with one MMA of the bias operands that overwrites the
  // accumulator with 1 * 2^23 in every element; the eight real K steps accumulate onto
  // it, so the f32 result is 2^23 + s, whose bits are the integer 0x4B000000 | s
  // (s < 2^23; exact: all values stay integers below 2^24).  No per-score add and no
  // refill of TMEM by the epilogue.  Bias core matrices: eight 16-byte rows each,
  // element 0 of every row set in the K 0..7 matrix (words 0..31), the K 8..15 matrix
  // (words 32..63) all zero.
  if (threadIdx.x < 64) {
    uint32_t* bias = reinterpret_cast<uint32_t*>(smem + OFF_BIAS);
    const int w = threadIdx.x;
    bias[w] = (w < 32 && (w & 3) == 0) ? 0x00003F80u : 0u;        // bf16 1.0
    bias[64 + w] = (w < 32 && (w & 3) == 0) ? 0x00004B00u : 0u;   // bf16 2^23
    fence_proxy_async_smem();
  }
  __syncthreads();
  // a small match launch may be placed beside the CTAs now; it waits for this grid
  if (P.early_dependents) grid_dep_launch();
  // everything above overlaps the staging kernel (programmatic dependent launch);
  // the staged operands, the cleared keys and the error word are read after this
  grid_dep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // (no_copies: the failure-detection test hook -- nothing is loaded, so the MMA's
    // bounded wait runs out and the call reports a timeout)
    if (lane == 0 && !P.no_copies) {
      uint32_t bcount = 0, nseg = 0;
      bool ok = true;
      Cursor cur{-1, 0, 0, 0};
      Segment g;
      for (; ok && next_segment(P, cur, g); ++nseg) {
        const FusedPair& fp = P.pairs[g.p];
        if (!mbar_wait(a_empty, (nseg & 1u) ^ 1u, abort_flag, P.err, ERR_TIMEOUT_PRODUCER, WAIT_LIMIT_NS)) break;
        mbar_arrive_expect_tx(a_full, A_BYTES);
        const int ay = fp.a_row0 + g.rt * BM;
        tma_load_2d(sA, &tmap, a_full, 0, ay);
        tma_load_2d(sA + A_HALF, &tmap, a_full, 64, ay);
        for (int ct = g.ct0; ct < g.ct1; ++ct, ++bcount) {
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
      uint32_t bcount = 0, tcount = 0, nseg = 0;
      const uint32_t a_addr = smem_u32(sA), b_addr = smem_u32(sB);
      const uint32_t bias_addr = smem_u32(smem + OFF_BIAS);
      const uint64_t a_bias = plain_kmajor_desc(bias_addr, 128, 0);
      const uint64_t b_bias = plain_kmajor_desc(bias_addr + 256, 128, 0);
      bool ok = true;
      Cursor cur{-1, 0, 0, 0};
      Segment g;
      for (; ok && next_segment(P, cur, g); ++nseg) {
        if (!mbar_wait(a_full, nseg & 1u, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS)) break;
        tc_fence_after();
        for (int ct = g.ct0; ct < g.ct1; ++ct, ++bcount, ++tcount) {
          const uint32_t st = bcount & 1u, ph = (bcount >> 1) & 1u;
          const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
          if (!mbar_wait(&b_full[st], ph, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS) ||
              !mbar_wait(&t_empty[acc], aph ^ 1u, abort_flag, P.err, ERR_TIMEOUT_MMA, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * BN;
          mma_bf16(d, a_bias, b_bias, IDESC, 0u);  // every element = 2^23
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk >> 2) * A_HALF + (kk & 3) * 32);
            const uint32_t kboff = static_cast<uint32_t>((kk >> 2) * B_HALF + (kk & 3) * 32);
            mma_bf16(d, sw128_kmajor_desc(a_addr + koff), sw128_kmajor_desc(b_addr + st * B_BYTES + kboff), IDESC,
                     1u);
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
  } else if constexpr (MODE >= MODE_TOPK4) {
    topk_epilogue<MODE>(P, tmem_base, t_full, t_empty, abort_flag, warp, lane);
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr bool DUMP = MODE == MODE_DUMP;
    const int e = warp - 2;       // 0..15
    const int q = warp & 3;       // TMEM lane quadrant this warp may read
    const int qt = e >> 2;        // which 64-column quarter of the tile
    const uint32_t rl = static_cast<uint32_t>(q * 32 + lane);  // row within the tile
    // keys are u * 256 + index bits (the multiply shifts the exponent bits out); 256
    // comes from a kernel parameter so that the compiler keeps each key one integer
    // multiply-add on the FMA pipe while the min/max trees keep the ALU pipe busy
    const uint32_t key_mult = P.key_mult;
    uint32_t tcount = 0;
    bool ok = true;
    // the second slot's update of the previous segment's row, deferred so that the
    // returning atomic's latency overlaps the next segment
    unsigned long long* pend_ptr = nullptr;
    unsigned long long pend_old = 0ull, pend_x1 = 0ull;
    Cursor cur{-1, 0, 0, 0};
    Segment g;
    while (next_segment(P, cur, g)) {
      const FusedPair& fp = P.pairs[g.p];
      // the row's top-2 over the segment as tile keys (s << 8 | 255 - column in the
      // tile) with the column tile each came from; 0 = empty
      uint32_t R1 = 0u, R2 = 0u;
      int C1 = 0, C2 = 0;
      for (int ct = g.ct0; ct < g.ct1; ++ct, ++tcount) {
        const uint32_t acc = tcount & 1u, aph = (tcount >> 1) & 1u;
        {  // every lane tests the barrier (no broadcast), one vote for the outcome; on a
           // timeout keep going (the results are flagged invalid)
          const bool w = mbar_wait(&t_full[acc], aph, abort_flag, P.err, ERR_TIMEOUT_EPILOGUE, WAIT_LIMIT_NS);
          if (!__all_sync(0xffffffffu, w)) ok = false;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + qt * 64;
        float t1 = 0.f, t2 = 0.f;  // the row's top-2 over this tile (8-bit column index)
        {
          uint32_t v[64];
          tmem_ld_32x32b_x64(taddr, v);
          tmem_wait_ld();
          if constexpr (DUMP) {
            const int row = g.rt * BM + static_cast<int>(rl);
            if (row < fp.n_a) {
#pragma unroll
              for (int k = 0; k < 64; ++k) {
                const int col = ct * BN + qt * 64 + k;
                if (col < fp.n_b && ((row + col) & 1) == fp.transposed) {
                  const int64_t at = fp.transposed ? static_cast<int64_t>(col) * P.dump_ld + row
                                                   : static_cast<int64_t>(row) * P.dump_ld + col;
                  P.dump[at] = static_cast<int32_t>(v[k] & 0x7FFFFFu);  // bits of 2^23 + s
                }
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < 2; ++c) {  // two 32-column halves, keys with a 5-bit index
              float rk[32];
#pragma unroll
              for (int k = 0; k < 32; ++k) rk[k] = __uint_as_float(mad_lo(v[32 * c + k], key_mult, 31u - k));
              float a1, a2;
              tree_top2(rk, a1, a2);
              // half index (31 - k) -> tile-local 255 - (64 qt + 32 c + k)
              const uint32_t chb = static_cast<uint32_t>(7 - 2 * qt - c) << 5;
              merge2(t1, t2, __uint_as_float(__float_as_uint(a1) | chb), __uint_as_float(__float_as_uint(a2) | chb));
            }
          }
        }
        // hand the buffer back to the MMA: every thread once its own loads are done
        tc_fence_before();
        mbar_arrive(&t_empty[acc]);
        if constexpr (!DUMP) {
          // fold the tile's top-2 into the segment's.  Tiles come in column order, so a
          // tile key displaces a held one only with a strictly larger score
          // (k > (R | 255)); on equal scores the earlier, lower column stays.
          const uint32_t k1t = __float_as_uint(t1), k2t = __float_as_uint(t2);
          if (k1t > (R2 | 255u)) {
            if (k1t > (R1 | 255u)) {
              const bool t2_wins = k2t > (R1 | 255u);
              R2 = t2_wins ? k2t : R1;
              C2 = t2_wins ? ct : C1;
              R1 = k1t;
              C1 = ct;
            } else {
              R2 = k1t;
              C2 = ct;
            }
          }
        }
      }
      if constexpr (!DUMP) {
        if (pend_ptr) {
          const unsigned long long lo = pend_old < pend_x1 ? pend_old : pend_x1;
          if (lo) atomicMax(pend_ptr, lo);
          pend_ptr = nullptr;
        }
        const int i = g.rt * BM + static_cast<int>(rl);
        const unsigned long long K1 = key64(R1, static_cast<uint32_t>(C1 * BN));
        const unsigned long long K2 = key64(R2, static_cast<uint32_t>(C2 * BN));
        if (ok && i < fp.n_a && K1) {
          unsigned long long* rk = fp.keys + 2 * static_cast<int64_t>(i);
          pend_old = atomicMax(rk, K1);
          pend_x1 = K1;
          pend_ptr = rk + 1;
          if (K2) atomicMax(rk + 1, K2);
        }
      }
    }
    if (pend_ptr) {
      const unsigned long long lo = pend_old < pend_x1 ? pend_old : pend_x1;
      if (lo) atomicMax(pend_ptr, lo);
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

namespace {
template <int MODE>
cudaError_t launch_mode(const FusedParams& p, const CUtensorMap& map, void* stream) {
  // the opt-in to more than 48 KB of dynamic shared memory is an attribute of the
  // function on the current device: set it on every launch (cheap), so that every
  // device the caller makes current gets it
  cudaError_t e =
      cudaFuncSetAttribute(fused_top2_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(FUSED_THREADS);
  cfg.dynamicSmemBytes = SMEM_TOTAL;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_top2_kernel<MODE>, p, map);
}
}  // namespace

int launch_fused(const FusedParams& p, const void* tmap, int mode, void* stream) {
  CUtensorMap map;
  memcpy(&map, tmap, sizeof(map));
  switch (mode) {
    case MODE_TOP2: return static_cast<int>(launch_mode<MODE_TOP2>(p, map, stream));
    case MODE_DUMP: return static_cast<int>(launch_mode<MODE_DUMP>(p, map, stream));
    case MODE_TOPK4: return static_cast<int>(launch_mode<MODE_TOPK4>(p, map, stream));
    case MODE_TOPK8: return static_cast<int>(launch_mode<MODE_TOPK8>(p, map, stream));
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

}  // namespace serac
