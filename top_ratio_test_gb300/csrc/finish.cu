// Operand staging, partial reduction and the match decision with compaction.
//
//   stage:  u8 descriptors -> bf16 rows of the staged buffer, each image zero-padded
//           to a multiple of 256 rows (bytes 0..255 are exact in bf16).
//   reduce: per row, fold the row partials of its column splits; per column, fold
//           the per-row-tile column partials ("Wider tiles" on the "SERAC" page: the
//           column-partial table that ColMatch consumes) into the final top-2 with
//           global indices, ties to the lower index.
//   match:  per pair, one block tests every row, looks up its best column, applies
//           the mutual check and the column test, and writes the kept (i, j) in
//           ascending i with a warp-ballot / block-scan compaction.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "serac.h"
#include "serac_internal.h"

namespace serac {

namespace {

__global__ void __launch_bounds__(256) stage_kernel(const __grid_constant__ StageParams P) {
  const StageImage im = P.images[blockIdx.y];
  const int64_t n_pad = round_up(im.n, PAD_ROWS);
  const int64_t chunks = n_pad * (KDIM / 16);  // 16-byte input chunks
  const uint4* src = reinterpret_cast<const uint4*>(im.src);
  uint4* dst = reinterpret_cast<uint4*>(P.staged + static_cast<int64_t>(im.row0) * KDIM);
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint4 in = make_uint4(0u, 0u, 0u, 0u);
    if ((c >> 3) < im.n) in = __ldg(src + c);
    const uint32_t w[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 lo =
          __floats2bfloat162_rn(static_cast<float>(w[i] & 0xFFu), static_cast<float>((w[i] >> 8) & 0xFFu));
      const __nv_bfloat162 hi =
          __floats2bfloat162_rn(static_cast<float>((w[i] >> 16) & 0xFFu), static_cast<float>(w[i] >> 24));
      o[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
      o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
    }
    dst[2 * c] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * c + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

__device__ __forceinline__ void ins2_64(uint64_t& k1, uint64_t& k2, uint64_t x) {
  if (x > k1) { k2 = k1; k1 = x; } else if (x > k2) { k2 = x; }
}

// 64-bit key (s << 32 | 0xFFFFFFFF - index), 0 = empty -> (s1, i1, s2, i2)
__device__ __forceinline__ int4 decode2(uint64_t k1, uint64_t k2) {
  int4 r;
  r.x = static_cast<int>(k1 >> 32);
  r.y = k1 ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k1)) : -1;
  r.z = static_cast<int>(k2 >> 32);
  r.w = k2 ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k2)) : -1;
  return r;
}

template <typename F>
__device__ __forceinline__ int find_pair(const FinishParams& P, int64_t t, F base_of) {
  int lo = 0, hi = P.n_pairs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base_of(P.pairs[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(256) reduce_kernel(const __grid_constant__ FinishParams P) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t < P.total_rows) {
    const int p = find_pair(P, t, [](const FinishPair& f) { return static_cast<int64_t>(f.row_base); });
    const FinishPair& fp = P.pairs[p];
    const int i = static_cast<int>(t - fp.row_base);
    uint64_t k1 = 0, k2 = 0;
    if (fp.nsplit > 0) {
      const int rt = i / BM, rl = i - rt * BM;
      for (int s = 0; s < fp.nsplit; ++s) {
        const int64_t item = static_cast<int64_t>(fp.item_base) + static_cast<int64_t>(rt) * fp.nsplit + s;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const ulonglong2 x = P.rowpart[(item * 2 + h) * BM + rl];
          ins2_64(k1, k2, x.x);
          ins2_64(k1, k2, x.y);
        }
      }
    }
    const int4 r = decode2(k1, k2);
    P.rowfinal[t] = r;
    if (fp.row_top2) reinterpret_cast<int4*>(fp.row_top2)[i] = r;
  } else if (t < static_cast<int64_t>(P.total_rows) + P.total_cols) {
    const int64_t tc = t - P.total_rows;
    const int p = find_pair(P, tc, [](const FinishPair& f) { return static_cast<int64_t>(f.col_base); });
    const FinishPair& fp = P.pairs[p];
    const int j = static_cast<int>(tc - fp.col_base);
    uint64_t k1 = 0, k2 = 0;
    if (fp.nsplit > 0) {
      const int rts = (fp.n_a + BM - 1) / BM;
      const int64_t nb_pad = round_up(fp.n_b, PAD_ROWS);
      for (int rt = 0; rt < rts; ++rt) {
        const uint2 x = P.colpart[fp.colpart_base + rt * nb_pad + j];
        const uint32_t kk[2] = {x.x, x.y};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t s = kk[u] >> 8;
          if (s) {
            const uint32_t i = static_cast<uint32_t>(rt * BM) + (127u - (kk[u] & 255u));
            ins2_64(k1, k2, (static_cast<uint64_t>(s) << 32) | (0xFFFFFFFFu - i));
          }
        }
      }
    }
    const int4 r = decode2(k1, k2);
    P.colfinal[tc] = r;
    if (fp.col_top2) reinterpret_cast<int4*>(fp.col_top2)[j] = r;
  }
}

__device__ __forceinline__ bool passes(const FinishParams& P, const int4& t) {
  if (t.y < 0) return false;
  const int64_t lhs = static_cast<int64_t>(P.ratio_den_sq) * (static_cast<int64_t>(P.norm_sq) - t.x);
  const int64_t rhs = static_cast<int64_t>(P.ratio_num_sq) * (static_cast<int64_t>(P.norm_sq) - t.z);
  return lhs < rhs && t.x >= P.min_score;
}

constexpr int MATCH_THREADS = 1024;

__global__ void __launch_bounds__(MATCH_THREADS) match_kernel(const __grid_constant__ FinishParams P) {
  const FinishPair& fp = P.pairs[blockIdx.x];
  __shared__ int warp_off[32];
  __shared__ int block_total;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int base = 0;
  for (int i0 = 0; i0 < fp.n_a; i0 += MATCH_THREADS) {
    const int i = i0 + static_cast<int>(threadIdx.x);
    int j = -1;
    if (i < fp.n_a) {
      const int4 r = P.rowfinal[fp.row_base + i];
      if (passes(P, r)) {
        const int4 c = P.colfinal[fp.col_base + r.y];
        if ((!P.mutual || c.y == i) && (!P.col_ratio || passes(P, c))) j = r.y;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, j >= 0);
    if (lane == 0) warp_off[w] = __popc(m);
    __syncthreads();
    if (w == 0) {
      const int v = warp_off[lane];
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      warp_off[lane] = incl - v;
      if (lane == 31) block_total = incl;
    }
    __syncthreads();
    if (j >= 0) {
      const int pos = base + warp_off[w] + __popc(m & ((1u << lane) - 1u));
      if (pos < fp.capacity) {
        fp.matches[2 * static_cast<int64_t>(pos)] = i;
        fp.matches[2 * static_cast<int64_t>(pos) + 1] = j;
      }
    }
    base += block_total;
    __syncthreads();
  }
  if (threadIdx.x == 0) *fp.count = (*P.err != 0) ? SERAC_ETIMEOUT : base;
}

}  // namespace

int launch_stage(const StageParams& p, int64_t max_chunks, void* stream) {
  if (p.n_images == 0) return 0;
  int64_t blocks = (max_chunks + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  stage_kernel<<<dim3(static_cast<unsigned>(blocks), p.n_images), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

int launch_reduce(const FinishParams& p, void* stream) {
  const int64_t n = static_cast<int64_t>(p.total_rows) + p.total_cols;
  if (n == 0) return 0;
  reduce_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

int launch_match(const FinishParams& p, void* stream) {
  if (p.n_pairs == 0) return 0;
  match_kernel<<<p.n_pairs, MATCH_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace serac
