// Operand staging and the match decision with compaction.
//
//   stage:  u8 descriptors -> bf16 rows of the staged buffer, each image zero-padded
//           to a multiple of 256 rows (bytes 0..255 are exact in bf16); an extra row
//           of blocks clears the key arrays the fused kernel merges into.
//   match:  per pair, blocks of 512 rows decode every row's top-2 key, test it, look
//           up its best column's top-2, apply the mutual check and the column test
//           ("SERAC", "Exactness": ratio test, cross check), and write the kept (i, j)
//           in ascending i: a block-wide scan of per-thread counts, then a decoupled
//           look-back over the pair's earlier blocks for the block's offset.  Each
//           launch also clears the other launch chunk's key region.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "serac.h"
#include "ptx.cuh"
#include "serac_internal.h"

namespace serac {

namespace {

// At most 32 registers per thread (256 threads x 8 blocks): four-warp blocks then fit
// beside a fused CTA (see launch_stage).
__global__ void __launch_bounds__(256, 8) stage_kernel(const __grid_constant__ StageParams P) {
  grid_dep_launch();  // the fused kernel may start its prologue alongside the last blocks
  if (blockIdx.y == static_cast<unsigned>(P.n_images)) {
    // clear the key arrays and the error word
    if (blockIdx.x >= static_cast<unsigned>(P.zero_blocks)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) *P.err = 0;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < P.zero_n;
         c += static_cast<int64_t>(P.zero_blocks) * blockDim.x)
      P.zero[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
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

// (best, second) 64-bit keys (s << 32 | 0xFFFFFFFF - index, 0 = empty) -> (s1, i1, s2, i2)
__device__ __forceinline__ int4 decode2(unsigned long long k1, unsigned long long k2) {
  int4 r;
  r.x = static_cast<int>(k1 >> 32);
  r.y = k1 ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k1)) : -1;
  r.z = static_cast<int>(k2 >> 32);
  r.w = k2 ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k2)) : -1;
  return r;
}

__device__ __forceinline__ bool passes(const FinishParams& P, const int4& t) {
  if (t.y < 0) return false;
  const int64_t lhs = static_cast<int64_t>(P.ratio_den_sq) * (static_cast<int64_t>(P.norm_sq) - t.x);
  const int64_t rhs = static_cast<int64_t>(P.ratio_num_sq) * (static_cast<int64_t>(P.norm_sq) - t.z);
  return lhs < rhs && t.x >= P.min_score;
}

constexpr unsigned long long LB_AGG = 1ull << 32;   // status word: block aggregate published
constexpr unsigned long long LB_INCL = 2ull << 32;  // status word: inclusive prefix published
constexpr uint64_t LB_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// At most 32 registers per thread, so that the four-warp blocks fit beside a fused CTA.
__global__ void __launch_bounds__(MATCH_THREADS, 65536 / (MATCH_THREADS * 32)) match_kernel(
    const __grid_constant__ FinishParams P) {
  // launched early (programmatic dependent launch): wait for the fused kernel's keys
  grid_dep_wait();
  // this block's pair
  int lo = 0, hi = P.n_pairs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.pairs[mid].blk_base <= static_cast<int>(blockIdx.x)) lo = mid; else hi = mid - 1;
  }
  const FinishPair& fp = P.pairs[lo];
  const ulonglong2* rk = reinterpret_cast<const ulonglong2*>(P.rowkeys) + fp.row_base;
  const ulonglong2* ck = reinterpret_cast<const ulonglong2*>(P.colkeys) + fp.col_base;
  __shared__ int s_b, s_prefix;
  __shared__ int warp_off[MATCH_THREADS / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // block order within the pair: a ticket, taken by the block once it runs, so that a
  // block only ever waits on blocks that already hold a ticket and are running --
  // whatever else shares the GPU and whichever blocks it keeps from being scheduled
  if (threadIdx.x == 0) s_b = atomicAdd(&P.tickets[lo], 1);
  __syncthreads();
  const int b = s_b;

  const int ib = b * MATCH_ROWS_PER_BLOCK + static_cast<int>(threadIdx.x) * MATCH_ROWS_PER_THREAD;
  int4 rt[MATCH_ROWS_PER_THREAD];
#pragma unroll
  for (int k = 0; k < MATCH_ROWS_PER_THREAD; ++k) {
    const ulonglong2 x = (ib + k < fp.n_a) ? rk[ib + k] : make_ulonglong2(0ull, 0ull);
    rt[k] = decode2(x.x, x.y);
    if (fp.row_top2 && ib + k < fp.n_a) reinterpret_cast<int4*>(fp.row_top2)[ib + k] = rt[k];
  }
  ulonglong2 cx[MATCH_ROWS_PER_THREAD];
#pragma unroll
  for (int k = 0; k < MATCH_ROWS_PER_THREAD; ++k)
    cx[k] = passes(P, rt[k]) ? ck[rt[k].y] : make_ulonglong2(0ull, 0ull);
  int cnt = 0;
  uint32_t keep = 0;
#pragma unroll
  for (int k = 0; k < MATCH_ROWS_PER_THREAD; ++k) {
    if (!passes(P, rt[k])) continue;
    const int4 c = decode2(cx[k].x, cx[k].y);
    if ((!P.mutual || c.y == ib + k) && (!P.col_ratio || passes(P, c))) {
      keep |= 1u << k;
      ++cnt;
    }
  }
  // exclusive scan of per-thread counts over the block (thread order = row order)
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_off[w] = incl;
  __syncthreads();
  if (w == 0) {
    constexpr int NW = MATCH_THREADS / 32;
    const int v = lane < NW ? warp_off[lane] : 0;
    int s = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += y;
    }
    if (lane < NW) warp_off[lane] = s - v;
    // decoupled look-back over the pair's earlier blocks, 32 at a time: lane i reads
    // the status word of block k0 - i; the nearest block with an inclusive prefix
    // ends the walk, the aggregates of the blocks after it are added to that prefix
    const int total = __shfl_sync(0xffffffffu, s, 31);
    unsigned long long* st = P.status + fp.blk_base;
    int prefix = 0;
    if (b == 0) {
      if (lane == 0) atomicExch(&st[0], LB_INCL | static_cast<uint32_t>(total));
    } else {
      if (lane == 0) atomicExch(&st[b], LB_AGG | static_cast<uint32_t>(total));
      const uint64_t t0 = now_ns();
      for (int k0 = b - 1; k0 >= 0; k0 -= 32) {
        const int k = k0 - lane;
        unsigned long long wv = LB_INCL;  // before block 0: an inclusive prefix of 0
        bool late = false;
        if (k >= 0) {
          wv = *reinterpret_cast<volatile unsigned long long*>(&st[k]);
          while (wv == 0ull) {  // every block before this one holds a ticket and publishes
            if (now_ns() - t0 > LB_LIMIT_NS) {
              late = true;
              break;
            }
            wv = *reinterpret_cast<volatile unsigned long long*>(&st[k]);
          }
        }
        if (__any_sync(0xffffffffu, late)) {
          if (lane == 0) atomicOr(P.err, ERR_TIMEOUT_LOOKBACK);
          break;
        }
        const unsigned incl = __ballot_sync(0xffffffffu, (wv & ~0xFFFFFFFFull) == LB_INCL);
        const int stop = incl ? __ffs(incl) - 1 : 31;
        const int val = (lane <= stop) ? static_cast<int>(static_cast<uint32_t>(wv)) : 0;
        prefix += __reduce_add_sync(0xffffffffu, val);
        if (incl) break;
      }
      if (lane == 0) atomicExch(&st[b], LB_INCL | static_cast<uint32_t>(prefix + total));
    }
    if (lane == 0) {
      s_prefix = prefix;
      if (b == fp.nblk - 1) *fp.count = (*reinterpret_cast<volatile int32_t*>(P.err) != 0) ? SERAC_ETIMEOUT : prefix + total;
    }
  }
  __syncthreads();
  int pos = s_prefix + warp_off[w] + incl - cnt;
#pragma unroll
  for (int k = 0; k < MATCH_ROWS_PER_THREAD; ++k) {
    if (keep & (1u << k)) {
      if (pos < fp.capacity) {
        fp.matches[2 * static_cast<int64_t>(pos)] = ib + k;
        fp.matches[2 * static_cast<int64_t>(pos) + 1] = rt[k].y;
      }
      ++pos;
    }
  }
  // optional column top-2, split over the pair's blocks
  if (fp.col_top2) {
    const int per = (fp.n_b + fp.nblk - 1) / fp.nblk;
    const int j1 = min(fp.n_b, (b + 1) * per);
    for (int j = b * per + static_cast<int>(threadIdx.x); j < j1; j += MATCH_THREADS) {
      const ulonglong2 x = ck[j];
      reinterpret_cast<int4*>(fp.col_top2)[j] = decode2(x.x, x.y);
    }
  }
  // clear the other chunk's key region, split over the whole launch
  const int64_t per = (P.zero_n + P.total_blocks - 1) / P.total_blocks;
  const int64_t z1 = min(P.zero_n, (static_cast<int64_t>(blockIdx.x) + 1) * per);
  for (int64_t z = static_cast<int64_t>(blockIdx.x) * per + threadIdx.x; z < z1; z += MATCH_THREADS)
    P.zero[z] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

int launch_stage(const StageParams& p, int64_t max_chunks, void* stream, bool beside_fused) {
  // Beside a running fused kernel (one CTA of 18 warps x 96 registers per SM) an SM
  // sub-partition holding five of its warps has 1,024 registers left: one warp of 32
  // registers.  Blocks of four warps (one per sub-partition) then fit beside it; blocks
  // of eight would wait for the fused kernel to end.
  const int threads = beside_fused ? 128 : 256;
  int64_t blocks = (max_chunks + threads - 1) / threads;
  if (blocks > 2048) blocks = 2048;
  if (blocks < p.zero_blocks) blocks = p.zero_blocks;
  if (blocks < 1) blocks = 1;
  stage_kernel<<<dim3(static_cast<unsigned>(blocks), p.n_images + 1), threads, 0,
                 static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

int launch_match(const FinishParams& p, void* stream) {
  if (p.total_blocks == 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.total_blocks);
  cfg.blockDim = dim3(MATCH_THREADS);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, match_kernel, p));
}

}  // namespace serac
