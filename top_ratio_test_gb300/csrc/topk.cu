// Row top-k (guided matching): the merge of the segment lists.
//
// The fused kernel's top-k modes leave, for every segment of the row problem and every
// 64-column quarter of its tiles, each row's K largest 64-bit keys (score << 32 |
// ~column) in descending order (serac_internal.h, topk_list_index).  This kernel takes
// the lists of the segments of each row's row tile, keeps the K largest keys of their
// union (keys are distinct, so the order of merges is free) and writes the first k as
// (score, column), a missing entry or a zero score as (0, -1):
// the candidate list of the "SERAC" page's "Exactness" order (score descending, lower
// index first, the zero floor) cut after k instead of after two.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"
#include "serac.h"
#include "serac_internal.h"
#include "topk_net.cuh"

namespace serac {
namespace {

constexpr int MERGE_THREADS = 128;  // 32 rows per block, four threads per row

// Thread 4 r + q of a block merges quarter q's lists of row r (one per segment of its
// row tile) into one descending top-K; the row's four threads then merge theirs by
// two shuffle rounds, and the first writes the row.
template <int K>
__global__ void __launch_bounds__(MERGE_THREADS) topk_merge_kernel(const TopkMergeParams p) {
  grid_dep_wait();  // the fused kernel's lists and error word
  const int t = static_cast<int>(blockIdx.x) * MERGE_THREADS + static_cast<int>(threadIdx.x);
  if (t == 0 && p.status) *p.status = *p.err ? SERAC_ETIMEOUT : SERAC_OK;
  const int i = t >> 2, quarter = t & 3;
  const bool live = i < p.n_a;  // every lane takes part in the shuffles
  unsigned long long top[K];
#pragma unroll
  for (int j = 0; j < K; ++j) top[j] = 0ull;
  if (live && p.n_b > 0) {
    const int ct_total = (p.n_b + BN - 1) / BN;
    const int64_t tiles = static_cast<int64_t>((p.n_a + BM - 1) / BM) * ct_total;
    const int rt = i / BM;
    const int64_t t0 = static_cast<int64_t>(rt) * ct_total;
    const int64_t t1 = t0 + ct_total < tiles ? t0 + ct_total : tiles;
    const int slots = piece_of(t1 - 1, tiles, p.npieces) - piece_of(t0, tiles, p.npieces) + 1;
    for (int slot = 0; slot < slots; ++slot) {
      unsigned long long y[K];
#pragma unroll
      for (int j = 0; j < K; ++j) y[j] = __ldcg(p.lists + topk_list_index(slot, quarter, j, K, p.ldl, i));
      merge_top<K>(top, y);
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    unsigned long long y[K];
#pragma unroll
    for (int j = 0; j < K; ++j) y[j] = __shfl_xor_sync(0xffffffffu, top[j], m);
    merge_top<K>(top, y);
  }
  if (!live || quarter != 0) return;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    if (j >= p.k) break;
    const unsigned long long x = top[j];
    const int64_t at = static_cast<int64_t>(i) * p.k + j;
    p.scores[at] = x ? static_cast<int32_t>(x >> 32) : 0;
    p.index[at] = x ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(x)) : -1;
  }
}

}  // namespace

int launch_topk_merge(const TopkMergeParams& p, int K, void* stream) {
  cudaLaunchConfig_t cfg = {};
  const int64_t threads = 4 * static_cast<int64_t>(p.n_a);
  cfg.gridDim = dim3(static_cast<unsigned>(threads > 0 ? (threads + MERGE_THREADS - 1) / MERGE_THREADS : 1));
  cfg.blockDim = dim3(MERGE_THREADS);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (K == 4) return static_cast<int>(cudaLaunchKernelEx(&cfg, topk_merge_kernel<4>, p));
  if (K == 8) return static_cast<int>(cudaLaunchKernelEx(&cfg, topk_merge_kernel<8>, p));
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace serac
