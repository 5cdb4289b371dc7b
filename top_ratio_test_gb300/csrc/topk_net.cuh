// Sorting networks for the row top-k (k = 4 or 8) on distinct keys, largest first,
// shared by the fused kernel's top-k epilogue and the merge of its segment lists.
#pragma once
#include <stdint.h>

namespace serac {

__device__ __forceinline__ void ce(float& a, float& b) {  // a <- max, b <- min
  const float hi = fmaxf(a, b), lo = fminf(a, b);
  a = hi;
  b = lo;
}
__device__ __forceinline__ void ce64(unsigned long long& a, unsigned long long& b) {
  const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}
// Sorts x[0..K) in descending order (K = 4: 5 compare-exchanges; K = 8: Batcher's
// odd-even merge sort, 19).
template <int K>
__device__ __forceinline__ void sort_net(float* x) {
  if constexpr (K == 4) {
    ce(x[0], x[1]); ce(x[2], x[3]); ce(x[0], x[2]); ce(x[1], x[3]); ce(x[1], x[2]);
  } else {
    ce(x[0], x[1]); ce(x[2], x[3]); ce(x[4], x[5]); ce(x[6], x[7]);
    ce(x[0], x[2]); ce(x[1], x[3]); ce(x[4], x[6]); ce(x[5], x[7]);
    ce(x[1], x[2]); ce(x[5], x[6]);
    ce(x[0], x[4]); ce(x[1], x[5]); ce(x[2], x[6]); ce(x[3], x[7]);
    ce(x[2], x[4]); ce(x[3], x[5]);
    ce(x[1], x[2]); ce(x[3], x[4]); ce(x[5], x[6]);
  }
}
// a <- the K largest of a and b, both sorted descending: the larger of a[i] and
// b[K-1-i] are the K largest and form a bitonic sequence, which a bitonic merge sorts.
__device__ __forceinline__ float max_of(float a, float b) { return fmaxf(a, b); }
__device__ __forceinline__ unsigned long long max_of(unsigned long long a, unsigned long long b) { return a > b ? a : b; }
__device__ __forceinline__ void cex(float& a, float& b) { ce(a, b); }
__device__ __forceinline__ void cex(unsigned long long& a, unsigned long long& b) { ce64(a, b); }
template <int K, typename T>
__device__ __forceinline__ void merge_top(T* a, const T* b) {
#pragma unroll
  for (int i = 0; i < K; ++i) a[i] = max_of(a[i], b[K - 1 - i]);
#pragma unroll
  for (int w = K / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < K; ++i)
      if ((i & w) == 0) cex(a[i], a[i + w]);
}
}  // namespace serac
