// lpt_order.cuh — longest-queue-first launch order of the work units of a
// pass (one CTA): order[r] = the unit with the r-th longest queue, ties in
// index order. Queue lengths come from CSR offsets (off[i+1] - off[i]).
// Up to 1024 units: each thread ranks its unit against all others (a stable
// rank sort, no barriers in the loop); up to kMaxSort: bitonic sort of
// (length, -index) keys; beyond that, index order.
#pragma once
#include <cstdint>

namespace fm {
namespace {  // one copy per translation unit that launches it

constexpr int kLptMaxSort = 4096;

__global__ void __launch_bounds__(1024) lpt_order_kernel(const int32_t* __restrict__ off, int count,
                                                         int32_t* __restrict__ order) {
  __shared__ unsigned long long key[kLptMaxSort];
  if (count > kLptMaxSort) {
    for (int i = threadIdx.x; i < count; i += blockDim.x) order[i] = i;
    return;
  }
  if (count <= 1024) {
    int* len = reinterpret_cast<int*>(key);
    for (int i = threadIdx.x; i < count; i += blockDim.x) len[i] = off[i + 1] - off[i];
    __syncthreads();
    const int i = threadIdx.x;
    if (i < count) {
      const int li = len[i];
      int rank = 0;
      for (int j = 0; j < count; ++j) {
        const int lj = len[j];
        rank += (lj > li) | ((lj == li) & (j < i));
      }
      order[rank] = i;
    }
    return;
  }
  int n2 = 1;
  while (n2 < count) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += blockDim.x)
    key[i] = (i < count) ? (((unsigned long long)(uint32_t)(off[i + 1] - off[i]) << 32) | (0xFFFFFFFFu - (uint32_t)i))
                         : 0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const bool desc = (i & k) == 0;
          const unsigned long long a = key[i], c = key[ixj];
          if ((a < c) == desc) {
            key[i] = c;
            key[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < count; i += blockDim.x) order[i] = (int32_t)(0xFFFFFFFFu - (uint32_t)key[i]);
}

}  // namespace
}  // namespace fm
