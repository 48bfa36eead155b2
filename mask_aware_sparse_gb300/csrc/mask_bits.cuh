// mask_bits.cuh — bit-matrix helpers for applying the column-wise interval
// mask (FlashMask project page §3.1: key column j is masked for rows in
// [LTS_j, LTE_j) and [UTS_j, UTE_j)) to 32-row windows of a tile.
#pragma once
#include <cstdint>

namespace fm {

// Bits [a, b) of a 32-bit word (clipped to [0, 32)); 0 when the range is empty.
__device__ __forceinline__ uint32_t rows_bits(int a, int b) {
  a = max(a, 0);
  b = min(b, 32);
  if (a >= b) return 0u;
  const uint32_t hi = (b == 32) ? 0xffffffffu : ((1u << b) - 1u);
  return hi & ~((1u << a) - 1u);
}

// Bits of the rows [a, b) that fall in the 32-row window [w0, w0 + 32), as
// offsets from w0. Any int32 a, b (no overflow): the bounds are first clamped
// to the window, which for rows of the window is the same as clamping them
// to [0, N].
__device__ __forceinline__ uint32_t window_bits(int a, int b, int w0) {
  const int lo = min(max(a, w0), w0 + 32) - w0;
  const int hi = min(max(b, w0), w0 + 32) - w0;
  const uint32_t hm = (hi >= 32) ? 0xffffffffu : ((1u << hi) - 1u);
  const uint32_t lm = (lo >= 32) ? 0xffffffffu : ((1u << lo) - 1u);
  return hm & ~lm;  // empty when hi <= lo
}

// Transpose a 32 x 32 bit matrix held one row per lane (bit c of lane r's word
// is element (r, c)): on return lane r holds column r (bit c = element (c, r)).
// Recursive block swap: at step j, lanes exchange the off-diagonal j x j blocks
// of each 2j x 2j block with the lane j away.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint32_t m = (j == 16) ? 0x0000FFFFu
                       : (j == 8) ? 0x00FF00FFu
                       : (j == 4) ? 0x0F0F0F0Fu
                       : (j == 2) ? 0x33333333u
                                  : 0x55555555u;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

}  // namespace fm
