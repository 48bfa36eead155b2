// fm_multi.cu — merging the parts of a multi-interval mask.
//
// FlashMask Guide, after the DPO example: a key column may be visible to up
// to M disjoint row intervals [FMS^(m)_j, FME^(m)_j]. For a fixed query row
// the keys visible through different intervals are then disjoint sets, so
// softmax attention over their union is the log-sum-exp merge of one
// single-interval attention per interval (the online-softmax combination of
// "Flash MSA Attention Kernel Implementation", "The Flash Core", applied to
// whole partial results):
//   LSE = log sum_m exp(LSE_m),   O = sum_m exp(LSE_m - LSE) O_m,
// and the gradients are the sums of the parts' backward passes taken with the
// merged O and LSE. merge_parts_kernel does the first, sum_parts_kernel the
// second; both are elementwise and read / write 16 bytes per thread.
#include <cuda_bf16.h>
#include "fm_internal.h"

namespace fm {
namespace {

struct Parts {
  const __nv_bfloat16* o[kMaxParts];
  const float* lse[kMaxParts];
};

// one thread per 8 output elements of a row (d / 8 threads per row)
__global__ void merge_parts_kernel(Parts parts, int M, int64_t rows, int d, __nv_bfloat16* __restrict__ o,
                                   float* __restrict__ lse) {
  const int per_row = d >> 3;
  const int64_t n = rows * per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / per_row;
    const int c = (int)(t - r * per_row);
    float l[kMaxParts];
    float top = -INFINITY;
    for (int m = 0; m < M; ++m) {
      l[m] = parts.lse[m][r];
      top = fmaxf(top, l[m]);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float L = -INFINITY;
    if (top != -INFINITY) {
      float s = 0.f;
      for (int m = 0; m < M; ++m) s += (l[m] == -INFINITY) ? 0.f : expf(l[m] - top);
      L = top + logf(s);
      for (int m = 0; m < M; ++m) {
        if (l[m] == -INFINITY) continue;
        const float w = expf(l[m] - L);
        const uint4 raw = reinterpret_cast<const uint4*>(parts.o[m] + r * d)[c];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 f = __bfloat1622float2(h[x]);
          acc[2 * x] += w * f.x;
          acc[2 * x + 1] += w * f.y;
        }
      }
    }
    uint4 out;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
    for (int x = 0; x < 4; ++x) h[x] = __floats2bfloat162_rn(acc[2 * x], acc[2 * x + 1]);
    reinterpret_cast<uint4*>(o + r * d)[c] = out;
    if (c == 0) lse[r] = L;
  }
}

struct Addends {
  const __nv_bfloat16* p[kMaxParts];
};

// out = sum_m p[m] in fp32, rounded once; 8 elements per thread where the
// pointers and n allow it, element by element otherwise
__global__ void sum_parts_kernel(Addends a, int M, int64_t n, bool vec, __nv_bfloat16* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t done = 0;
  if (vec) {
    const int64_t n8 = n >> 3;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += stride) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int m = 0; m < M; ++m) {
        const uint4 raw = reinterpret_cast<const uint4*>(a.p[m])[t];
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 f = __bfloat1622float2(h[x]);
          acc[2 * x] += f.x;
          acc[2 * x + 1] += f.y;
        }
      }
      uint4 o;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int x = 0; x < 4; ++x) h[x] = __floats2bfloat162_rn(acc[2 * x], acc[2 * x + 1]);
      reinterpret_cast<uint4*>(out)[t] = o;
    }
    done = n8 << 3;
  }
  for (int64_t t = done + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride) {
    float s = 0.f;
    for (int m = 0; m < M; ++m) s += __bfloat162float(a.p[m][t]);
    out[t] = __float2bfloat16_rn(s);
  }
}

unsigned grid_for(int64_t items) {
  int64_t blocks = (items + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_merge_parts(int M, const void* const* o_parts, const float* const* lse_parts, int64_t rows, int d,
                               void* o, float* lse, cudaStream_t s) {
  Parts p = {};
  for (int m = 0; m < M; ++m) {
    p.o[m] = static_cast<const __nv_bfloat16*>(o_parts[m]);
    p.lse[m] = lse_parts[m];
  }
  merge_parts_kernel<<<grid_for(rows * (d / 8)), 256, 0, s>>>(p, M, rows, d, static_cast<__nv_bfloat16*>(o), lse);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_sum_parts(int M, const void* const* parts, int64_t n, void* out, cudaStream_t s) {
  Addends a = {};
  uintptr_t bits = reinterpret_cast<uintptr_t>(out);
  for (int m = 0; m < M; ++m) {
    a.p[m] = static_cast<const __nv_bfloat16*>(parts[m]);
    bits |= reinterpret_cast<uintptr_t>(parts[m]);
  }
  const bool vec = (bits & 15) == 0;
  sum_parts_kernel<<<grid_for(vec ? (n + 7) / 8 : n), 256, 0, s>>>(a, M, n, vec, static_cast<__nv_bfloat16*>(out));
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fm
