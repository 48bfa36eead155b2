// fm_convert.cu — the FlashMask Guide's FMS / FME vectors as the four boundary vectors.
//
// FlashMask Guide, "The Solution: FlashMask Sparse Mask Representation"
// ("Column-Wise Sparse Representation"): key column j is visible exactly to
// query rows FMS_j <= i <= FME_j, one inclusive interval, causality written
// into FMS. Its complement is two masked intervals, [0, FMS_j) and
// [FME_j + 1, N), i.e. UTS = 0, UTE = FMS, LTS = FME + 1, LTE = N, each
// clipped to [0, N]; the result is used with causal off. Elementwise over
// every column of every batch entry, int4 loads and stores where aligned.
#include "fm_internal.h"

namespace fm {
namespace {

__device__ __forceinline__ int32_t clip_rows(long long x, int n) { return (int32_t)(x < 0 ? 0 : (x > n ? n : x)); }

__global__ void from_fms_fme_kernel(const int32_t* __restrict__ fms, const int32_t* __restrict__ fme, int64_t m,
                                    int n, int32_t* __restrict__ lts, int32_t* __restrict__ lte,
                                    int32_t* __restrict__ uts, int32_t* __restrict__ ute) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(fms) | reinterpret_cast<uintptr_t>(fme) |
                     reinterpret_cast<uintptr_t>(lts) | reinterpret_cast<uintptr_t>(lte) |
                     reinterpret_cast<uintptr_t>(uts) | reinterpret_cast<uintptr_t>(ute)) & 15) == 0;
  int64_t done = 0;
  if (vec) {
    const int64_t m4 = m >> 2;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < m4; t += stride) {
      const int4 s = reinterpret_cast<const int4*>(fms)[t];
      const int4 e = reinterpret_cast<const int4*>(fme)[t];
      reinterpret_cast<int4*>(lts)[t] = make_int4(clip_rows((long long)e.x + 1, n), clip_rows((long long)e.y + 1, n),
                                                  clip_rows((long long)e.z + 1, n), clip_rows((long long)e.w + 1, n));
      reinterpret_cast<int4*>(lte)[t] = make_int4(n, n, n, n);
      reinterpret_cast<int4*>(uts)[t] = make_int4(0, 0, 0, 0);
      reinterpret_cast<int4*>(ute)[t] = make_int4(clip_rows(s.x, n), clip_rows(s.y, n), clip_rows(s.z, n),
                                                  clip_rows(s.w, n));
    }
    done = m4 << 2;
  }
  for (int64_t t = done + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < m; t += stride) {
    lts[t] = clip_rows((long long)fme[t] + 1, n);
    lte[t] = n;
    uts[t] = 0;
    ute[t] = clip_rows(fms[t], n);
  }
}

}  // namespace

cudaError_t launch_from_fms_fme(const int32_t* fms, const int32_t* fme, int64_t m, int n, int32_t* lts, int32_t* lte,
                                int32_t* uts, int32_t* ute, cudaStream_t s) {
  int64_t blocks = ((m + 3) / 4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  from_fms_fme_kernel<<<(unsigned)blocks, 256, 0, s>>>(fms, fme, m, n, lts, lte, uts, ute);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fm
