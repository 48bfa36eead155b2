// fm_localize.cu — clip-shift-max mask localization, and the bounded-wait self-test.
//
// FlashMask-3 project page, §3.2 ("Zero-communication mask localization"):
// a rank that owns kappa chunks of C query rows starting at global rows
// O_0 < O_1 < ... renumbers every global row boundary x into its own rows as
//   x_local = max_i [ clip(x - O_i, 0, C) + i*C*1(clip(x - O_i, 0, C) > 0) ],
// the number of the rank's rows before global row x. Elementwise over all
// boundary values; the offsets sit in shared memory; loads and stores are
// coalesced (int4 where the pointers allow it).
#include "fm_internal.h"
#include "sm100.cuh"

namespace fm {
namespace {

constexpr int kMaxKappa = 4096;

__device__ __forceinline__ int32_t localize_one(int32_t x, const int32_t* off, int kappa, int C) {
  long long best = 0;
  for (int i = 0; i < kappa; ++i) {
    long long c = (long long)x - off[i];
    c = c < 0 ? 0 : (c > C ? C : c);
    const long long v = c + (c > 0 ? (long long)i * C : 0);
    best = v > best ? v : best;
  }
  return (int32_t)best;
}

__global__ void localize_kernel(const int32_t* __restrict__ x, int64_t n, const int32_t* __restrict__ off, int kappa,
                                int C, int32_t* __restrict__ out) {
  __shared__ int32_t s_off[kMaxKappa];
  for (int i = threadIdx.x; i < kappa; i += blockDim.x) s_off[i] = off[i];
  __syncthreads();
  const bool vec = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) == 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (vec) {
    const int64_t n4 = n >> 2;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += stride) {
      int4 v = reinterpret_cast<const int4*>(x)[t];
      v.x = localize_one(v.x, s_off, kappa, C);
      v.y = localize_one(v.y, s_off, kappa, C);
      v.z = localize_one(v.z, s_off, kappa, C);
      v.w = localize_one(v.w, s_off, kappa, C);
      reinterpret_cast<int4*>(out)[t] = v;
    }
    for (int64_t t = (n4 << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride)
      out[t] = localize_one(x[t], s_off, kappa, C);
  } else {
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += stride)
      out[t] = localize_one(x[t], s_off, kappa, C);
  }
}

// One CTA waits on an mbarrier that nothing arrives at; the bounded wait must
// expire, record FM_DEV_ERR_TIMEOUT and return.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_localize(const int32_t* x, int64_t n, const int32_t* off, int kappa, int C, int32_t* out,
                            cudaStream_t s) {
  if (kappa > kMaxKappa) return cudaErrorInvalidValue;
  const int64_t items = (n + 3) / 4;
  int64_t blocks = (items + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  localize_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, n, off, kappa, C, out);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s, int* err) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fm
