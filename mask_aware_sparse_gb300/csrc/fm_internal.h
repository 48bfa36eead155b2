// fm_internal.h — declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/fm.h"

namespace fm {

// Device error word of the current device (address of a __device__ int).
int* device_error_word();

// Classification (fm_classify.cu).
size_t classify_ws_bytes(int B, int nQ, int nK);
size_t classify_multi_ws_bytes(int M, int B, int nQ, int nK, int Nk);
cudaError_t launch_classify_multi(const fm_problem& p, int M, int bm, int bn, int nQ, int nK, const int32_t* fms,
                                  const int32_t* fme, uint8_t* tile_class, int32_t* q_off, int32_t* q_queue,
                                  int32_t* k_off, int32_t* k_queue, void* ws, cudaStream_t s, int* err);
cudaError_t launch_classify(const fm_problem& p, int bm, int bn, int nQ, int nK, const int32_t* lts,
                            const int32_t* lte, const int32_t* uts, const int32_t* ute, uint8_t* tile_class,
                            int32_t* q_off, int32_t* q_queue, int32_t* k_off, int32_t* k_queue, void* ws,
                            cudaStream_t s, int* err);

// Localization (fm_localize.cu).
// parts of a multi-interval mask (fm_multi.cu)
constexpr int kMaxParts = 8;
cudaError_t launch_merge_parts(int M, const void* const* o_parts, const float* const* lse_parts, int64_t rows, int d,
                               void* o, float* lse, cudaStream_t s);
cudaError_t launch_sum_parts(int M, const void* const* parts, int64_t n, void* out, cudaStream_t s);
cudaError_t launch_from_fms_fme(const int32_t* fms, const int32_t* fme, int64_t m, int n, int32_t* lts, int32_t* lte,
                                int32_t* uts, int32_t* ute, cudaStream_t s);
cudaError_t launch_localize(const int32_t* x, int64_t n, const int32_t* off, int kappa, int C, int32_t* out,
                            cudaStream_t s);

// Bounded-wait self-test (fm_localize.cu).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t s, int* err);

// Forward (fm_fwd.cu).
size_t fwd_ws_bytes(const fm_problem& p);
cudaError_t launch_fwd(const fm_problem& p, const void* q, const void* k, const void* v, const int32_t* lts,
                       const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                       const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err);

// Forward with per-head mask vectors (fm_fwd.cu): vectors (B, H_q, N_kv) and
// queues of a classification over B * H_q rows; one head per work unit.
size_t fwd_heads_ws_bytes(const fm_problem& p);
cudaError_t launch_fwd_heads(const fm_problem& P, const void* q, const void* k, const void* v, const int32_t* lts,
                             const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                             const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err);

// FP8 forward (fm_fwd.cu): e4m3 Q / K / V (value = stored x scale), d = 128,
// bf16 O; same workspace as launch_fwd.
cudaError_t launch_fwd_fp8(const fm_problem& P, const void* q, const void* k, const void* v, float q_scale,
                           float k_scale, float v_scale, const int32_t* lts, const int32_t* lte, const int32_t* uts,
                           const int32_t* ute, const int32_t* q_off, const int32_t* q_queue, void* o, float* lse,
                           void* ws, cudaStream_t s, int* err);

// Forward for d = 256 (fm_fwd256.cu): same arguments and workspace as launch_fwd.
cudaError_t launch_fwd256(const fm_problem& p, const void* q, const void* k, const void* v, const int32_t* lts,
                          const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                          const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err,
                          bool per_head = false, int M = 0);
// Multi-interval masks: FMS / FME (M, B, N_kv), the union classification's
// queues (M >= 1).
cudaError_t launch_fwd_multi(const fm_problem& P, int M, const void* q, const void* k, const void* v,
                             const int32_t* fms, const int32_t* fme, const int32_t* q_off, const int32_t* q_queue,
                             void* o, float* lse, void* ws, cudaStream_t s, int* err);

// The forward's fixed scratch for fm_attn_fwd_noalloc (fm_fwd.cu): device
// address of the library-owned launch-order array of the current device, or
// nullptr if it could not be looked up.
int32_t* fwd_noalloc_scratch();

// Backward (fm_bwd.cu).
size_t bwd_ws_bytes(const fm_problem& p);
cudaError_t launch_bwd(const fm_problem& p, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, const int32_t* lts, const int32_t* lte,
                       const int32_t* uts, const int32_t* ute, const int32_t* k_off, const int32_t* k_queue,
                       void* dq, void* dk, void* dv, void* ws, cudaStream_t s, int* err, bool per_head = false,
                       int M = 0);  // M >= 1: multi-interval masks (lts / lte hold FMS / FME, (M, B, N_kv))

// Main kernel of the d = 256 backward (fm_bwd256.cu); row terms, launch
// order and dQ conversion come from launch_bwd.
cudaError_t launch_bwd256_main(const fm_problem& P, const void* q, const void* k, const void* v, const void* dout,
                               const int32_t* lts, const int32_t* lte, const int32_t* uts, const int32_t* ute,
                               const int32_t* k_off, const int32_t* k_queue, const int32_t* order, const float* nl,
                               const float* dsum, float* dq_acc, void* dk, void* dv, cudaStream_t s, int* err,
                               int mode = 0, int M = 0);  // mode: 0 shared, 1 per-head, 2 multi-interval masks

// Number of SMs of the current device (cached per device).
int sm_count();

// Natural launch order beats longest-queue-first once a pass spans many
// waves of CTAs: CTAs that run together then share K / V (forward) or Q / dO
// (backward) tiles in L2, and the tail is a small part of the pass.
inline bool use_natural_order(long long ctas) { return ctas >= 8LL * sm_count(); }

// Tensor maps (fm_api.cu): 3-D bf16 map over a contiguous (BH, N, d) tensor,
// box {64, box_rows, 1}, 128-byte swizzle; rows >= N read as zero.
bool make_tmap_bhnd(void* out_tmap /* CUtensorMap* */, const void* base, int64_t BH, int64_t N, int64_t d,
                    int box_rows = 128);
// Same for a one-byte (e4m3) (BH, N, d) tensor: box {128, 128, 1}, 128-byte swizzle.
bool make_tmap_u8_bhnd(void* out_tmap /* CUtensorMap* */, const void* base, int64_t BH, int64_t N, int64_t d);
// Same for an fp32 (BH, N, d) tensor, box {box_cols, box_rows, 1}, no swizzle
// (used as the destination of TMA reduce-adds).
bool make_tmap_f32_bhnd(void* out_tmap /* CUtensorMap* */, const void* base, int64_t BH, int64_t N, int64_t d,
                        int box_cols, int box_rows);
// Same bf16 tensor, box {32, 32, 1}, 64-byte swizzle: one warp's 32 rows x 32
// columns of a store (rows >= N are not written).
bool make_tmap_bhnd_w32(void* out_tmap /* CUtensorMap* */, const void* base, int64_t BH, int64_t N, int64_t d);

constexpr int kTile = 128;  // attention tile (block_m = block_n)

// Key / value rows of a problem (N_kv = 0 stands for N_kv = N).
inline int kv_rows(const fm_problem& p) { return p.N_kv > 0 ? p.N_kv : p.N; }

// Launch accounting and optional event timing of the main kernels (fm_api.cu).
void count_launches(int n);
enum { kTimedFwd = 0, kTimedBwd = 1 };
// Records an event before the launch it brackets and one after (destructor),
// when fm_profile_enable(1) is in effect.
class KernelTimer {
 public:
  KernelTimer(cudaStream_t s, int kind);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  cudaStream_t s_;
  int kind_;
  void* a_ = nullptr;
  void* b_ = nullptr;
};

}  // namespace fm
