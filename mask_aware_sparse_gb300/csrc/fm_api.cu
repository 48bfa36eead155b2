// fm_api.cu — the extern "C" boundary: argument validation, workspace
// sizing, tensor-map encoding and the device error word. Every compute entry
// point validates on the host, then enqueues kernels on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>
#include <cuda.h>
#include <cudaTypedefs.h>
#include "fm_internal.h"

namespace fm {

// One error word per device; kernels OR FM_DEV_ERR_* bits into it.
static __device__ int g_error_word = 0;

int* device_error_word() {
  static std::mutex mu;
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(ptr);
  }
  return cached[dev];
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_tmap_bhnd(void* out, const void* base, int64_t BH, int64_t N, int64_t d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(N * d * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8_bhnd(void* out, const void* base, int64_t BH, int64_t N, int64_t d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)(N * d)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32_bhnd(void* out, const void* base, int64_t BH, int64_t N, int64_t d, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 4), (cuuint64_t)(N * d * 4)};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bhnd_w32(void* out, const void* base, int64_t BH, int64_t N, int64_t d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(N * d * 2)};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// ---------------------------------------------------------------- measurement
namespace {
std::atomic<long long> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
  cudaEvent_t a, b;
  int kind;
};
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

KernelTimer::KernelTimer(cudaStream_t s, int kind) : s_(s), kind_(kind) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on) return;
  cudaEvent_t a = take_event(), b = take_event();
  if (!a || !b) return;
  if (cudaEventRecord(a, s_) != cudaSuccess) return;
  a_ = a;
  b_ = b;
}

KernelTimer::~KernelTimer() {
  if (!a_) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEvent_t a = static_cast<cudaEvent_t>(a_), b = static_cast<cudaEvent_t>(b_);
  if (cudaEventRecord(b, s_) == cudaSuccess) g_recs.push_back({a, b, kind_});
}

}  // namespace fm

using namespace fm;

namespace {

bool valid_tile(int x) { return x == 32 || x == 64 || x == 128 || x == 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Shape checks shared by every attention-side call. *empty is set when there
// is nothing to compute (B, H_q or N is zero).
fm_status check_problem(const fm_problem* p, bool* empty) {
  if (!p) return FM_ERR_INVALID_ARG;
  if (p->B < 0 || p->H_q < 0 || p->H_kv < 0 || p->N < 0 || p->N_kv < 0 || p->d <= 0) return FM_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale)) return FM_ERR_INVALID_ARG;
  *empty = (p->B == 0 || p->H_q == 0 || p->N == 0);
  if (*empty) return FM_OK;
  if (p->H_kv == 0 || p->H_q % p->H_kv != 0) return FM_ERR_INVALID_ARG;
  // int32 indexing limits of the kernels: rows of one head and heads per batch
  if ((int64_t)p->B * p->H_q > (1 << 30) || (int64_t)p->N > (1 << 30) || (int64_t)p->N_kv > (1 << 30))
    return FM_ERR_UNSUPPORTED;
  return FM_OK;
}

// Head dimensions with a kernel: 64, 128 and 256.
fm_status check_attn_shape(const fm_problem* p, bool /*backward*/) {
  if (p->d != 64 && p->d != 128 && p->d != 256) return FM_ERR_UNSUPPORTED;
  return FM_OK;
}

fm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FM_OK : FM_ERR_CUDA; }

}  // namespace

extern "C" {

int32_t fm_abi_version(void) { return FM_ABI_VERSION; }

const char* fm_status_string(fm_status s) {
  switch (s) {
    case FM_OK: return "ok";
    case FM_ERR_INVALID_ARG: return "invalid argument";
    case FM_ERR_UNSUPPORTED: return "unsupported shape";
    case FM_ERR_WORKSPACE: return "workspace missing or too small";
    case FM_ERR_CUDA: return "CUDA error";
    case FM_ERR_TIMEOUT: return "device wait timed out";
    case FM_ERR_DEVICE: return "device reported bad input";
  }
  return "unknown status";
}

fm_status fm_attn_tiling(fm_tiling* out) {
  if (!out) return FM_ERR_INVALID_ARG;
  out->block_m = kTile;
  out->block_n = kTile;
  return FM_OK;
}

fm_status fm_tile_counts(const fm_problem* p, const fm_tiling* t, int32_t* nq, int32_t* nk) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK) return st;
  if (!t || !valid_tile(t->block_m) || !valid_tile(t->block_n) || !nq || !nk) return FM_ERR_INVALID_ARG;
  *nq = (p->N + t->block_m - 1) / t->block_m;
  *nk = (kv_rows(*p) + t->block_n - 1) / t->block_n;
  return FM_OK;
}

size_t fm_classify_workspace_bytes(const fm_problem* p, const fm_tiling* t) {
  int32_t nq = 0, nk = 0;
  if (fm_tile_counts(p, t, &nq, &nk) != FM_OK) return 0;
  return classify_ws_bytes(p->B, nq, nk);
}

fm_status fm_classify_tiles(const fm_problem* p, const fm_tiling* t, const int32_t* lts, const int32_t* lte,
                            const int32_t* uts, const int32_t* ute, uint8_t* tile_class, int32_t* q_off,
                            int32_t* q_queue, int32_t* k_off, int32_t* k_queue, void* ws, size_t ws_bytes,
                            void* stream) {
  int32_t nq = 0, nk = 0;
  fm_status st = fm_tile_counts(p, t, &nq, &nk);
  if (st != FM_OK) return st;
  if (p->B == 0 || p->N == 0) return FM_OK;
  if (!lts || !lte || !uts || !ute || !tile_class || !q_off || !q_queue || !k_off || !k_queue)
    return FM_ERR_INVALID_ARG;
  if ((int64_t)p->B * nq * nk > INT32_MAX) return FM_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < classify_ws_bytes(p->B, nq, nk)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_classify(*p, t->block_m, t->block_n, nq, nk, lts, lte, uts, ute, tile_class, q_off, q_queue,
                                   k_off, k_queue, ws, static_cast<cudaStream_t>(stream), err));
}

size_t fm_classify_multi_workspace_bytes(const fm_problem* p, const fm_tiling* t, int32_t M) {
  int32_t nq = 0, nk = 0;
  if (M < 1 || M > 4 || fm_tile_counts(p, t, &nq, &nk) != FM_OK) return 0;
  return classify_multi_ws_bytes(M, p->B, nq, nk, kv_rows(*p));
}

fm_status fm_classify_tiles_multi(const fm_problem* p, const fm_tiling* t, int32_t M, const int32_t* fms,
                                  const int32_t* fme, uint8_t* tile_class, int32_t* q_off, int32_t* q_queue,
                                  int32_t* k_off, int32_t* k_queue, void* ws, size_t ws_bytes, void* stream) {
  int32_t nq = 0, nk = 0;
  fm_status st = fm_tile_counts(p, t, &nq, &nk);
  if (st != FM_OK) return st;
  if (M < 1 || M > 4) return FM_ERR_INVALID_ARG;
  if (p->B == 0 || p->N == 0) return FM_OK;
  if (!fms || !fme || !tile_class || !q_off || !q_queue || !k_off || !k_queue) return FM_ERR_INVALID_ARG;
  if ((int64_t)M * p->B * nq * nk > INT32_MAX || (int64_t)M * p->B * kv_rows(*p) > INT32_MAX)
    return FM_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < classify_multi_ws_bytes(M, p->B, nq, nk, kv_rows(*p))) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_classify_multi(*p, M, t->block_m, t->block_n, nq, nk, fms, fme, tile_class, q_off,
                                         q_queue, k_off, k_queue, ws, static_cast<cudaStream_t>(stream), err));
}

size_t fm_attn_fwd_workspace_bytes(const fm_problem* p) {
  bool empty = false;
  if (check_problem(p, &empty) != FM_OK || empty) return 0;
  return fwd_ws_bytes(*p);
}

fm_status fm_attn_fwd(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                      const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                      const int32_t* q_queue, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if ((st = check_attn_shape(p, false)) != FM_OK) return st;
  if (!q || !k || !v || !lts || !lte || !uts || !ute || !q_off || !q_queue || !o || !lse) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  const size_t need = fwd_ws_bytes(*p);
  if (need > 0 && (!ws || ws_bytes < need)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_fwd(*p, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws,
                              static_cast<cudaStream_t>(stream), err));
}

size_t fm_attn_fwd_heads_workspace_bytes(const fm_problem* p) {
  bool empty = false;
  if (check_problem(p, &empty) != FM_OK || empty) return 0;
  return fwd_heads_ws_bytes(*p);
}

// Per-head masks: at most 64 query heads per kv head (the backward stages one
// queue per head of a group).
static fm_status check_heads_shape(const fm_problem* p) {
  if (check_attn_shape(p, false) != FM_OK) return FM_ERR_UNSUPPORTED;
  if (p->H_q / p->H_kv > 64) return FM_ERR_UNSUPPORTED;
  return FM_OK;
}

fm_status fm_attn_fwd_heads(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                            const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                            const int32_t* q_queue, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if ((st = check_heads_shape(p)) != FM_OK) return st;
  if (!q || !k || !v || !lts || !lte || !uts || !ute || !q_off || !q_queue || !o || !lse) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < fwd_heads_ws_bytes(*p)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_fwd_heads(*p, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws,
                                    static_cast<cudaStream_t>(stream), err));
}

fm_status fm_attn_bwd_heads(const fm_problem* p, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, const int32_t* lts, const int32_t* lte,
                            const int32_t* uts, const int32_t* ute, const int32_t* k_off, const int32_t* k_queue,
                            void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if ((st = check_heads_shape(p)) != FM_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !lts || !lte || !uts || !ute || !k_off || !k_queue || !dq || !dk ||
      !dv)
    return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < bwd_ws_bytes(*p)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_bwd(*p, q, k, v, o, lse, dout, lts, lte, uts, ute, k_off, k_queue, dq, dk, dv, ws,
                              static_cast<cudaStream_t>(stream), err, true));
}

fm_status fm_attn_fwd_multi(const fm_problem* p, int32_t M, const void* q, const void* k, const void* v,
                            const int32_t* fms, const int32_t* fme, const int32_t* q_off, const int32_t* q_queue,
                            void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK) return st;
  if (M < 1 || M > 4) return FM_ERR_INVALID_ARG;
  if (empty) return FM_OK;
  if ((st = check_attn_shape(p, false)) != FM_OK) return st;
  if (!q || !k || !v || !fms || !fme || !q_off || !q_queue || !o || !lse) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < fwd_ws_bytes(*p)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_fwd_multi(*p, M, q, k, v, fms, fme, q_off, q_queue, o, lse, ws,
                                    static_cast<cudaStream_t>(stream), err));
}

fm_status fm_attn_bwd_multi(const fm_problem* p, int32_t M, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, const int32_t* fms,
                            const int32_t* fme, const int32_t* k_off, const int32_t* k_queue, void* dq, void* dk,
                            void* dv, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK) return st;
  if (M < 1 || M > 4) return FM_ERR_INVALID_ARG;
  if (empty) return FM_OK;
  if ((st = check_attn_shape(p, true)) != FM_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !fms || !fme || !k_off || !k_queue || !dq || !dk || !dv)
    return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < bwd_ws_bytes(*p)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_bwd(*p, q, k, v, o, lse, dout, fms, fme, nullptr, nullptr, k_off, k_queue, dq, dk, dv, ws,
                              static_cast<cudaStream_t>(stream), err, false, M));
}

fm_status fm_attn_fwd_fp8(const fm_problem* p, const void* q, const void* k, const void* v, float q_scale,
                          float k_scale, float v_scale, const int32_t* lts, const int32_t* lte, const int32_t* uts,
                          const int32_t* ute, const int32_t* q_off, const int32_t* q_queue, void* o, float* lse,
                          void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if (p->d != 128) return FM_ERR_UNSUPPORTED;
  for (float x : {q_scale, k_scale, v_scale})
    if (!std::isfinite(x) || x <= 0.f) return FM_ERR_INVALID_ARG;
  if (!q || !k || !v || !lts || !lte || !uts || !ute || !q_off || !q_queue || !o || !lse) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  const size_t need = fwd_ws_bytes(*p);
  if (need > 0 && (!ws || ws_bytes < need)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_fwd_fp8(*p, q, k, v, q_scale, k_scale, v_scale, lts, lte, uts, ute, q_off, q_queue, o, lse,
                                  ws, static_cast<cudaStream_t>(stream), err));
}

fm_status fm_attn_fwd_noalloc(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                              const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                              const int32_t* q_queue, void* o, float* lse, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if ((st = check_attn_shape(p, false)) != FM_OK) return st;
  if (!q || !k || !v || !lts || !lte || !uts || !ute || !q_off || !q_queue || !o || !lse) return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FM_ERR_INVALID_ARG;
  // the fixed scratch holds one entry per Q block of the whole batch
  const int64_t qblocks = (int64_t)p->B * ((p->N + kTile - 1) / kTile);
  if (qblocks > FM_NOALLOC_MAX_QBLOCKS) return FM_ERR_WORKSPACE;
  int32_t* scratch = fwd_noalloc_scratch();
  int* err = device_error_word();
  if (!scratch || !err) return FM_ERR_CUDA;
  return from_cuda(launch_fwd(*p, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, scratch,
                              static_cast<cudaStream_t>(stream), err));
}

size_t fm_attn_bwd_workspace_bytes(const fm_problem* p) {
  bool empty = false;
  if (check_problem(p, &empty) != FM_OK || empty) return 0;
  return bwd_ws_bytes(*p);
}

fm_status fm_attn_bwd(const fm_problem* p, const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, const int32_t* lts, const int32_t* lte,
                      const int32_t* uts, const int32_t* ute, const int32_t* k_off, const int32_t* k_queue,
                      void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream) {
  bool empty = false;
  fm_status st = check_problem(p, &empty);
  if (st != FM_OK || empty) return st;
  if ((st = check_attn_shape(p, true)) != FM_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !lts || !lte || !uts || !ute || !k_off || !k_queue || !dq || !dk ||
      !dv)
    return FM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < bwd_ws_bytes(*p)) return FM_ERR_WORKSPACE;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_bwd(*p, q, k, v, o, lse, dout, lts, lte, uts, ute, k_off, k_queue, dq, dk, dv, ws,
                              static_cast<cudaStream_t>(stream), err));
}

fm_status fm_localize(const int32_t* x_global, int64_t n, const int32_t* chunk_off, int32_t kappa, int32_t C,
                      int32_t* x_local, void* stream) {
  if (n < 0 || kappa < 1 || kappa > 4096 || C < 1) return FM_ERR_INVALID_ARG;
  if (n == 0) return FM_OK;
  if (!x_global || !chunk_off || !x_local) return FM_ERR_INVALID_ARG;
  return from_cuda(launch_localize(x_global, n, chunk_off, kappa, C, x_local, static_cast<cudaStream_t>(stream)));
}

fm_status fm_from_fms_fme(const int32_t* fms, const int32_t* fme, int64_t n_values, int32_t N, int32_t* lts,
                          int32_t* lte, int32_t* uts, int32_t* ute, void* stream) {
  if (n_values < 0 || N < 0 || N > (1 << 30)) return FM_ERR_INVALID_ARG;
  if (n_values == 0) return FM_OK;
  if (!fms || !fme || !lts || !lte || !uts || !ute) return FM_ERR_INVALID_ARG;
  return from_cuda(
      launch_from_fms_fme(fms, fme, n_values, N, lts, lte, uts, ute, static_cast<cudaStream_t>(stream)));
}

fm_status fm_merge_parts(int32_t M, const void* const* o_parts, const float* const* lse_parts, int64_t rows,
                         int32_t d, void* o, float* lse, void* stream) {
  if (M < 1 || M > kMaxParts || rows < 0 || d < 8 || d % 8 != 0) return FM_ERR_INVALID_ARG;
  if (rows == 0) return FM_OK;
  if (!o_parts || !lse_parts || !o || !lse || !aligned16(o)) return FM_ERR_INVALID_ARG;
  for (int m = 0; m < M; ++m)
    if (!o_parts[m] || !lse_parts[m] || !aligned16(o_parts[m])) return FM_ERR_INVALID_ARG;
  return from_cuda(launch_merge_parts(M, o_parts, lse_parts, rows, d, o, lse, static_cast<cudaStream_t>(stream)));
}

fm_status fm_sum_parts(int32_t M, const void* const* parts, int64_t n, void* out, void* stream) {
  if (M < 1 || M > kMaxParts || n < 0) return FM_ERR_INVALID_ARG;
  if (n == 0) return FM_OK;
  if (!parts || !out) return FM_ERR_INVALID_ARG;
  for (int m = 0; m < M; ++m)
    if (!parts[m]) return FM_ERR_INVALID_ARG;
  return from_cuda(launch_sum_parts(M, parts, n, out, static_cast<cudaStream_t>(stream)));
}

fm_status fm_device_status(void* stream, int32_t* bits) {
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FM_ERR_CUDA;
  int host = 0;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FM_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FM_ERR_CUDA;
  }
  if (bits) *bits = host;
  if (host == 0) return FM_OK;
  return (host & FM_DEVERR_TIMEOUT) ? FM_ERR_TIMEOUT : FM_ERR_DEVICE;
}

fm_status fm_selftest_wait_timeout(int64_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 10000000) return FM_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (!err) return FM_ERR_CUDA;
  return from_cuda(launch_wait_selftest((uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream), err));
}

fm_status fm_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
  return FM_OK;
}

fm_status fm_profile_read(double* fwd_ms, int32_t* fwd_launches, double* bwd_ms, int32_t* bwd_launches) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    recs.swap(g_recs);
  }
  double ms[2] = {0.0, 0.0};
  int32_t cnt[2] = {0, 0};
  fm_status st = FM_OK;
  for (const ProfRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) st = FM_ERR_CUDA;
    ms[r.kind] += t;
    cnt[r.kind] += 1;
  }
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (const ProfRec& r : recs) {
      g_pool.push_back(r.a);
      g_pool.push_back(r.b);
    }
  }
  if (fwd_ms) *fwd_ms = ms[0];
  if (fwd_launches) *fwd_launches = cnt[0];
  if (bwd_ms) *bwd_ms = ms[1];
  if (bwd_launches) *bwd_launches = cnt[1];
  return st;
}

int64_t fm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
