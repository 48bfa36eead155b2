// fm_host.cpp — one forward + backward from host buffers: the C ABI entry
// point that copies a step's inputs to the device, runs classification,
// forward and backward, and copies every output back, all on the caller's
// stream and inside the caller's device workspace (the library allocates
// nothing here either).
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>
#include "../../include/fm.h"

namespace {

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// Device workspace of one host call: the device copies of every input and
// output, the queues, and the three kernels' own workspaces.
struct HostWs {
  size_t q, kv, lse, vec, cls, qoff, queue, koff, cws, fws, bws;  // sizes in bytes
  int32_t nq, nk;
  size_t total;
};

bool layout(const fm_problem* p, HostWs* w) {
  fm_tiling t;
  if (fm_attn_tiling(&t) != FM_OK) return false;
  if (fm_tile_counts(p, &t, &w->nq, &w->nk) != FM_OK) return false;
  const int64_t Nk = p->N_kv > 0 ? p->N_kv : p->N;
  const size_t B = (size_t)p->B;
  w->q = (size_t)B * p->H_q * p->N * p->d * 2;
  w->kv = (size_t)B * p->H_kv * Nk * p->d * 2;
  w->lse = (size_t)B * p->H_q * p->N * 4;
  w->vec = (size_t)B * Nk * 4;
  w->cls = B * (size_t)w->nq * w->nk;
  w->qoff = (B * w->nq + 1) * 4;
  w->queue = (w->cls > 0 ? w->cls : 1) * 4;
  w->koff = (B * w->nk + 1) * 4;
  w->cws = fm_classify_workspace_bytes(p, &t);
  w->fws = fm_attn_fwd_workspace_bytes(p);
  w->bws = fm_attn_bwd_workspace_bytes(p);
  w->total = 4 * a256(w->q) + 4 * a256(w->kv) + a256(w->lse) + 4 * a256(w->vec) + a256(w->cls) + a256(w->qoff) +
             2 * a256(w->queue) + a256(w->koff) + a256(w->cws) + a256(w->fws) + a256(w->bws);
  return true;
}

struct Carver {
  uint8_t* p;
  void* take(size_t n) {
    void* r = p;
    p += a256(n);
    return r;
  }
};

}  // namespace

extern "C" {

size_t fm_attn_host_workspace_bytes(const fm_problem* p) {
  if (!p || p->B <= 0 || p->H_q <= 0 || p->N <= 0) return 0;
  HostWs w;
  return layout(p, &w) ? w.total : 0;
}

fm_status fm_attn_fwd_bwd_host(const fm_problem* p, const void* q, const void* k, const void* v, const void* dout,
                               const int32_t* lts, const int32_t* lte, const int32_t* uts, const int32_t* ute,
                               void* o, float* lse, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                               void* stream) {
  if (!p) return FM_ERR_INVALID_ARG;
  if (p->B == 0 || p->H_q == 0 || p->N == 0) return FM_OK;
  if (p->B < 0 || p->H_q < 0 || p->N < 0) return FM_ERR_INVALID_ARG;
  if (!q || !k || !v || !dout || !lts || !lte || !uts || !ute || !o || !lse || !dq || !dk || !dv)
    return FM_ERR_INVALID_ARG;
  HostWs w;
  if (!layout(p, &w)) return FM_ERR_INVALID_ARG;
  if (!ws || ws_bytes < w.total) return FM_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Carver c{static_cast<uint8_t*>(ws)};
  void* d_q = c.take(w.q);
  void* d_do = c.take(w.q);
  void* d_o = c.take(w.q);
  void* d_dq = c.take(w.q);
  void* d_k = c.take(w.kv);
  void* d_v = c.take(w.kv);
  void* d_dk = c.take(w.kv);
  void* d_dv = c.take(w.kv);
  float* d_lse = static_cast<float*>(c.take(w.lse));
  int32_t* d_vec[4];
  for (int i = 0; i < 4; ++i) d_vec[i] = static_cast<int32_t*>(c.take(w.vec));
  uint8_t* d_cls = static_cast<uint8_t*>(c.take(w.cls));
  int32_t* d_qoff = static_cast<int32_t*>(c.take(w.qoff));
  int32_t* d_qq = static_cast<int32_t*>(c.take(w.queue));
  int32_t* d_koff = static_cast<int32_t*>(c.take(w.koff));
  int32_t* d_kq = static_cast<int32_t*>(c.take(w.queue));
  void* d_cws = c.take(w.cws);
  void* d_fws = c.take(w.fws);
  void* d_bws = c.take(w.bws);
  // inputs in: one copy per tensor
  const void* hin[8] = {q, k, v, dout, lts, lte, uts, ute};
  void* din[8] = {d_q, d_k, d_v, d_do, d_vec[0], d_vec[1], d_vec[2], d_vec[3]};
  const size_t nin[8] = {w.q, w.kv, w.kv, w.q, w.vec, w.vec, w.vec, w.vec};
  for (int i = 0; i < 8; ++i)
    if (cudaMemcpyAsync(din[i], hin[i], nin[i], cudaMemcpyHostToDevice, s) != cudaSuccess) return FM_ERR_CUDA;
  fm_tiling t;
  fm_status st = fm_attn_tiling(&t);
  if (st == FM_OK)
    st = fm_classify_tiles(p, &t, d_vec[0], d_vec[1], d_vec[2], d_vec[3], d_cls, d_qoff, d_qq, d_koff, d_kq, d_cws,
                           w.cws, stream);
  if (st == FM_OK)
    st = fm_attn_fwd(p, d_q, d_k, d_v, d_vec[0], d_vec[1], d_vec[2], d_vec[3], d_qoff, d_qq, d_o, d_lse, d_fws, w.fws,
                     stream);
  if (st == FM_OK)
    st = fm_attn_bwd(p, d_q, d_k, d_v, d_o, d_lse, d_do, d_vec[0], d_vec[1], d_vec[2], d_vec[3], d_koff, d_kq, d_dq,
                     d_dk, d_dv, d_bws, w.bws, stream);
  if (st != FM_OK) return st;
  // outputs back
  void* hout[5] = {o, lse, dq, dk, dv};
  const void* dout_[5] = {d_o, d_lse, d_dq, d_dk, d_dv};
  const size_t nout[5] = {w.q, w.lse, w.q, w.kv, w.kv};
  for (int i = 0; i < 5; ++i)
    if (cudaMemcpyAsync(hout[i], dout_[i], nout[i], cudaMemcpyDeviceToHost, s) != cudaSuccess) return FM_ERR_CUDA;
  return FM_OK;
}

}  // extern "C"
