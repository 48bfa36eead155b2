// fm_classify.cu — tile classification and compacted queue construction.
//
// FlashMask-3 project page, §3.1: block-wise min/max of LTS/LTE/UTS/UTE
// classify each (Q-block, KV-block) tile as skip / partial / unmasked and each
// Q block gets a queue of valid KV blocks tagged partial or unmasked, visited
// right to left. The rule (generalised to intervals that end inside the
// sequence, plus the causal term) is stated in include/fm.h.
//
// Pipeline (all int32, all on the caller's stream):
//   1. block_minmax   one warp per KV block: 8 reductions (min/max of the four
//                     vectors), coalesced loads + warp-shuffle reductions.
//   2. classify_rows  one CTA per (b, qb): class of every tile of the row,
//                     count of non-skipped tiles.
//      (the same kernel counts each column's non-skipped tiles with integer
//      atomics; block_minmax zeroes those counters first)
//   3. scan           exclusive prefix sums -> q_off, k_off (one CTA).
//   4. emit_queues    one warp per queue: (b, qb) rows in descending kb and
//                     (b, kb) columns in ascending qb, compaction by ballot.
#include <climits>
#include "fm_internal.h"
#include "sm100.cuh"

namespace fm {
namespace {

struct Minmax {
  int v[8];  // min LTS, max LTS, min LTE, max LTE, min UTS, max UTS, min UTE, max UTE
};

__device__ __forceinline__ int clamp_flag(int x, int n, bool& bad) {
  if (x < 0) { bad = true; return 0; }
  if (x > n) { bad = true; return n; }
  return x;
}

// N: query rows (the range of the values); Nk: key columns (the vectors' length)
__global__ void block_minmax_kernel(const int32_t* __restrict__ lts, const int32_t* __restrict__ lte,
                                    const int32_t* __restrict__ uts, const int32_t* __restrict__ ute, int B, int N,
                                    int Nk, int bn, int nK, Minmax* __restrict__ out, int32_t* __restrict__ col_cnt,
                                    int* err) {
  const int wpb = blockDim.x >> 5;
  const long long gw = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
  if (gw >= (long long)B * nK) return;
  const int lane = threadIdx.x & 31;
  const int b = (int)(gw / nK), kb = (int)(gw % nK);
  const int k0 = kb * bn, k1 = min(k0 + bn, Nk);
  const size_t base = (size_t)b * Nk;
  int mn[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX}, mx[4] = {INT_MIN, INT_MIN, INT_MIN, INT_MIN};
  bool bad = false;
  for (int j = k0 + lane; j < k1; j += 32) {
    const int x[4] = {clamp_flag(lts[base + j], N, bad), clamp_flag(lte[base + j], N, bad),
                      clamp_flag(uts[base + j], N, bad), clamp_flag(ute[base + j], N, bad)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mn[c] = min(mn[c], x[c]);
      mx[c] = max(mx[c], x[c]);
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(err, FM_DEV_ERR_RANGE);
  Minmax r;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    r.v[2 * c] = __reduce_min_sync(0xffffffffu, mn[c]);
    r.v[2 * c + 1] = __reduce_max_sync(0xffffffffu, mx[c]);
  }
  if (lane == 0) {
    out[gw] = r;
    col_cnt[gw] = 0;  // per-column tile counts, accumulated by classify_rows_kernel
  }
}

// Class of tile (q0,q1) x (k0,k1) from the block min/max.
__device__ __forceinline__ uint8_t tile_class(const Minmax& m, int q0, int q1, int k0, int k1, int causal) {
  const bool skip = (q0 >= m.v[1] && q1 <= m.v[2]) || (q0 >= m.v[5] && q1 <= m.v[6]) || (causal && q1 <= k0);
  if (skip) return 0;
  const bool unm = (q1 <= m.v[0] || q0 >= m.v[3]) && (q1 <= m.v[4] || q0 >= m.v[7]) && (!causal || q0 >= k1 - 1);
  return unm ? 2 : 1;
}

__global__ void classify_rows_kernel(const Minmax* __restrict__ mm, int N, int Nk, int bm, int bn, int nQ, int nK,
                                     int causal,
                                     uint8_t* __restrict__ cls, int32_t* __restrict__ row_cnt,
                                     int32_t* __restrict__ col_cnt) {
  const int b = blockIdx.y, qb = blockIdx.x;
  const int q0 = qb * bm, q1 = min(q0 + bm, N);
  int cnt = 0;
  uint8_t* crow = cls + ((size_t)b * nQ + qb) * nK;
  for (int kb = threadIdx.x; kb < nK; kb += blockDim.x) {
    const int k0 = kb * bn, k1 = min(k0 + bn, Nk);
    const uint8_t c = tile_class(mm[(size_t)b * nK + kb], q0, q1, k0, k1, causal);
    crow[kb] = c;
    cnt += (c != 0);
    if (c != 0) atomicAdd(&col_cnt[(size_t)b * nK + kb], 1);
  }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  __shared__ int part[32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
    row_cnt[(size_t)b * nQ + qb] = t;
  }
}

// Exclusive scan of cnt[0..n) into off[0..n] by one CTA of 1024 threads.
__device__ void block_exclusive_scan(const int32_t* __restrict__ cnt, int n, int32_t* __restrict__ off) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int x = (i < n) ? cnt[i] : 0;
    int incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sums[w] = incl;
    __syncthreads();
    if (w == 0) {
      int ws = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, ws, d);
        if (lane >= d) ws += y;
      }
      warp_sums[lane] = ws;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (w > 0 ? warp_sums[w - 1] : 0);
    if (i < n) off[i] = before + incl - x;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) off[n] = carry;
}

__global__ void scan_kernel(const int32_t* row_cnt, int n_rows, int32_t* q_off, const int32_t* col_cnt, int n_cols,
                            int32_t* k_off) {
  if (blockIdx.x == 0)
    block_exclusive_scan(row_cnt, n_rows, q_off);
  else
    block_exclusive_scan(col_cnt, n_cols, k_off);
}

// Queue emission, one warp per queue: warps [0, B*nQ) emit the Q-side queues
// (descending kb), warps [B*nQ, B*nQ + B*nK) the KV-side queues (ascending qb).
// Class bytes are loaded eight 32-entry chunks at a time before the ballots,
// so the loads are not serialised behind the running position.
__global__ void emit_queues_kernel(const uint8_t* __restrict__ cls, int B, int nQ, int nK,
                                   const int32_t* __restrict__ q_off, int32_t* __restrict__ q_queue,
                                   const int32_t* __restrict__ k_off, int32_t* __restrict__ k_queue) {
  const int wpb = blockDim.x >> 5;
  const long long w = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
  const long long nrow = (long long)B * nQ;
  if (w >= nrow + (long long)B * nK) return;
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  if (w < nrow) {
    const uint8_t* crow = cls + (size_t)w * nK;
    int pos = q_off[w];
    for (int top = nK - 1; top >= 0; top -= 256) {
      uint8_t c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int kb = top - 32 * i - lane;  // descending
        c[i] = (kb >= 0) ? crow[kb] : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int kb = top - 32 * i - lane;
        const unsigned bal = __ballot_sync(0xffffffffu, c[i] != 0);
        if (c[i] != 0) q_queue[pos + __popc(bal & below)] = (kb << 1) | (c[i] == 1 ? 1 : 0);
        pos += __popc(bal);
      }
    }
  } else {
    const long long r = w - nrow;
    const int b = (int)(r / nK), kb = (int)(r % nK);
    const uint8_t* ccol = cls + (size_t)b * nQ * nK + kb;
    int pos = k_off[r];
    for (int lo = 0; lo < nQ; lo += 256) {
      uint8_t c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int qb = lo + 32 * i + lane;  // ascending
        c[i] = (qb < nQ) ? ccol[(size_t)qb * nK] : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int qb = lo + 32 * i + lane;
        const unsigned bal = __ballot_sync(0xffffffffu, c[i] != 0);
        if (c[i] != 0) k_queue[pos + __popc(bal & below)] = (qb << 1) | (c[i] == 1 ? 1 : 0);
        pos += __popc(bal);
      }
    }
  }
}

// Multi-interval masks: the class of a tile is the most visible of the run
// slots' own classes (skip < partial < unmasked), one CTA per (b, qb):
// the row's classes, its count of non-skipped tiles and, by integer atomics,
// each column's (zeroed by the caller).
__global__ void union_classes_kernel(const uint8_t* __restrict__ cls_m, int M, int B, int nQ, int nK,
                                     uint8_t* __restrict__ cls, int32_t* __restrict__ row_cnt,
                                     int32_t* __restrict__ col_cnt) {
  const int qb = blockIdx.x, b = blockIdx.y;
  int cnt = 0;
  for (int kb = threadIdx.x; kb < nK; kb += blockDim.x) {
    uint8_t c = 0;
    for (int m = 0; m < M; ++m) {
      const uint8_t x = cls_m[(((size_t)m * B + b) * nQ + qb) * nK + kb];
      c = x > c ? x : c;
    }
    cls[((size_t)b * nQ + qb) * nK + kb] = c;
    if (c != 0) {
      ++cnt;
      atomicAdd(col_cnt + (size_t)b * nK + kb, 1);
    }
  }
  __shared__ int red[32];
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    row_cnt[(size_t)b * nQ + qb] = t;
  }
}

// Multi-interval masks: each key column's visible rows (the union of its M
// inclusive intervals [FMS, FME] within [0, n)) rewritten as their maximal
// runs, ascending, run k in slot k, and each slot's masked complement written
// as the four vectors of vector row (k * B + b): UTS = 0, UTE = start,
// LTS = end + 1, LTE = n. A slot past the last run is empty, start n and
// end -1 (UTE = n, LTS = 0: the whole column masked, without lowering the
// block's smallest UTE or raising its largest LTS). One thread per
// (b, column); the intervals are clipped, sorted by start and joined where
// one overlaps or touches the run before it, so the classes depend only on
// the mask.
__global__ void union_runs_kernel(const int32_t* __restrict__ fms, const int32_t* __restrict__ fme, int M, int B,
                                  int Nk, int n, int32_t* __restrict__ lts, int32_t* __restrict__ lte,
                                  int32_t* __restrict__ uts, int32_t* __restrict__ ute) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)B * Nk) return;
  const int b = (int)(t / Nk), j = (int)(t - (long long)b * Nk);
  int rs[4], re[4], cnt = 0;
  for (int m = 0; m < M; ++m) {
    const size_t vi = ((size_t)m * B + b) * Nk + j;
    const int a = max(fms[vi], 0), e = min(fme[vi], n - 1);
    if (a > e) continue;
    int k = cnt++;  // insertion by start
    while (k > 0 && rs[k - 1] > a) {
      rs[k] = rs[k - 1];
      re[k] = re[k - 1];
      --k;
    }
    rs[k] = a;
    re[k] = e;
  }
  int runs = 0;
  for (int k = 0; k < cnt; ++k) {
    if (runs > 0 && rs[k] <= re[runs - 1] + 1) {
      re[runs - 1] = max(re[runs - 1], re[k]);
    } else {
      rs[runs] = rs[k];
      re[runs] = re[k];
      ++runs;
    }
  }
  for (int k = 0; k < M; ++k) {
    const size_t vo = ((size_t)k * B + b) * Nk + j;
    const bool live = k < runs;
    lts[vo] = live ? re[k] + 1 : 0;
    lte[vo] = n;
    uts[vo] = 0;
    ute[vo] = live ? rs[k] : n;
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t classify_ws_bytes(int B, int nQ, int nK) {
  return align256(sizeof(Minmax) * (size_t)B * nK) + align256(4 * (size_t)B * nQ) + align256(4 * (size_t)B * nK);
}

// Multi-interval masks: the run slots' complements (M * B vector rows), their
// classes, the union classes and the queues.
size_t classify_multi_ws_bytes(int M, int B, int nQ, int nK, int Nk) {
  const size_t R = (size_t)M * B;
  return 4 * align256(4 * R * Nk) + classify_ws_bytes((int)R, nQ, nK) + align256(R * nQ * nK) +
         classify_ws_bytes(B, nQ, nK);
}

cudaError_t launch_classify_multi(const fm_problem& p, int M, int bm, int bn, int nQ, int nK, const int32_t* fms,
                                  const int32_t* fme, uint8_t* tile_class, int32_t* q_off, int32_t* q_queue,
                                  int32_t* k_off, int32_t* k_queue, void* ws, cudaStream_t s, int* err) {
  const int B = p.B, Nk = kv_rows(p);
  const size_t R = (size_t)M * B;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* vec[4];
  for (int i = 0; i < 4; ++i) {
    vec[i] = reinterpret_cast<int32_t*>(w);
    w += align256(4 * R * Nk);
  }
  void* ws_m = w;  // the per-interval classification
  w += classify_ws_bytes((int)R, nQ, nK);
  uint8_t* cls_m = w;
  w += align256(R * nQ * nK);
  uint8_t* wu = w;  // the union's: minmax (unused), row and column counts
  wu += align256(sizeof(Minmax) * (size_t)B * nK);
  int32_t* row_cnt = reinterpret_cast<int32_t*>(wu);
  wu += align256(4 * (size_t)B * nQ);
  int32_t* col_cnt = reinterpret_cast<int32_t*>(wu);
  const long long cols = (long long)B * Nk;
  union_runs_kernel<<<(unsigned)((cols + 255) / 256), 256, 0, s>>>(fms, fme, M, B, Nk, p.N, vec[0], vec[1], vec[2],
                                                                   vec[3]);
  fm_problem pm = p;
  pm.B = (int32_t)R;
  uint8_t* wm = static_cast<uint8_t*>(ws_m);
  Minmax* mm = reinterpret_cast<Minmax*>(wm);
  wm += align256(sizeof(Minmax) * R * nK);
  int32_t* row_cnt_m = reinterpret_cast<int32_t*>(wm);
  wm += align256(4 * R * nQ);
  int32_t* col_cnt_m = reinterpret_cast<int32_t*>(wm);
  block_minmax_kernel<<<(unsigned)((R * nK + 7) / 8), 256, 0, s>>>(vec[0], vec[1], vec[2], vec[3], (int)R, p.N, Nk,
                                                                   bn, nK, mm, col_cnt_m, err);
  classify_rows_kernel<<<dim3(nQ, (unsigned)R), 256, 0, s>>>(mm, p.N, Nk, bm, bn, nQ, nK, p.causal, cls_m,
                                                             row_cnt_m, col_cnt_m);
  cudaError_t e = cudaMemsetAsync(col_cnt, 0, 4 * (size_t)B * nK, s);
  if (e != cudaSuccess) return e;
  union_classes_kernel<<<dim3(nQ, B), 256, 0, s>>>(cls_m, M, B, nQ, nK, tile_class, row_cnt, col_cnt);
  const long long nkb = (long long)B * nK, nqb = (long long)B * nQ;
  scan_kernel<<<2, 1024, 0, s>>>(row_cnt, (int)nqb, q_off, col_cnt, (int)nkb, k_off);
  emit_queues_kernel<<<(unsigned)((nqb + nkb + 7) / 8), 256, 0, s>>>(tile_class, B, nQ, nK, q_off, q_queue, k_off,
                                                                     k_queue);
  count_launches(6);  // runs, minmax, classify rows, union, scan, emit
  return cudaGetLastError();
}

cudaError_t launch_classify(const fm_problem& p, int bm, int bn, int nQ, int nK, const int32_t* lts,
                            const int32_t* lte, const int32_t* uts, const int32_t* ute, uint8_t* tile_class,
                            int32_t* q_off, int32_t* q_queue, int32_t* k_off, int32_t* k_queue, void* ws,
                            cudaStream_t s, int* err) {
  const int B = p.B, N = p.N, Nk = kv_rows(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  Minmax* mm = reinterpret_cast<Minmax*>(w);
  w += align256(sizeof(Minmax) * (size_t)B * nK);
  int32_t* row_cnt = reinterpret_cast<int32_t*>(w);
  w += align256(4 * (size_t)B * nQ);
  int32_t* col_cnt = reinterpret_cast<int32_t*>(w);

  const long long nkb = (long long)B * nK, nqb = (long long)B * nQ;
  block_minmax_kernel<<<(unsigned)((nkb + 7) / 8), 256, 0, s>>>(lts, lte, uts, ute, B, N, Nk, bn, nK, mm, col_cnt,
                                                                err);
  classify_rows_kernel<<<dim3(nQ, B), 256, 0, s>>>(mm, N, Nk, bm, bn, nQ, nK, p.causal, tile_class, row_cnt,
                                                   col_cnt);
  scan_kernel<<<2, 1024, 0, s>>>(row_cnt, (int)nqb, q_off, col_cnt, (int)nkb, k_off);
  emit_queues_kernel<<<(unsigned)((nqb + nkb + 7) / 8), 256, 0, s>>>(tile_class, B, nQ, nK, q_off, q_queue, k_off,
                                                                     k_queue);
  count_launches(4);
  return cudaGetLastError();
}

}  // namespace fm
