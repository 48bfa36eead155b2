// fm_fwd256.cu — masked attention forward for head dimension 256 on sm_103a.
//
// Same computation as fm_fwd.cu (FlashMask-3 project page, §3.1: only queued
// KV blocks are loaded and the row-interval mask is applied only on partial
// blocks; the online softmax of "Flash MSA Attention Kernel Implementation",
// "The Flash Core: Tiling Over the Memory Hierarchy"), for d = 256, the head
// size of the FlashMask Guide's usage example ("Complete PyTorch
// Implementation", dim = 256).
//
// At d = 256 a 128-row bf16 tile is 64 KB and one head's O accumulator takes
// 256 of TMEM's 512 columns, so the two-head unit of the d <= 128 kernel does
// not fit. Here a CTA computes one (batch, Q block, query head) unit:
//   shared memory  Q (64 KB), one K slot (64 KB), one V slot (64 KB), two
//                  mask-vector slots, one 2 KB O staging slot per softmax warp;
//   TMEM           S_0 [0, 128), S_1 [128, 256), O [256, 512): S is double
//                  buffered so S(j+1) runs on the tensor core while the
//                  softmax works on S(j); P(j) is written back as bf16 over
//                  the first 64 columns of its S buffer and read from TMEM by
//                  the PV MMA.
// Roles (256 threads):
//   warps 0-3  softmax, one thread per query row (running max m, sum l,
//              lazy rescale of O by more than 8 in log2 units, as in
//              fm_fwd.cu), then the epilogue O / l through the staging slot
//              and TMA stores, and LSE;
//   warp 4     K producer: Q once, then K of each queued block, and the mask
//              vectors of partial blocks;
//   warp 5     S issuer: S(j) = Q K(j)^T into S_(j&1) once K(j) has landed
//              and PV(j-2) (the last reader of that buffer) has completed;
//              owns the TMEM allocation;
//   warp 6     PV issuer: O += P(j) V(j) once the softmax has written P(j);
//   warp 7     V producer: V of each queued block.
// Two producers and two issuers let K(j+1) load and S(j+1) run while V(j)
// waits for PV(j-1): one thread blocked on one chain would stall the other.
// With one K and one V slot, a tile could only load once the MMA reading the
// previous one had finished, and a 64 KB load takes longer than that MMA. So
// the slots are refilled in quarters with their own barriers: K by its four
// 64-column boxes (S(j)'s k-steps over box x free it), V by 32-key quarters
// (PV(j)'s two k-steps over those keys free it); the next block's quarter
// loads while the rest of the current MMA runs.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cuda.h>
#include "fm_internal.h"
#include "mask_bits.cuh"
#include "sm100.cuh"
#include "lpt_order.cuh"

namespace fm {
namespace {

constexpr unsigned kFull256 = 0xffffffffu;
constexpr float kLn2f = 0.69314718055994530942f;

struct F256 {
  static constexpr int D = 256;
  static constexpr int TILE = 128 * D * 2;  // 64 KB
  static constexpr int BOXES = D / 64;     // 64-column TMA boxes per tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + TILE;
  // 2 mask slots of {LTS, LTE, UTS, UTE}[128] int32 (multi-interval masks:
  // {FMS, FME}[128] of up to four intervals)
  static constexpr int M_OFF = V_OFF + TILE;
  static constexpr int M_BYTES = 4 * 2 * 128 * 4;
  static constexpr int O_OFF = M_OFF + 2 * M_BYTES;  // 4 warps x 2 KB
  static constexpr int O_SLOT = 32 * 32 * 2;
  static constexpr int BAR_OFF = O_OFF + 4 * O_SLOT;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;    // [4] per 64-column box of K
  static constexpr int B_KEMPTY = 5;   // [4]
  static constexpr int B_VFULL = 9;    // [4] per 32-key quarter of V
  static constexpr int B_VEMPTY = 13;  // [4]
  static constexpr int B_MFULL = 17;   // [2]
  static constexpr int B_MEMPTY = 19;  // [2]
  static constexpr int B_SFULL = 21;   // [2]
  static constexpr int B_PREADY = 23;  // [2]
  static constexpr int B_ODONE = 25;   // [2]
  static constexpr int NBAR = 27;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
};
static_assert(F256::SMEM_ALLOC <= 232448, "d = 256 forward exceeds shared memory");

struct Fwd256Params {
  const int32_t* lts;
  const int32_t* lte;
  const int32_t* uts;
  const int32_t* ute;
  const int32_t* q_off;
  const int32_t* q_queue;
  const int32_t* order;  // order of (b, qb) (per-head masks: of queue rows), or null: natural order
  float* lse;
  int B, H_q, H_kv, N, Nk, nQ, nK, G, causal;
  int per_head;  // vectors (B, H_q, N_kv), one queue per (b, h, qb) row
  // multi-interval masks: lts / lte hold FMS / FME, (M, B, N_kv), M >= 1
  // (the MI instantiation); 0 otherwise
  int M;
  float scale_log2;
  int* err;
};

__device__ __forceinline__ bool partial256(const Fwd256Params& p, int e) {
  return (e & 1) || ((e >> 1) == p.nK - 1 && (p.Nk & 127));
}

// MI: multi-interval masks (mask slots hold FMS / FME of every interval).
template <bool MI>
__global__ void __launch_bounds__(256, 1)
    fwd256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  const Fwd256Params p) {
  using C = F256;
  constexpr int D = C::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  FM_DEBUG_BEGIN();
  // unit: (b, qb) from the launch order, query head h (fastest: the heads of
  // one GQA group run side by side and share K / V tiles in L2)
  int b, qb, h, row;  // row: this unit's queue
  if (!p.per_head) {
    const int oi = blockIdx.x / p.H_q;
    h = blockIdx.x - oi * p.H_q;
    row = p.order ? p.order[oi] : oi;
    b = row / p.nQ;
    qb = row - b * p.nQ;
  } else {
    // queue rows (b * H_q + h) * nQ + qb, from the order table or with the
    // heads of one (b, qb) side by side
    if (p.order) {
      row = p.order[blockIdx.x];
    } else {
      const int oi = blockIdx.x / p.H_q, hh = blockIdx.x - oi * p.H_q;
      const int bb = oi / p.nQ;
      row = (bb * p.H_q + hh) * p.nQ + (oi - bb * p.nQ);
    }
    const int bhr = row / p.nQ;
    qb = row - bhr * p.nQ;
    b = bhr / p.H_q;
    h = bhr - b * p.H_q;
  }
  const int g = h / p.G;
  const int qbeg = p.q_off[row];
  const int n = p.q_off[row + 1] - qbeg;
  const int bh = b * p.H_q + h;
  const size_t vbase = (size_t)(p.per_head ? bh : b) * p.Nk;

  if (threadIdx.x == 0) {
    *abort_flag = timeout_pending(p.err) ? 1 : 0;
    mbar_init(&bars[C::B_QFULL], 1);
    for (int x = 0; x < 4; ++x) {
      mbar_init(&bars[C::B_KFULL + x], 1);
      mbar_init(&bars[C::B_KEMPTY + x], 1);
      mbar_init(&bars[C::B_VFULL + x], 1);
      mbar_init(&bars[C::B_VEMPTY + x], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[C::B_MFULL + s], 1);
      mbar_init(&bars[C::B_MEMPTY + s], 4);
      mbar_init(&bars[C::B_SFULL + s], 1);
      mbar_init(&bars[C::B_PREADY + s], 128);
      mbar_init(&bars[C::B_ODONE + s], 1);
    }
    fence_mbar_init();
  }
  if constexpr (MI) {
    // the interval places past M of both mask slots hold an empty interval
    // (FMS 1, FME 0) for the whole launch: the producer never writes them, and
    // the softmax warps read two or four intervals without a per-interval test
    int* mv = reinterpret_cast<int*>(smem + C::M_OFF);
    for (int i = threadIdx.x; i < 2 * 1024; i += blockDim.x)
      if (((i & 1023) >> 8) >= p.M) mv[i] = (i & 255) < 128 ? 1 : 0;
  }
  if (warp == 5) tmem_alloc<512>(tmem_slot);
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
  }
  if (warp == 7 && lane == 0) tma_prefetch_desc(&tv);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (*abort_flag) {
    // an unread timeout from an earlier launch: skip the work
  } else if (n < 0) {
    if (threadIdx.x == 0) record_error(p.err, FM_DEV_ERR_QUEUE);
  } else if (warp == 4) {
    // ---------------------------------------------------------- K producer
    bool ok = true;
    uint32_t pidx = 0;
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(&bars[C::B_QFULL], C::TILE);
      for (int x = 0; x < C::BOXES; ++x)
        tma_load_3d(smem + C::Q_OFF + x * 16384, &tq, &bars[C::B_QFULL], x * 64, qb * 128, bh);
    }
    for (int j = 0; j < n && ok; ++j) {
      const int e = p.q_queue[qbeg + j];
      const int kb = e >> 1;
      if (kb < 0 || kb >= p.nK) {
        if (lane == 0) record_error(p.err, FM_DEV_ERR_QUEUE);
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        // box by box, each as soon as S(j-1) has read that box
        for (int x = 0; x < C::BOXES && ok; ++x) {
          ok = mbar_wait(&bars[C::B_KEMPTY + x], ((uint32_t)j & 1u) ^ 1u, abort_flag, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&bars[C::B_KFULL + x], 16384);
            tma_load_3d(smem + C::K_OFF + x * 16384, &tk, &bars[C::B_KFULL + x], x * 64, kb * 128, b * p.H_kv + g);
          }
        }
      }
      ok = __shfl_sync(kFull256, ok, 0);
      if (!ok || !partial256(p, e)) continue;
      // the block's four mask vectors, raw (LTS, LTE, UTS, UTE x 128; with
      // multi-interval masks FMS, FME x 128 of every interval, a key beyond
      // Nk an empty interval); the softmax warps clamp them to their 32-row
      // windows
      const int ms = pidx & 1;
      ok = __all_sync(kFull256, mbar_wait(&bars[C::B_MEMPTY + ms], ((pidx >> 1) & 1u) ^ 1u, abort_flag, p.err));
      if (!ok) break;
      uint8_t* sm = smem + C::M_OFF + ms * C::M_BYTES;
      const int c0 = kb * 128;
      if constexpr (MI) {
        bool al = c0 + 128 <= p.Nk;
        for (int mi = 0; mi < p.M; ++mi) {
          const size_t o = ((size_t)mi * p.B + b) * p.Nk + c0;
          al = al && ((reinterpret_cast<uintptr_t>(p.lts + o) | reinterpret_cast<uintptr_t>(p.lte + o)) & 15u) == 0;
        }
        if (al) {
          if (lane == 0) {
            uint64_t* fb = &bars[C::B_MFULL + ms];
            mbar_arrive_expect_tx(fb, 2 * 512 * p.M);
            for (int mi = 0; mi < p.M; ++mi) {
              const size_t o = ((size_t)mi * p.B + b) * p.Nk + c0;
              bulk_load(sm + mi * 1024, p.lts + o, 512, fb);
              bulk_load(sm + mi * 1024 + 512, p.lte + o, 512, fb);
            }
          }
        } else {
          int* vv = reinterpret_cast<int*>(sm);
          for (int mi = 0; mi < p.M; ++mi) {
            const size_t o = ((size_t)mi * p.B + b) * p.Nk;
            for (int c = lane; c < 128; c += 32) {
              const int col = c0 + c;
              const bool in = col < p.Nk;
              vv[mi * 256 + c] = in ? p.lts[o + col] : 1;
              vv[mi * 256 + 128 + c] = in ? p.lte[o + col] : 0;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[C::B_MFULL + ms]);
        }
        ++pidx;
        continue;
      }
      const size_t vb = vbase;
      const size_t o = vb + c0;
      const bool aligned = ((reinterpret_cast<uintptr_t>(p.lts + o) | reinterpret_cast<uintptr_t>(p.lte + o) |
                             reinterpret_cast<uintptr_t>(p.uts + o) | reinterpret_cast<uintptr_t>(p.ute + o)) &
                            15u) == 0;
      if (c0 + 128 <= p.Nk && aligned) {
        if (lane == 0) {
          uint64_t* fb = &bars[C::B_MFULL + ms];
          mbar_arrive_expect_tx(fb, 4 * 512);
          bulk_load(sm + 0, p.lts + o, 512, fb);
          bulk_load(sm + 512, p.lte + o, 512, fb);
          bulk_load(sm + 1024, p.uts + o, 512, fb);
          bulk_load(sm + 1536, p.ute + o, 512, fb);
        }
      } else {
        int* vv = reinterpret_cast<int*>(sm);
        for (int c = lane; c < 128; c += 32) {
          const int col = c0 + c;
          const bool in = col < p.Nk;  // a key beyond Nk is masked for every row
          vv[c] = in ? p.lts[vb + col] : 0;
          vv[128 + c] = in ? p.lte[vb + col] : p.N;
          vv[256 + c] = in ? p.uts[vb + col] : 0;
          vv[384 + c] = in ? p.ute[vb + col] : 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_MFULL + ms]);
      }
      ++pidx;
    }
  } else if (warp == 7) {
    // ---------------------------------------------------------- V producer
    if (lane == 0) {
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int kb = p.q_queue[qbeg + j] >> 1;
        if (kb < 0 || kb >= p.nK) break;  // flagged by the K producer
        // 32 keys at a time (all four 64-column boxes), each quarter as soon
        // as PV(j-1) has read it
        for (int qq = 0; qq < 4 && ok; ++qq) {
          ok = mbar_wait(&bars[C::B_VEMPTY + qq], ((uint32_t)j & 1u) ^ 1u, abort_flag, p.err);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars[C::B_VFULL + qq], 4 * 4096);
          for (int x = 0; x < C::BOXES; ++x)
            tma_load_3d(smem + C::V_OFF + x * 16384 + qq * 4096, &tv, &bars[C::B_VFULL + qq], x * 64,
                        kb * 128 + 32 * qq, b * p.H_kv + g);
        }
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- S issuer
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 128, 0, 0);  // S = Q K^T, both K-major
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::K_OFF), 16, 1024);
      bool ok = mbar_wait(&bars[C::B_QFULL], 0, abort_flag, p.err);
      for (int j = 0; j < n && ok; ++j) {
        // S_(j&1) last held P(j-2): PV(j-2) must have read it
        if (j >= 2) ok = mbar_wait(&bars[C::B_ODONE + (j & 1)], ((uint32_t)(j - 2) >> 1) & 1u, abort_flag, p.err);
        const uint32_t tS = tbase + 128u * (uint32_t)(j & 1);
        // four k-steps per 64-column box of K, each box released once read
        for (int x = 0; x < C::BOXES && ok; ++x) {
          ok = mbar_wait(&bars[C::B_KFULL + x], (uint32_t)j & 1u, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * x + k4;
            const uint64_t off = (uint64_t)(x * 1024 + k4 * 2);
            mma_ss(tS, dQ0 + off, dK0 + off, id_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars[C::B_KEMPTY + x]);
        }
        if (ok) mma_commit(&bars[C::B_SFULL + (j & 1)]);
      }
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------- PV issuer
    if (lane == 0 && n > 0) {
      const uint32_t id_o = idesc_bf16_f32(128, D, 0, 1);  // O += P V, V is MN-major
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::V_OFF), 16384, 1024);
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        ok = mbar_wait(&bars[C::B_PREADY + (j & 1)], ((uint32_t)j >> 1) & 1u, abort_flag, p.err);
        const uint32_t tS = tbase + 128u * (uint32_t)(j & 1);
        // two k-steps (16 keys each) per 32-key quarter of V, each quarter
        // released once read
        for (int qq = 0; qq < 4 && ok; ++qq) {
          ok = mbar_wait(&bars[C::B_VFULL + qq], (uint32_t)j & 1u, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int kk = 2 * qq + k2;
            mma_ts(tbase + 256u, tS + (uint32_t)(kk * 8), dV0 + (uint64_t)(kk * 128), id_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars[C::B_VEMPTY + qq]);
        }
        if (ok) mma_commit(&bars[C::B_ODONE + (j & 1)]);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int row = (warp << 5) + lane;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int q0 = qb * 128, i = q0 + row, w0 = q0 + (warp << 5);
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const uint32_t tO = tbase + lane_off + 256u;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t pidx = 0;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int e = p.q_queue[qbeg + j];
      const int kb = e >> 1;
      const bool part = partial256(p, e);
      // partial block: masked-row bits of this thread's row over the 128 key
      // columns (lane c builds column 32k + c over the warp's 32 rows, then a
      // bit transpose hands each lane its own row)
      uint32_t rb[4] = {0u, 0u, 0u, 0u};
      if (part) {
        const int ms = pidx & 1;
        ok = __all_sync(kFull256, mbar_wait(&bars[C::B_MFULL + ms], (pidx >> 1) & 1u, abort_flag, p.err));
        if (!ok) break;
        const uint32_t sm = smem_u32(smem + C::M_OFF + ms * C::M_BYTES);
        const int kc0 = kb * 128;
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int c = 32 * kq + lane;
          uint32_t colbits;
          if constexpr (MI) {
            // masked unless one interval [FMS, FME] holds the row (the places
            // past M hold empty intervals)
            auto iv = [&](int mi) -> uint32_t {
              const int f0 = lds_s32(sm + mi * 1024 + 4 * c), f1 = lds_s32(sm + mi * 1024 + 512 + 4 * c);
              return window_bits(f0, min(f1, p.N) + 1, w0);
            };
            const uint32_t vis = (p.M <= 2) ? (iv(0) | iv(1)) : (iv(0) | iv(1) | iv(2) | iv(3));
            colbits = ~vis | (causal ? window_bits(w0, kc0 + c, w0) : 0u);
          } else {
            const int a0 = lds_s32(sm + 4 * c), a1 = lds_s32(sm + 512 + 4 * c);
            const int u0 = lds_s32(sm + 1024 + 4 * c), u1 = lds_s32(sm + 1536 + 4 * c);
            colbits = window_bits(a0, a1, w0) | window_bits(u0, u1, w0) | (causal ? window_bits(w0, kc0 + c, w0) : 0u);
          }
          rb[kq] = warp_transpose32(colbits, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_MEMPTY + ms]);
        ++pidx;
      }
      ok = __all_sync(kFull256, mbar_wait(&bars[C::B_SFULL + (j & 1)], ((uint32_t)j >> 1) & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tbase + lane_off + 128u * (uint32_t)(j & 1);
      uint32_t sr[128];
      {
        uint32_t(&r0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
        uint32_t(&r1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
        uint32_t(&r2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
        uint32_t(&r3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
        tmem_ld32(tS + 0, r0);
        tmem_ld32(tS + 32, r1);
        tmem_ld32(tS + 64, r2);
        tmem_ld32(tS + 96, r3);
        tmem_ld_wait();
      }
      if (part) {
#pragma unroll
        for (int c = 0; c < 128; ++c) sr[c] = ((rb[c >> 5] >> (c & 31)) & 1u) ? __float_as_uint(-INFINITY) : sr[c];
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 8) {
        mx0 = max3f(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        mx1 = max3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
        mx2 = max3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
        mx3 = max3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
      }
      const float m_blk = max3f(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
      const float m_new = fmaxf(m_run, m_blk);
      const bool resc = m_new > m_run + 8.0f;
      float factor = 1.f;
      if (resc) {
        factor = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      const float msafe = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-msafe, -msafe);
      uint64_t rs0 = f2_pack(0.f, 0.f), rs1 = rs0;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2x2, nm2), x0, x1);
        const float a = ex2_approx(x0), bb = ex2_approx(x1);
        if (c & 1) rs1 = f2_add(rs1, f2_pack(a, bb));
        else rs0 = f2_add(rs0, f2_pack(a, bb));
        pk[c] = pack_bf16x2(a, bb);
      }
      float r0a, r0b, r1a, r1b;
      f2_unpack(rs0, r0a, r0b);
      f2_unpack(rs1, r1a, r1b);
      l_run = l_run * factor + ((r0a + r0b) + (r1a + r1b));
      {
        const uint32_t(&p0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]);
        const uint32_t(&p1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]);
        const uint32_t(&p2)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[32]);
        const uint32_t(&p3)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[48]);
        tmem_st16(tS + 0, p0);
        tmem_st16(tS + 16, p1);
        tmem_st16(tS + 32, p2);
        tmem_st16(tS + 48, p3);
        tmem_st_wait();
      }
      if (j > 0 && __any_sync(kFull256, resc)) {
        // O holds PV of the earlier blocks: wait for the last of them, rescale
        ok = __all_sync(kFull256, mbar_wait(&bars[C::B_ODONE + ((j - 1) & 1)], ((uint32_t)(j - 1) >> 1) & 1u,
                                            abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * factor);
          tmem_st32(tO + c0, r);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars[C::B_PREADY + (j & 1)]);
    }
    // epilogue: O / l, 32 columns at a time, through this warp's staging slot
    // (64-byte swizzle: row r's 16-byte chunk c at chunk c ^ ((r >> 1) & 3))
    // to TMA stores of the warp's 32 rows (rows past N are clipped); a unit
    // with an empty queue stores zeros and LSE = -inf
    if (ok && n > 0) {
      ok = __all_sync(kFull256, mbar_wait(&bars[C::B_ODONE + ((n - 1) & 1)], ((uint32_t)(n - 1) >> 1) & 1u,
                                          abort_flag, p.err));
      tc_fence_after();
    }
    if (ok) {
      const uint32_t oslot = smem_u32(smem + C::O_OFF + warp * C::O_SLOT);
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t w[16];
        if (n > 0) {
          uint32_t r[32];
          tmem_ld32(tO + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            w[c] = pack_bf16x2(__uint_as_float(r[2 * c]) * inv, __uint_as_float(r[2 * c + 1]) * inv);
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) w[c] = 0u;
        }
        if (lane == 0) bulk_wait_group_read0();  // the slot's previous store has read it
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          sts_b32x4(oslot + 64 * lane + 16 * (c ^ ((lane >> 1) & 3)), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                    w[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&to, oslot, c0, w0, bh);
          bulk_commit_group();
        }
      }
      if (i < p.N) p.lse[(size_t)bh * p.N + i] = (l_run > 0.f) ? (m_run * kLn2f + logf(l_run)) : -INFINITY;
    }
  }

  // the staging slots stay valid until the TMA stores have read them
  if (warp < 4 && lane == 0) bulk_wait_group_read0();
  tc_fence_before();
  __syncthreads();
  FM_DEBUG_END(p.err);
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tbase);
  }
}

}  // namespace

// d = 256: one CTA per (batch, Q block, query head); the workspace is the
// forward's (unit-order table, then a counter this kernel does not use).
// per_head: vectors (B, H_q, N_kv) and queues over B * H_q * nQ rows.
cudaError_t launch_fwd256(const fm_problem& P, const void* q, const void* k, const void* v, const int32_t* lts,
                          const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                          const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err,
                          bool per_head, int M) {
  using C = F256;
  const int nQ = (P.N + kTile - 1) / kTile;
  const int Nk = kv_rows(P);
  const long long grid = (long long)P.B * nQ * P.H_q;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  // longest queue first for passes of a few waves, natural order for long ones
  const bool natural = use_natural_order(grid);
  int32_t* order = natural ? nullptr : static_cast<int32_t*>(ws);
  if (!natural) lpt_order_kernel<<<1, 1024, 0, s>>>(q_off, per_head ? P.B * P.H_q * nQ : P.B * nQ, order);
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bhnd(&tq, q, (int64_t)P.B * P.H_q, P.N, P.d) || !make_tmap_bhnd(&tk, k, (int64_t)P.B * P.H_kv, Nk, P.d) ||
      !make_tmap_bhnd(&tv, v, (int64_t)P.B * P.H_kv, Nk, P.d, 32) ||
      !make_tmap_bhnd_w32(&to, o, (int64_t)P.B * P.H_q, P.N, P.d))
    return cudaErrorInvalidValue;
  Fwd256Params prm;
  prm.lts = lts;
  prm.lte = lte;
  prm.uts = uts;
  prm.ute = ute;
  prm.q_off = q_off;
  prm.q_queue = q_queue;
  prm.order = order;
  prm.lse = lse;
  prm.B = P.B;
  prm.H_q = P.H_q;
  prm.H_kv = P.H_kv;
  prm.N = P.N;
  prm.Nk = Nk;
  prm.nQ = nQ;
  prm.nK = (Nk + kTile - 1) / kTile;
  prm.G = P.H_q / P.H_kv;
  prm.causal = P.causal ? 1 : 0;
  prm.per_head = per_head ? 1 : 0;
  prm.M = M;
  prm.scale_log2 = P.scale * 1.4426950408889634f;
  prm.err = err;
  static bool attr_done[2] = {false, false};
  const bool mi = M > 0;
  if (!attr_done[mi]) {
    cudaError_t e = cudaFuncSetAttribute(mi ? fwd256_kernel<true> : fwd256_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_done[mi] = true;
  }
  {
    KernelTimer timer(s, kTimedFwd);
    if (mi)
      fwd256_kernel<true><<<(unsigned)grid, 256, C::SMEM_ALLOC, s>>>(tq, tk, tv, to, prm);
    else
      fwd256_kernel<false><<<(unsigned)grid, 256, C::SMEM_ALLOC, s>>>(tq, tk, tv, to, prm);
  }
  count_launches(natural ? 1 : 2);  // [LPT order] + main kernel
  return cudaGetLastError();
}

}  // namespace fm
