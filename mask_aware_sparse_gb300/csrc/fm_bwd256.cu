// fm_bwd256.cu — masked attention backward main kernel for head dimension 256
// on sm_103a (tcgen05 + TMEM + TMA).
//
// Same computation as fm_bwd.cu ("Flash MSA Attention Kernel Implementation",
// "The Backward Pass: The Real Beast"; the mask and tile skipping of
// FlashMask-3 project page §3.1): P = exp(scale S - LSE), dV = P^T dO,
// dP = dO V^T, dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q, over the
// tiles of each KV block's queue, masking only partial tiles, with dK and dV
// summed over the query heads of each GQA group.
//
// At d = 256 the dK and dV accumulators of a 128-row KV block would fill all
// 512 TMEM columns, so each KV block is handled by two CTAs, one per half of
// the head dimension (dh = 0, 1): both recompute S^T = K Q^T and dP^T = V dO^T
// over the whole head dimension, and each accumulates its own 128 columns of
// dV, dK and dQ. TMEM per CTA: S^T [0, 64), dP^T [128, 192), dQ^T [192, 256),
// dV [256, 384), dK [384, 512).
// Shared memory: K and V of the block (64 KB each, for the full-width S^T and
// dP^T), one stage of Q and dO (32 KB each: 64 query rows), one dS^T buffer
// (16 KB), the dQ drain's transpose slots (16 KB). The stages cannot be
// doubled, so each Q / dO tile is handled as two head-dim halves with their
// own barriers: the other CTA's half (columns this CTA does not output) feeds
// only S^T and dP^T, and is released as soon as those k-steps are done; this
// CTA's own half also feeds dK and dV and is released after dK. The MMA lane
// issues the next unit's other-half k-steps of S^T and dP^T at the end of the
// current unit, so both halves of the next unit load under the current
// unit's MMAs.
//
// Roles (448 threads):
//   warps 0-7  compute: thread j of warp w owns KV row j = 32*(w%4) + lane and
//              query columns [32*(w/4), +32) of the unit: P^T (bf16, back to
//              TMEM over S^T) and dS^T (bf16, to shared memory);
//   warps 8-11 dQ drain: TMEM lane c = head-dim index 128*dh + c of dQ^T, to
//              the fp32 accumulator by TMA reduce-adds of 32 x 32 boxes; at
//              the end the dK half;
//   warp 12    TMA producer (K, V once; per unit the other halves of Q and
//              dO with the row terms (two slots), then the own halves);
//   warp 13    MMA issuer and TMEM owner: per unit u the own-half k-steps of
//              S^T(u) and dP^T(u), dV(u) after P^T(u), dK(u) and dQ^T(u) after
//              dS^T(u), then the other-half k-steps of S^T(u+1) and dP^T(u+1).
#include <climits>
#include <cmath>
#include <cuda.h>
#include "fm_internal.h"
#include "mask_bits.cuh"
#include "sm100.cuh"

namespace fm {
namespace {

constexpr unsigned kFullB = 0xffffffffu;

struct B256 {
  static constexpr int D = 256;
  static constexpr int DH = 128;                 // output columns per CTA
  static constexpr int KV_TILE = 128 * D * 2;    // 64 KB
  static constexpr int Q_TILE = 64 * D * 2;      // 32 KB
  static constexpr int K_OFF = 0;                // 4 boxes of 128 rows x 64 columns (16 KB)
  static constexpr int V_OFF = K_OFF + KV_TILE;
  static constexpr int Q_OFF = V_OFF + KV_TILE;  // 4 boxes of 64 rows x 64 columns (8 KB)
  static constexpr int DO_OFF = Q_OFF + Q_TILE;
  static constexpr int DS_OFF = DO_OFF + Q_TILE;  // 128 KV rows x 64 query columns bf16
  static constexpr int XPOSE_OFF = DS_OFF + 16384;  // 4 drain warps x 32 x 32 fp32
  static constexpr int ROW_OFF = XPOSE_OFF + 4 * 4096;  // two slots of {nl[64], D[64]} fp32
  static constexpr int QUEUE_CAP = 128;
  static constexpr int QUEUE_OFF = ROW_OFF + 2 * 512;
  // per-head masks: each group head's first entry in the heads' queues back
  // to back (a prefix, 65 entries)
  static constexpr int HEADS_OFF = QUEUE_OFF + QUEUE_CAP * 4;
  static constexpr int BAR_OFF = HEADS_OFF + 272;
  static constexpr int B_KV = 0;
  static constexpr int B_OFULL = 1;   // [2] other halves of Q, dO + row terms of unit u, by u & 1
  static constexpr int B_OEMPTY = 3;  // other halves free (S^T(u), dP^T(u) done)
  static constexpr int B_MFULL = 4;   // own halves of Q, dO
  static constexpr int B_MEMPTY = 5;  // own halves free (dV(u), dK(u) done)
  static constexpr int B_SFULL = 6;
  static constexpr int B_PREADY = 7;
  static constexpr int B_DPFULL = 8;
  static constexpr int B_READY = 9;
  static constexpr int B_DQFULL = 10;
  static constexpr int B_DQEMPTY = 11;
  static constexpr int B_FINAL = 12;
  static constexpr int B_VSTAGED = 13;
  static constexpr int B_KSTAGED = 14;
  static constexpr int NBAR = 15;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = BYTES + 1024;
};
static_assert(B256::SMEM_ALLOC <= 232448, "d = 256 backward exceeds shared memory");

struct Bwd256Params {
  const int32_t* lts;
  const int32_t* lte;
  const int32_t* uts;
  const int32_t* ute;
  const int32_t* k_off;
  const int32_t* k_queue;
  const int32_t* order;  // launch order of (b, kb), or null: natural order (always with per-head masks)
  const float* nl;       // (B*H_q, Npad): -LSE*log2(e), -inf for empty / padded rows
  const float* dsum;     // (B*H_q, Npad): D = rowsum(dO * O)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int B, H_q, H_kv, N, Nk, Npad, nK, G, causal;
  int M;  // multi-interval masks: FMS / FME (M, B, N_kv) (1 otherwise)
  float scale, scale_log2;
  int* err;
};

// Query heads per GQA group with per-head mask vectors (the staged prefix).
constexpr int kMaxHeads256 = 64;

struct Unit256 {
  int h, qb, half, part;
};
__device__ __forceinline__ Unit256 decode256(const Bwd256Params& p, int u, int L, int kbeg, int g, bool force_part,
                                             uint32_t s_queue) {
  Unit256 r;
  const int hi = u / (2 * L);
  const int rem = u - hi * 2 * L;
  const int pos = rem >> 1;
  const int e = (pos < B256::QUEUE_CAP) ? lds_s32(s_queue + 4 * pos) : p.k_queue[kbeg + pos];
  r.h = g * p.G + hi;
  r.qb = e >> 1;
  r.half = rem & 1;
  r.part = (e & 1) | (force_part ? 1 : 0);
  return r;
}
// The same with per-head mask vectors: head hi of the group owns the units
// [2 hoff[hi], 2 hoff[hi + 1]) (its own queue for this KV block); the staged
// entries are the heads' queues back to back. hi is the caller's cursor (units
// are visited in increasing order).
__device__ __forceinline__ Unit256 decode256_ph(const Bwd256Params& p, int u, int b, int kb, int g,
                                                bool force_part, uint32_t s_queue, const int* hoff, int& hi) {
  while (u >= 2 * hoff[hi + 1]) ++hi;
  const int rem = u - 2 * hoff[hi];
  const int pos = hoff[hi] + (rem >> 1);
  Unit256 r;
  r.h = g * p.G + hi;
  const int e = (pos < B256::QUEUE_CAP)
                    ? lds_s32(s_queue + 4 * pos)
                    : p.k_queue[p.k_off[((size_t)b * p.H_q + r.h) * p.nK + kb] + (rem >> 1)];
  r.qb = e >> 1;
  r.half = rem & 1;
  r.part = (e & 1) | (force_part ? 1 : 0);
  return r;
}
// MODE 0: mask vectors (B, N_kv) shared by the heads; 1: per-head vectors
// (B, H_q, N_kv) and queues over B * H_q rows; 2: multi-interval masks (lts /
// lte hold FMS / FME, (M, B, N_kv); the union classification's queues).
template <int MODE>
__global__ void __launch_bounds__(448, 1)
    bwd256_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                  const __grid_constant__ CUtensorMap tdq, const Bwd256Params p) {
  using C = B256;
  constexpr int DH = C::DH;
  constexpr bool PH = MODE == 1, MI = MODE == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  FM_DEBUG_BEGIN();
  // CTA = (launch-order position, kv head, head-dim half); the two halves of
  // one KV block are neighbours and share every tile in L2
  const int dh = blockIdx.x & 1;
  const int og = blockIdx.x >> 1;
  const int oi = og / p.H_kv, g = og - oi * p.H_kv;
  const int bk = p.order ? p.order[oi] : oi;
  const int nK = p.nK;
  const int b = bk / nK, kb = bk - b * nK;
  int kbeg = 0, L = 0;  // per-head masks: L sums the heads' queue lengths
  if constexpr (PH) {
    for (int hi = 0; hi < p.G; ++hi) {
      const int r = (b * p.H_q + g * p.G + hi) * nK + kb;
      L += p.k_off[r + 1] - p.k_off[r];
    }
  } else {
    kbeg = p.k_off[bk];
    L = p.k_off[bk + 1] - kbeg;
  }
  const int U = PH ? 2 * L : 2 * L * p.G;
  const int k0 = kb * 128;
  const int c0h = dh * DH;  // first head-dim column of this CTA's outputs
  const bool force_part = (kb == nK - 1) && (p.Nk & 127);

  if (U <= 0) {
    // No query row sees this KV block: this half of dK and dV is 0.
    if (L < 0 && threadIdx.x == 0) record_error(p.err, FM_DEV_ERR_QUEUE);
    if (warp < 4) {
      const int j = k0 + (warp << 5) + lane;
      if (j < p.Nk) {
        const size_t row = ((size_t)b * p.H_kv + g) * p.Nk + j;
        uint4* a = reinterpret_cast<uint4*>(p.dk + row * C::D + c0h);
        uint4* c = reinterpret_cast<uint4*>(p.dv + row * C::D + c0h);
#pragma unroll
        for (int x = 0; x < DH / 8; ++x) a[x] = c[x] = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    *abort_flag = timeout_pending(p.err) ? 1 : 0;
    mbar_init(&bars[C::B_KV], 1);
    mbar_init(&bars[C::B_OFULL], 1);
    mbar_init(&bars[C::B_OFULL + 1], 1);
    mbar_init(&bars[C::B_OEMPTY], 1);
    mbar_init(&bars[C::B_MFULL], 1);
    mbar_init(&bars[C::B_MEMPTY], 1);
    mbar_init(&bars[C::B_SFULL], 1);
    mbar_init(&bars[C::B_PREADY], 256);
    mbar_init(&bars[C::B_DPFULL], 1);
    mbar_init(&bars[C::B_READY], 256);
    mbar_init(&bars[C::B_DQFULL], 1);
    mbar_init(&bars[C::B_DQEMPTY], 128);
    mbar_init(&bars[C::B_FINAL], 1);
    mbar_init(&bars[C::B_VSTAGED], 128);
    mbar_init(&bars[C::B_KSTAGED], 128);
    fence_mbar_init();
  }
  const uint32_t s_queue = smem_u32(smem + C::QUEUE_OFF);
  int* hoff = reinterpret_cast<int*>(smem + C::HEADS_OFF);
  {
    int* sq = reinterpret_cast<int*>(smem + C::QUEUE_OFF);
    if constexpr (PH) {
      if (threadIdx.x == 0) {
        int acc = 0;
        for (int hi = 0; hi < p.G; ++hi) {
          const int r = (b * p.H_q + g * p.G + hi) * nK + kb;
          hoff[hi] = acc;
          acc += p.k_off[r + 1] - p.k_off[r];
        }
        hoff[p.G] = acc;
      }
      __syncthreads();
      for (int t = threadIdx.x; t < L && t < C::QUEUE_CAP; t += blockDim.x) {
        int hi = 0;
        while (hi + 1 < p.G && hoff[hi + 1] <= t) ++hi;
        sq[t] = p.k_queue[p.k_off[(b * p.H_q + g * p.G + hi) * nK + kb] + (t - hoff[hi])];
      }
    } else {
      for (int t = threadIdx.x; t < L && t < C::QUEUE_CAP; t += blockDim.x) sq[t] = p.k_queue[kbeg + t];
    }
  }
  // the unit decoder of every role (a cursor over the heads with per-head masks)
  auto decode = [&](int u, int& hcur) -> Unit256 {
    if constexpr (PH) return decode256_ph(p, u, b, kb, g, force_part, s_queue, hoff, hcur);
    else return decode256(p, u, L, kbeg, g, force_part, s_queue);
  };
  if (warp == 13) tmem_alloc<512>(tmem_slot);
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t T_S = 0, T_DP = 128, T_DQ = 192, T_DV = 256, T_DK = 384;

  if (*abort_flag) {
    // an unread timeout from an earlier launch: skip the work
  } else if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(&bars[C::B_KV], 2 * C::KV_TILE);
      for (int x = 0; x < 4; ++x) {
        tma_load_3d(smem + C::K_OFF + x * 16384, &tk, &bars[C::B_KV], x * 64, k0, b * p.H_kv + g);
        tma_load_3d(smem + C::V_OFF + x * 16384, &tv, &bars[C::B_KV], x * 64, k0, b * p.H_kv + g);
      }
      // Q / dO boxes (64 columns each) of the other CTA's half, then of this one's
      const int xo = 2 * (1 - dh), xm = 2 * dh;
      int hcur = 0;  // head cursor (per-head masks)
      for (int u = 0; u < U && ok; ++u) {
        const Unit256 un = decode(u, hcur);
        const uint32_t pe = ((uint32_t)u & 1u) ^ 1u;
        const int r0 = un.qb * 128 + un.half * 64;
        const int bh = b * p.H_q + un.h;
        ok = mbar_wait(&bars[C::B_OEMPTY], pe, abort_flag, p.err);
        if (!ok) break;
        uint64_t* fo = &bars[C::B_OFULL + (u & 1)];
        uint8_t* rows = smem + C::ROW_OFF + (u & 1) * 512;
        mbar_arrive_expect_tx(fo, C::Q_TILE + 512);
        for (int x = xo; x < xo + 2; ++x) {
          tma_load_3d(smem + C::Q_OFF + x * 8192, &tq, fo, x * 64, r0, bh);
          tma_load_3d(smem + C::DO_OFF + x * 8192, &tdo, fo, x * 64, r0, bh);
        }
        bulk_load(rows, p.nl + (size_t)bh * p.Npad + r0, 256, fo);
        bulk_load(rows + 256, p.dsum + (size_t)bh * p.Npad + r0, 256, fo);
        ok = mbar_wait(&bars[C::B_MEMPTY], pe, abort_flag, p.err);
        if (!ok) break;
        uint64_t* fm_ = &bars[C::B_MFULL];
        mbar_arrive_expect_tx(fm_, C::Q_TILE);
        for (int x = xm; x < xm + 2; ++x) {
          tma_load_3d(smem + C::Q_OFF + x * 8192, &tq, fm_, x * 64, r0, bh);
          tma_load_3d(smem + C::DO_OFF + x * 8192, &tdo, fm_, x * 64, r0, bh);
        }
      }
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);  // S^T, dP^T: A, B K-major
      const uint32_t id_g = idesc_bf16_f32(128, DH, 0, 1);  // dV, dK: B MN-major (this CTA's half)
      const uint32_t id_q = idesc_bf16_f32(128, 64, 1, 1);  // dQ^T: A, B MN-major
      const uint64_t dKk = sdesc_sw128(smem_u32(smem + C::K_OFF), 16, 1024);
      const uint64_t dVk = sdesc_sw128(smem_u32(smem + C::V_OFF), 16, 1024);
      const uint64_t dKt = sdesc_sw128(smem_u32(smem + C::K_OFF + 2 * dh * 16384), 16384, 1024);
      const uint64_t dQk = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t dOk = sdesc_sw128(smem_u32(smem + C::DO_OFF), 16, 1024);
      const uint64_t dQm = sdesc_sw128(smem_u32(smem + C::Q_OFF + 2 * dh * 8192), 8192, 1024);
      const uint64_t dOm = sdesc_sw128(smem_u32(smem + C::DO_OFF + 2 * dh * 8192), 8192, 1024);
      const uint64_t dSk = sdesc_sw128(smem_u32(smem + C::DS_OFF), 16, 1024);
      const uint64_t dSm = sdesc_sw128(smem_u32(smem + C::DS_OFF), 8192, 1024);
      // S^T = K Q^T or dP^T = V dO^T over one head-dim half (8 of the 16
      // k-steps): half hs of the columns; fresh: the first k-step overwrites
      auto issue_sk = [&](uint64_t ad0, uint64_t bd0, uint32_t dst, int hs, bool fresh) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int k = 8 * hs + kk;
          mma_ss(tbase + dst, ad0 + (uint64_t)((k >> 2) * 1024 + (k & 3) * 2),
                 bd0 + (uint64_t)((k >> 2) * 512 + (k & 3) * 2), id_s, (fresh && kk == 0) ? 0u : 1u);
        }
      };
      // the other half's k-steps of S^T(v) and dP^T(v), once its tiles landed
      auto issue_other = [&](int v) -> bool {
        if (!mbar_wait(&bars[C::B_OFULL + (v & 1)], ((uint32_t)v >> 1) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        issue_sk(dKk, dQk, T_S, 1 - dh, true);
        issue_sk(dVk, dOk, T_DP, 1 - dh, true);
        mma_commit(&bars[C::B_OEMPTY]);  // the other halves of Q(v), dO(v)
        return true;
      };
      bool ok = mbar_wait(&bars[C::B_KV], 0, abort_flag, p.err);
      if (ok) ok = issue_other(0);
      for (int u = 0; u < U && ok; ++u) {
        const uint32_t ph = (uint32_t)u & 1u;
        ok = mbar_wait(&bars[C::B_MFULL], ph, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        issue_sk(dKk, dQk, T_S, dh, false);  // S^T(u) over P^T(u-1), read by dV(u-1) issued earlier
        mma_commit(&bars[C::B_SFULL]);
        issue_sk(dVk, dOk, T_DP, dh, false);  // dP^T(u-1) was read before READY(u-1)
        mma_commit(&bars[C::B_DPFULL]);
        // dV += P^T dO (A = P^T from TMEM: two 16-column blocks per compute half)
        ok = mbar_wait(&bars[C::B_PREADY], ph, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a_t = tbase + T_S + (uint32_t)((k >> 1) * 32 + (k & 1) * 8);
          mma_ts(tbase + T_DV, a_t, dOm + (uint64_t)(k * 128), id_g, (u > 0 || k > 0) ? 1u : 0u);
        }
        // dK += dS^T Q and dQ^T = K^T dS^T once dS^T(u) is in shared memory
        ok = mbar_wait(&bars[C::B_READY], ph, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tbase + T_DK, dSk + (uint64_t)(k * 2), dQm + (uint64_t)(k * 128), id_g, (u > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bars[C::B_MEMPTY]);  // the own halves of Q(u), dO(u)
        if (u >= 1) {
          ok = mbar_wait(&bars[C::B_DQEMPTY], ph ^ 1u, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)  // 128 KV rows
          mma_ss(tbase + T_DQ, dKt + (uint64_t)(k * 128), dSm + (uint64_t)(k * 128), id_q, k > 0 ? 1u : 0u);
        mma_commit(&bars[C::B_DQFULL]);
        // S^T(u+1) overwrites P^T(u) after dV(u) (issued above: the MMAs of
        // this lane run in order); dP^T(u+1) after the compute warps read
        // dP^T(u) (READY(u))
        if (u + 1 < U) ok = issue_other(u + 1);
      }
      if (ok) mma_commit(&bars[C::B_FINAL]);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute
    const int j = ((warp & 3) << 5) + lane;  // KV row within the block = TMEM lane
    const int half = warp >> 2;              // query columns [32*half, 32*half + 32)
    const int kcol = k0 + j;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int lo0 = 0, lo1 = 0, up0 = 0, up1 = 0;
    const bool dead = kcol >= p.Nk;
    // this thread's key column's masked intervals, from vector row vrow (the
    // batch entry, or with per-head masks the (batch entry, head))
    auto load_mask = [&](int vrow) {
      lo0 = lo1 = up0 = up1 = 0;
      if (dead) return;
      const size_t vi = (size_t)vrow * p.Nk + kcol;
      int a0 = p.lts[vi], a1 = p.lte[vi], u0 = p.uts[vi], u1 = p.ute[vi];
      if ((a0 | a1 | u0 | u1) < 0 || a0 > p.N || a1 > p.N || u0 > p.N || u1 > p.N) record_error(p.err, FM_DEV_ERR_RANGE);
      a0 = min(max(a0, 0), p.N);
      a1 = min(max(a1, 0), p.N);
      u0 = min(max(u0, 0), p.N);
      u1 = min(max(u1, 0), p.N);
      if (a0 < a1) { lo0 = a0; lo1 = a1; }
      if (u0 < u1) { up0 = u0; up1 = u1; }
    };
    int mhead = -1;  // the head whose vectors are loaded (per-head masks)
    if constexpr (MODE == 0) load_mask(b);
    // multi-interval masks: this key column's visible rows [fs, fe] per
    // interval (unused intervals and keys beyond Nk empty), clamped to [-1, N]
    int fs[4] = {1, 1, 1, 1}, fe[4] = {0, 0, 0, 0};
    if constexpr (MI) {
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        if (mi < p.M && !dead) {
          const size_t vi = ((size_t)mi * p.B + b) * p.Nk + kcol;
          fs[mi] = min(max(p.lts[vi], -1), p.N);
          fe[mi] = min(max(p.lte[vi], -1), p.N);
        }
      }
    }
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const uint32_t rows_b = smem_u32(smem + C::ROW_OFF) + 128 * half;  // nl[32*half ..]; D at +256
    const uint32_t ds_row = smem_u32(smem + C::DS_OFF) + (uint32_t)((j >> 3) * 1024 + (j & 7) * 128);
    const uint32_t tS = tbase + lane_off + T_S + 32u * half;
    const uint32_t tDP = tbase + lane_off + T_DP + 32u * half;
    bool ok = true;
    int hcur = 0;  // head cursor (per-head masks)
    for (int u = 0; u < U && ok; ++u) {
      const Unit256 un = decode(u, hcur);
      if constexpr (PH) {
        if (un.h != mhead) {
          load_mask(b * p.H_q + un.h);
          mhead = un.h;
        }
      }
      const uint32_t ph = (uint32_t)u & 1u;
      const int r0 = un.qb * 128 + un.half * 64;
      // the row terms of unit u (slot u & 1; the slot is reloaded for u + 2 only
      // after this unit's READY)
      const uint32_t rows_a = rows_b + 512u * (uint32_t)(u & 1);
      ok = __all_sync(kFullB, mbar_wait(&bars[C::B_OFULL + (u & 1)], ((uint32_t)u >> 1) & 1u, abort_flag, p.err));
      if (ok) ok = __all_sync(kFullB, mbar_wait(&bars[C::B_SFULL], ph, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      // masked rows of this thread's key column within its 32-row window
      uint32_t mbits = 0u;
      if (un.part) {
        const int w0 = r0 + 32 * half;
        if constexpr (MI) {
          // masked unless one interval holds the row
          uint32_t vis = 0u;
#pragma unroll
          for (int mi = 0; mi < 4; ++mi) vis |= rows_bits(fs[mi] - w0, fe[mi] + 1 - w0);
          mbits = ~vis | (causal ? rows_bits(-w0, kcol - w0) : 0u) | (dead ? 0xffffffffu : 0u);
        } else {
          mbits = rows_bits(lo0 - w0, lo1 - w0) | rows_bits(up0 - w0, up1 - w0) |
                  (causal ? rows_bits(-w0, kcol - w0) : 0u) | (dead ? 0xffffffffu : 0u);
        }
      }
      // P part: P^T = exp2(scale*log2e*S^T - LSE*log2e), bf16, over this
      // half's first 16 S columns
      uint32_t sv[32];
      tmem_ld32(tS, sv);
      tmem_ld_wait();
      float pf[32];
      uint32_t pk[16];
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
      for (int r4 = 0; r4 < 8; ++r4) {
        const float4 nl4 = lds_f32x4(rows_a + 16 * r4);
        const uint64_t nlp[2] = {f2_pack(nl4.x, nl4.y), f2_pack(nl4.z, nl4.w)};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int rr = 4 * r4 + 2 * e2;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[rr]), __uint_as_float(sv[rr + 1])), sl2x2, nlp[e2]), x0, x1);
          x0 = ((mbits >> rr) & 1u) ? -INFINITY : x0;
          x1 = ((mbits >> (rr + 1)) & 1u) ? -INFINITY : x1;
          pf[rr] = ex2_approx(x0);
          pf[rr + 1] = ex2_approx(x1);
        }
        pk[2 * r4] = pack_bf16x2(pf[4 * r4], pf[4 * r4 + 1]);
        pk[2 * r4 + 1] = pack_bf16x2(pf[4 * r4 + 2], pf[4 * r4 + 3]);
      }
      tmem_st16(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars[C::B_PREADY]);
      // dS part: dS^T = P^T * (dP^T - D), bf16, to shared memory
      ok = __all_sync(kFullB, mbar_wait(&bars[C::B_DPFULL], ph, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      uint32_t pv[32];
      tmem_ld32(tDP, pv);
      tmem_ld_wait();
      uint32_t dk[16];
#pragma unroll
      for (int r4 = 0; r4 < 8; ++r4) {
        const float4 d4 = lds_f32x4(rows_a + 256 + 16 * r4);
        const uint64_t dp[2] = {f2_pack(d4.x, d4.y), f2_pack(d4.z, d4.w)};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int rr = 4 * r4 + 2 * e2;
          const uint64_t t = f2_sub(f2_pack(__uint_as_float(pv[rr]), __uint_as_float(pv[rr + 1])), dp[e2]);
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(pf[rr], pf[rr + 1]), t), d0, d1);
          dk[2 * r4 + e2] = pack_bf16x2(d0, d1);
        }
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        sts_b32x4(ds_row + ((uint32_t)((4 * half + q4) ^ (j & 7)) << 4), dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2],
                  dk[4 * q4 + 3]);
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(&bars[C::B_READY]);
    }
    // epilogue: this half of the dV rows (warps 0-3), staged in the V tile
    // (free once every MMA is done) for two TMA stores
    if (ok) ok = __all_sync(kFullB, mbar_wait(&bars[C::B_FINAL], 0, abort_flag, p.err));
    if (ok && half == 0) {
      tc_fence_after();
      uint8_t* stage = smem + C::V_OFF;
#pragma unroll 1
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tbase + lane_off + T_DV + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const float* f = reinterpret_cast<const float*>(&r[8 * v4]);
          const int col = c0 + 8 * v4;
          sts_b32x4(smem_u32(stage + (col >> 6) * 16384 + j * 128 + ((((col & 63) >> 3) ^ (j & 7)) << 4)),
                    pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[C::B_VSTAGED]);
      if (threadIdx.x == 0 && mbar_wait(&bars[C::B_VSTAGED], 0, abort_flag, p.err)) {
        for (int x = 0; x < DH / 64; ++x) tma_store_3d(&tdv, stage + x * 16384, c0h + x * 64, k0, b * p.H_kv + g);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain
    const int w4 = warp - 8;
    const int c = (w4 << 5) + lane;  // head-dim index within this half = TMEM lane
    const uint32_t lane_off = (uint32_t)(w4 * 32) << 16;
    const uint32_t xp = smem_u32(smem + C::XPOSE_OFF) + w4 * 4096;
    bool ok = true;
    int hcur = 0;  // head cursor (per-head masks)
    for (int u = 0; u < U && ok; ++u) {
      const Unit256 un = decode(u, hcur);
      ok = __all_sync(kFullB, mbar_wait(&bars[C::B_DQFULL], (uint32_t)u & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(tbase + lane_off + T_DQ, v0);
      tmem_ld32(tbase + lane_off + T_DQ + 32, v1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars[C::B_DQEMPTY]);
      // the 32 x 64 slice, 32 rows at a time, row-major through this warp's
      // 4 KB slot, to the fp32 accumulator by TMA reduce-adds (rows past N skipped)
      const int r0 = un.qb * 128 + un.half * 64;
      const int bh = b * p.H_q + un.h;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t* v = hh ? v1 : v0;
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 32; ++r) sts_f32(xp + r * 128 + lane * 4, __uint_as_float(v[r]));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tdq, smem + C::XPOSE_OFF + w4 * 4096, c0h + (w4 << 5), r0 + 32 * hh, bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group_read0();
    // epilogue: this half of the dK rows (thread = KV row j = TMEM lane),
    // scaled, staged in the K tile
    if (ok) ok = __all_sync(kFullB, mbar_wait(&bars[C::B_FINAL], 0, abort_flag, p.err));
    if (ok) {
      tc_fence_after();
      const int j = c;
      uint8_t* stage = smem + C::K_OFF;
      const float sc = p.scale;
#pragma unroll 1
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tbase + lane_off + T_DK + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const float* f = reinterpret_cast<const float*>(&r[8 * v4]);
          const int col = c0 + 8 * v4;
          sts_b32x4(smem_u32(stage + (col >> 6) * 16384 + j * 128 + ((((col & 63) >> 3) ^ (j & 7)) << 4)),
                    pack_bf16x2(f[0] * sc, f[1] * sc), pack_bf16x2(f[2] * sc, f[3] * sc),
                    pack_bf16x2(f[4] * sc, f[5] * sc), pack_bf16x2(f[6] * sc, f[7] * sc));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[C::B_KSTAGED]);
      if (threadIdx.x == 256 && mbar_wait(&bars[C::B_KSTAGED], 0, abort_flag, p.err)) {
        for (int x = 0; x < DH / 64; ++x) tma_store_3d(&tdk, stage + x * 16384, c0h + x * 64, k0, b * p.H_kv + g);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  FM_DEBUG_END(p.err);
  if (warp == 13) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tbase);
  }
}

}  // namespace

// The main kernel of the d = 256 backward: two CTAs per (batch, KV block, kv
// head), one per head-dim half. The row terms (nl, D), the zeroed fp32 dQ
// accumulator and the launch order come from launch_bwd (fm_bwd.cu), which
// also converts dQ afterwards.
cudaError_t launch_bwd256_main(const fm_problem& P, const void* q, const void* k, const void* v, const void* dout,
                               const int32_t* lts, const int32_t* lte, const int32_t* uts, const int32_t* ute,
                               const int32_t* k_off, const int32_t* k_queue, const int32_t* order, const float* nl,
                               const float* dsum, float* dq_acc, void* dk, void* dv, cudaStream_t s, int* err,
                               int mode, int M) {
  using C = B256;
  const int Nk = kv_rows(P);
  const int nK = (Nk + kTile - 1) / kTile;
  const long long BH = (long long)P.B * P.H_q;
  const long long grid = 2LL * P.B * nK * P.H_kv;
  if (grid > INT_MAX) return cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
  if (!make_tmap_bhnd(&tq, q, BH, P.N, C::D, 64) || !make_tmap_bhnd(&tdo, dout, BH, P.N, C::D, 64) ||
      !make_tmap_bhnd(&tk, k, (int64_t)P.B * P.H_kv, Nk, C::D, 128) ||
      !make_tmap_bhnd(&tv, v, (int64_t)P.B * P.H_kv, Nk, C::D, 128) ||
      !make_tmap_bhnd(&tdk, dk, (int64_t)P.B * P.H_kv, Nk, C::D, 128) ||
      !make_tmap_bhnd(&tdv, dv, (int64_t)P.B * P.H_kv, Nk, C::D, 128) ||
      !make_tmap_f32_bhnd(&tdq, dq_acc, BH, P.N, C::D, 32, 32))
    return cudaErrorInvalidValue;
  Bwd256Params prm;
  prm.lts = lts;
  prm.lte = lte;
  prm.uts = uts;
  prm.ute = ute;
  prm.k_off = k_off;
  prm.k_queue = k_queue;
  prm.order = order;
  prm.nl = nl;
  prm.dsum = dsum;
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  prm.B = P.B;
  prm.H_q = P.H_q;
  prm.H_kv = P.H_kv;
  prm.N = P.N;
  prm.Nk = Nk;
  prm.Npad = (P.N + kTile - 1) / kTile * kTile;
  prm.nK = nK;
  prm.G = P.H_q / P.H_kv;
  prm.causal = P.causal ? 1 : 0;
  prm.M = M;
  prm.scale = P.scale;
  prm.scale_log2 = P.scale * 1.4426950408889634f;
  prm.err = err;
  if (mode < 0 || mode > 2) return cudaErrorInvalidValue;
  if (mode == 1 && P.H_q / P.H_kv > kMaxHeads256) return cudaErrorInvalidValue;
  if (mode == 2 && (M < 1 || M > 4)) return cudaErrorInvalidValue;
  // the order table reads one queue per (batch, KV block): natural order with
  // per-head masks
  if (mode == 1) prm.order = nullptr;
  static bool attr_done[3] = {false, false, false};
  if (!attr_done[mode]) {
    cudaError_t e = cudaFuncSetAttribute(mode == 1 ? bwd256_kernel<1> : mode == 2 ? bwd256_kernel<2> : bwd256_kernel<0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_done[mode] = true;
  }
  {
    KernelTimer timer(s, kTimedBwd);
    if (mode == 1)
      bwd256_kernel<1><<<(unsigned)grid, 448, C::SMEM_ALLOC, s>>>(tq, tk, tv, tdo, tdk, tdv, tdq, prm);
    else if (mode == 2)
      bwd256_kernel<2><<<(unsigned)grid, 448, C::SMEM_ALLOC, s>>>(tq, tk, tv, tdo, tdk, tdv, tdq, prm);
    else
      bwd256_kernel<0><<<(unsigned)grid, 448, C::SMEM_ALLOC, s>>>(tq, tk, tv, tdo, tdk, tdv, tdq, prm);
  }
  return cudaGetLastError();
}

}  // namespace fm
