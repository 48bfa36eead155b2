// fm_fwd.cu — masked attention forward on sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes: FlashMask-3 project page, §3.1 — only KV blocks in the
// Q block's queue are loaded ("KV Loader"), scores, softmax and output are
// computed per block and the row-interval mask is applied only on blocks
// tagged partial ("MMA Consumer"). The online-softmax recurrence (running max
// m, running sum l, rescale of O, final O / l) is the one of "Flash MSA
// Attention Kernel Implementation", "The Flash Core: Tiling Over the Memory
// Hierarchy".
//
// GB300 design (not the pages' Hopper design):
//   * Work unit = (batch b, Q block qb, a PAIR of query heads of the same GQA
//     group). Both heads share the K/V head and the mask, so they share every
//     K/V tile load and the same queue.
//   * Persistent: one CTA per SM. Each CTA starts with unit blockIdx.x and
//     then takes the next unhandled unit from a work counter, so load balance
//     is dynamic and the units in flight stay close to the sequence order.
//     The producer decodes each unit into a two-slot unit ring in shared
//     memory (header + queue); all rings and barriers keep counting across
//     units, so the next unit's loads and first S MMAs overlap the current
//     unit's last softmax and epilogue, and the setup (barriers, TMEM
//     allocation) is paid once per SM.
//   * Warp roles (320 threads):
//       warps 0-3  softmax for query tile 0 (one thread per query row)
//       warps 4-7  softmax for query tile 1
//       warp  8    producer: unit ring, TMA loads of Q, K, V and the mask
//                  vectors of partial blocks into shared memory rings
//       warp  9    MMA issuer (one elected lane) and TMEM owner
//   * TMEM (512 columns x 128 lanes): S_t at columns [128t, 128t+128); P_t is
//     written back as bf16 over the first 64 columns of S_t and consumed from
//     TMEM by the PV MMA; O_t at [256 + t*d, 256 + (t+1)*d).
//   * The MMA warp interleaves the two tiles: PV_0(j-1), S_0(j), PV_1(j-1),
//     S_1(j), so the tensor core works on one tile while softmax works on the
//     other. A unit's last PV goes out before anything of the next unit.
//   * Rescaling of O is lazy: the running max used for exponentials only moves
//     when the block max exceeds it by more than 8 (log2 units), so P <= 256;
//     O and l are always scaled consistently, so O / l is unchanged.
//   * Epilogue: each softmax warp writes its 32 rows of O / l, 32 columns at
//     a time, into its own 2 KB shared-memory slot and stores them with one
//     TMA store (the Q tiles already hold the next unit's Q).
//   * Unit order: longest queue first (an LPT order computed on the device
//     from the queue offsets) for passes of a few waves, natural order for
//     long passes, where units of neighbouring query blocks share K / V tiles
//     in L2.
//   * One-head units (per-head vectors, or one query head per kv head: the
//     SINGLE instantiation): the second tile's S columns are a second S
//     buffer; block k uses buffer k % 2, S(k) is issued ahead of PV(k - 1),
//     so the next block's scores are computed while the softmax works on the
//     current one, and the softmax arrives on PREADY[k % 2] (one barrier per
//     buffer: the softmax may finish block k + 1 before PV(k) is issued, and
//     a single barrier would then be two phases ahead of the MMA warp's wait).
//   * Other mask forms: with per-head vectors a unit is one head with its own
//     queue and vector row; with multi-interval masks (the MI instantiation)
//     the queues are those of the union classification and a partial block's
//     mask is built from every interval's FMS / FME (a row is masked unless
//     one interval holds it).
#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>
#include <cuda.h>
#include "fm_internal.h"
#include "mask_bits.cuh"
#include "sm100.cuh"
#include "lpt_order.cuh"

namespace fm {
namespace {

// F8: Q, K, V (and P) are e4m3 instead of bf16 (the FP8 forward). MI:
// multi-interval masks (a mask slot holds FMS[128], FME[128] of up to four
// intervals).
template <int D, bool F8 = false, bool MI = false>
struct FwdCfg {
  static constexpr int ES = F8 ? 1 : 2;         // bytes per Q / K / V element
  static constexpr int TILE = 128 * D * ES;     // bytes of one 128-row tile
  static constexpr int BOX_COLS = 128 / ES;     // elements in one 128-byte swizzled row of a TMA box
  static constexpr int BOXES = D / BOX_COLS;    // 16 KB TMA boxes per tile
  static constexpr int STAGES = (F8 || D == 64) ? 4 : 2;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + STAGES * TILE;
  static constexpr int M_OFF = V_OFF + STAGES * TILE;
  // mask slot: LTS[128], LTE[128], UTS[128], UTE[128]; MI: FMS[128], FME[128] x 4
  static constexpr int M_BYTES = MI ? 4 * 2 * 128 * 4 : 4 * 128 * 4;
  // O staging: one 2 KB slot per softmax warp (32 rows x 32 columns bf16,
  // 64-byte swizzle), the source of that warp's TMA stores
  static constexpr int O_OFF = M_OFF + STAGES * M_BYTES;
  static constexpr int O_SLOT = 32 * 32 * 2;
  // unit ring: the producer decodes each unit once into one of two slots (a
  // header and the first QUEUE_CAP queue entries); the other roles read it there
  static constexpr int QUEUE_CAP = 512;
  static constexpr int U_HDR = 16;  // int32 header words
  static constexpr int U_BYTES = (U_HDR + QUEUE_CAP) * 4;
  static constexpr int U_OFF = O_OFF + 8 * O_SLOT;
  // deferred epilogue: per softmax thread {l, m, output row head, q0} of the
  // unit whose O is still in TMEM
  static constexpr int EPI_OFF = U_OFF + 2 * U_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + 256 * 16;
  static constexpr int B_QFULL = 0;
  static constexpr int B_QFREE = 1;
  static constexpr int B_UFULL = 2;   // [2]
  static constexpr int B_UEMPTY = 4;  // [2]
  static constexpr int B_KFULL = 6;
  static constexpr int B_KEMPTY = B_KFULL + STAGES;
  static constexpr int B_VFULL = B_KEMPTY + STAGES;
  static constexpr int B_VEMPTY = B_VFULL + STAGES;
  static constexpr int B_MFULL = B_VEMPTY + STAGES;
  static constexpr int B_MEMPTY = B_MFULL + STAGES;
  static constexpr int B_SFULL = B_MEMPTY + STAGES;  // [2]
  static constexpr int B_PREADY = B_SFULL + 2;       // [2]
  static constexpr int B_ODONE = B_PREADY + 2;       // [2]
  static constexpr int NBAR = B_ODONE + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
};

// unit header words in the unit ring
enum { UH_N = 0, UH_T = 1, UH_QB = 2, UH_B = 3, UH_H0 = 4, UH_G = 5, UH_QBEG = 6, UH_END = 7 };

struct FwdParams {
  const int32_t* lts;
  const int32_t* lte;
  const int32_t* uts;
  const int32_t* ute;
  const int32_t* q_off;
  const int32_t* q_queue;
  const int32_t* order;  // order of (b, qb) in the unit sequence, or null: natural order
  int* next_unit;        // work counter, zero at launch: units handed out past the first gridDim.x
  __nv_bfloat16* o;
  float* lse;
  int B, H_q, H_kv, N, Nk, nQ, nK, G, PG, causal;  // N query rows, Nk key rows
  int units;  // B * nQ * H_kv * PG work units (per-head masks: B * H_q * nQ)
  int per_head;  // mask vectors and queues per (batch, query head): one head per unit
  // multi-interval masks: lts / lte hold FMS / FME, (M, B, N_kv), M >= 1
  // (the MI instantiation); 0 otherwise
  int M;
  float scale_log2;
  float o_scale;  // multiplies O / l (the V dequantization scale of the FP8 forward; 1 otherwise)
  int* err;
};

constexpr float kLn2 = 0.69314718055994530942f;
constexpr unsigned kFull = 0xffffffffu;

// One work unit: (batch b, Q block qb, a pair of query heads h0, h0 + 1 of KV
// head g; T = 1 when the group has an odd head left over) and its queue.
struct Unit {
  int b, qb, g, h0, T, qbeg, n, vrow;  // vrow: the row of the mask vectors
};

__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int k) {
  Unit u;
  if (p.per_head) {
    // queue rows in (batch, head, Q block) order, one head per unit
    const int r = p.order ? p.order[k] : k;
    const int bh = r / p.nQ;
    u.qb = r - bh * p.nQ;
    u.b = bh / p.H_q;
    u.h0 = bh - u.b * p.H_q;
    u.g = u.h0 / p.G;
    u.T = 1;
    u.qbeg = p.q_off[r];
    u.n = p.q_off[r + 1] - u.qbeg;
    u.vrow = bh;
    return u;
  }
  const int per = p.H_kv * p.PG;
  const int oi = k / per, gp = k - oi * per;
  u.g = gp / p.PG;
  const int pp = gp - u.g * p.PG;
  const int bq = p.order ? p.order[oi] : oi;
  u.b = bq / p.nQ;
  u.qb = bq - u.b * p.nQ;
  u.h0 = u.g * p.G + 2 * pp;
  u.T = (2 * pp + 1 < p.G) ? 2 : 1;
  u.qbeg = p.q_off[bq];
  u.n = p.q_off[bq + 1] - u.qbeg;
  u.vrow = u.b;
  return u;
}

// A queue block is partial when the classification tagged it so, or when it
// is the last key block and N is not a multiple of 128 (its tail columns are
// masked for every row).
__device__ __forceinline__ bool block_partial(const FwdParams& p, int e) {
  return (e & 1) || ((e >> 1) == p.nK - 1 && (p.Nk & 127));
}

// MI: multi-interval masks (mask slots hold FMS / FME of every interval).
// SINGLE: every unit has one query head (per-head masks, or one query head per
// kv head): the second tile's S columns serve as a second S buffer, so S of a
// unit's next block is computed while the softmax works on the current one.
template <int D, bool F8, bool MI, bool SINGLE>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to, const FwdParams p) {
  using C = FwdCfg<D, F8, MI>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  FM_DEBUG_BEGIN();
  // heads per unit for the whole grid: 2 when the GQA group has two or more
  // query heads; an odd group also has single-head units
  const int tmax = (p.G >= 2 && !p.per_head) ? 2 : 1;

  if (threadIdx.x == 0) {
    // an unread timeout from an earlier launch: skip the work, keep the CTA cheap
    *abort_flag = timeout_pending(p.err) ? 1 : 0;
    mbar_init(&bars[C::B_QFULL], 1);
    mbar_init(&bars[C::B_QFREE], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[C::B_UFULL + s], 1);
      mbar_init(&bars[C::B_UEMPTY + s], 1 + 4 * tmax);  // the MMA lane and the softmax warps
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars[C::B_KFULL + s], 1);
      mbar_init(&bars[C::B_KEMPTY + s], 1);
      mbar_init(&bars[C::B_VFULL + s], 1);
      mbar_init(&bars[C::B_VEMPTY + s], 1);
      mbar_init(&bars[C::B_MFULL + s], 1);
      mbar_init(&bars[C::B_MEMPTY + s], 4 * tmax);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars[C::B_SFULL + t], 1);
      mbar_init(&bars[C::B_PREADY + t], 128);
      mbar_init(&bars[C::B_ODONE + t], 1);
    }
    fence_mbar_init();
  }
  if constexpr (MI) {
    // the interval places past M of every mask slot hold an empty interval
    // (FMS 1, FME 0) for the whole launch: the producer never writes them, and
    // the softmax warps read two or four intervals without a per-interval test
    int* mv = reinterpret_cast<int*>(smem + C::M_OFF);
    for (int i = threadIdx.x; i < S * 1024; i += blockDim.x)
      if (((i & 1023) >> 8) >= p.M) mv[i] = (i & 255) < 128 ? 1 : 0;
  }
  if (warp == 9) tmem_alloc<512>(tmem_slot);
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // unit ring slot us: header word w, queue entry j (entries past the
  // staged prefix come from global memory)
  auto hdr_at = [&](int us, int w) -> int { return lds_s32(smem_u32(smem + C::U_OFF + us * C::U_BYTES) + 4 * w); };
  auto queue_at = [&](int us, int j) -> int {
    return (j < C::QUEUE_CAP) ? lds_s32(smem_u32(smem + C::U_OFF + us * C::U_BYTES) + 4 * (C::U_HDR + j))
                              : p.q_queue[hdr_at(us, UH_QBEG) + j];
  };

  // Every role walks the CTA's unit sequence through the unit ring (filled by
  // the producer). Rings (units, K, V, mask vectors) and per-head barriers
  // keep counting across units, so the loads and MMAs of the next unit start
  // while the softmax warps finish the current one.
  if (*abort_flag) {
    // fall through to teardown
  } else if (warp == 8) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t jt = 0, pidx = 0, uq = 0;  // K/V blocks, partial blocks, non-empty units so far
    // Units are handed out dynamically: each CTA starts with unit blockIdx.x,
    // then takes the next unhandled one from the work counter, so CTAs that
    // drew short queues take more units and the units in flight stay close
    // to the sequence order (neighbours share K / V tiles in L2).
    int k = blockIdx.x;
    for (uint32_t ui = 0; ok; ++ui) {
      // decode the unit into the ring (its queue staged in shared memory)
      const int us = ui & 1;
      ok = __all_sync(kFull, mbar_wait(&bars[C::B_UEMPTY + us], ((ui >> 1) & 1u) ^ 1u, abort_flag, p.err));
      if (!ok) break;
      int* h = reinterpret_cast<int*>(smem + C::U_OFF + us * C::U_BYTES);
      if (k >= p.units) {
        // no work left: tell the other roles
        if (lane == 0) h[UH_END] = 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_UFULL + us]);
        break;
      }
      // the next unit's index, requested now and used after this unit
      int k_next = 0;
      if (lane == 0) k_next = (int)gridDim.x + atomicAdd(p.next_unit, 1);
      const Unit u = decode_unit(p, k);
      {
        if (lane == 0) {
          h[UH_END] = 0;
          h[UH_N] = u.n;
          h[UH_T] = u.T;
          h[UH_QB] = u.qb;
          h[UH_B] = u.b;
          h[UH_H0] = u.h0;
          h[UH_G] = u.g;
          h[UH_QBEG] = u.qbeg;
        }
        int* sq = h + C::U_HDR;
        const int m = min(u.n, C::QUEUE_CAP);
        for (int j0 = 0; j0 < m; j0 += 128) {
          int e[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int j = j0 + 32 * r + lane;
            e[r] = (j < m) ? p.q_queue[u.qbeg + j] : 0;
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int j = j0 + 32 * r + lane;
            if (j < m) sq[j] = e[r];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_UFULL + us]);
      }
      k = __shfl_sync(kFull, k_next, 0);
      if (u.n <= 0) continue;
      for (int j = 0; j < u.n && ok; ++j) {
        const int e = queue_at(us, j);
        const int kb = e >> 1;
        const size_t vbase = (size_t)u.vrow * p.Nk;
        if (kb < 0 || kb >= p.nK) {
          if (lane == 0) record_error(p.err, FM_DEV_ERR_QUEUE);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const bool part = block_partial(p, e);
        const int slot = jt % S;
        const uint32_t ph = (jt / S) & 1u;
        if (lane == 0) {
          ok = mbar_wait(&bars[C::B_KEMPTY + slot], ph ^ 1u, abort_flag, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&bars[C::B_KFULL + slot], C::TILE);
            for (int x = 0; x < C::BOXES; ++x)
              tma_load_3d(smem + C::K_OFF + slot * C::TILE + x * 16384, &tk, &bars[C::B_KFULL + slot],
                          x * C::BOX_COLS, kb * 128, u.b * p.H_kv + u.g);
          }
          if (ok && j == 0) {
            // the Q tiles of this unit, once the last S MMA of the previous one is done
            if (uq > 0) ok = mbar_wait(&bars[C::B_QFREE], (uq - 1) & 1u, abort_flag, p.err);
            if (ok) {
              mbar_arrive_expect_tx(&bars[C::B_QFULL], u.T * C::TILE);
              for (int t = 0; t < u.T; ++t)
                for (int x = 0; x < C::BOXES; ++x)
                  tma_load_3d(smem + C::Q_OFF + t * C::TILE + x * 16384, &tq, &bars[C::B_QFULL],
                              x * C::BOX_COLS, u.qb * 128, u.b * p.H_q + u.h0 + t);
            }
          }
        }
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
        if (part && MI) {
          // multi-interval masks: FMS[128], FME[128] of every interval, raw;
          // a key beyond Nk gets an empty interval
          const int ms = pidx % S;
          const uint32_t mph = (pidx / S) & 1u;
          ok = __all_sync(kFull, mbar_wait(&bars[C::B_MEMPTY + ms], mph ^ 1u, abort_flag, p.err));
          if (!ok) break;
          uint8_t* sm = smem + C::M_OFF + ms * C::M_BYTES;
          const int c0 = kb * 128;
          bool aligned = c0 + 128 <= p.Nk;
          for (int mi = 0; mi < p.M; ++mi) {
            const size_t o = ((size_t)mi * p.B + u.b) * p.Nk + c0;
            aligned = aligned && ((reinterpret_cast<uintptr_t>(p.lts + o) | reinterpret_cast<uintptr_t>(p.lte + o)) &
                                  15u) == 0;
          }
          if (aligned) {
            if (lane == 0) {
              uint64_t* fb = &bars[C::B_MFULL + ms];
              mbar_arrive_expect_tx(fb, 2 * 512 * p.M);
              for (int mi = 0; mi < p.M; ++mi) {
                const size_t o = ((size_t)mi * p.B + u.b) * p.Nk + c0;
                bulk_load(sm + mi * 1024, p.lts + o, 512, fb);
                bulk_load(sm + mi * 1024 + 512, p.lte + o, 512, fb);
              }
            }
          } else {
            int* v = reinterpret_cast<int*>(sm);
            for (int mi = 0; mi < p.M; ++mi) {
              const size_t o = ((size_t)mi * p.B + u.b) * p.Nk;
              for (int c = lane; c < 128; c += 32) {
                const int col = c0 + c;
                const bool in = col < p.Nk;
                v[mi * 256 + c] = in ? p.lts[o + col] : 1;
                v[mi * 256 + 128 + c] = in ? p.lte[o + col] : 0;
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[C::B_MFULL + ms]);
          }
          ++pidx;
        } else if (part) {
          // the block's four mask vectors, raw, as 4 x 128 int32 (LTS, LTE, UTS,
          // UTE); the softmax warps clamp and check them
          const int ms = pidx % S;
          const uint32_t mph = (pidx / S) & 1u;
          ok = __all_sync(kFull, mbar_wait(&bars[C::B_MEMPTY + ms], mph ^ 1u, abort_flag, p.err));
          if (!ok) break;
          uint8_t* sm = smem + C::M_OFF + ms * C::M_BYTES;
          const int c0 = kb * 128;
          const size_t o = vbase + c0;
          const bool aligned = ((reinterpret_cast<uintptr_t>(p.lts + o) | reinterpret_cast<uintptr_t>(p.lte + o) |
                                 reinterpret_cast<uintptr_t>(p.uts + o) | reinterpret_cast<uintptr_t>(p.ute + o)) &
                                15u) == 0;
          if (c0 + 128 <= p.Nk && aligned) {
            // whole block in range and 16-byte aligned: four bulk copies
            if (lane == 0) {
              uint64_t* fb = &bars[C::B_MFULL + ms];
              mbar_arrive_expect_tx(fb, 4 * 512);
              bulk_load(sm + 0, p.lts + o, 512, fb);
              bulk_load(sm + 512, p.lte + o, 512, fb);
              bulk_load(sm + 1024, p.uts + o, 512, fb);
              bulk_load(sm + 1536, p.ute + o, 512, fb);
            }
          } else {
            int* v = reinterpret_cast<int*>(sm);
            for (int c = lane; c < 128; c += 32) {
              const int col = c0 + c;
              const bool in = col < p.Nk;  // a key beyond Nk is masked for every row
              v[c] = in ? p.lts[vbase + col] : 0;
              v[128 + c] = in ? p.lte[vbase + col] : p.N;
              v[256 + c] = in ? p.uts[vbase + col] : 0;
              v[384 + c] = in ? p.ute[vbase + col] : 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[C::B_MFULL + ms]);
          }
          ++pidx;
        }
        if (lane == 0) {
          ok = mbar_wait(&bars[C::B_VEMPTY + slot], ph ^ 1u, abort_flag, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&bars[C::B_VFULL + slot], C::TILE);
            for (int x = 0; x < C::BOXES; ++x)
              tma_load_3d(smem + C::V_OFF + slot * C::TILE + x * 16384, &tv, &bars[C::B_VFULL + slot],
                          x * C::BOX_COLS, kb * 128, u.b * p.H_kv + u.g);
          }
        }
        ok = __shfl_sync(kFull, ok, 0);
        ++jt;
      }
      ++uq;
    }
  } else if (warp == 9) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // S = Q K^T, both K-major; O += P V, V MN-major
      const uint32_t id_s = F8 ? idesc_e4m3_f32(128, 128, 0, 0) : idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t id_o = F8 ? idesc_e4m3_f32(128, D, 0, 1) : idesc_bf16_f32(128, D, 0, 1);
      // descriptors built once; per MMA only the start-address field moves
      // (a 64-bit add of a constant), which keeps the issue ahead of the tensor core
      constexpr uint64_t kTileStep = C::TILE >> 4;
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::Q_OFF), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::K_OFF), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::V_OFF), 16384, 1024);
      bool ok = true;
      uint32_t jt = 0, uq = 0, ui = 0;
      uint32_t npv0 = 0u, npv1 = 0u;  // PV MMAs issued per head so far
      // PV of one block for head t: V from ring slot vs; the unit's first
      // block overwrites O instead of accumulating
      auto issue_pv = [&](int t, uint32_t vs, bool first, int pb) -> bool {
        // one-head units: one PREADY per S buffer (block k arrives on PREADY[k % 2],
        // phase k / 2), so the softmax, which may finish block k + 1 before PV(k)
        // is issued, is never two phases ahead of this wait
        const uint32_t pr = SINGLE ? (uint32_t)pb : (uint32_t)t;
        const uint32_t pph = SINGLE ? (npv0 >> 1) : (t ? npv1 : npv0);
        if (!mbar_wait(&bars[C::B_PREADY + pr], pph & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t tS = tbase + (uint32_t)(pb * 128);  // P over S buffer pb
        const uint32_t tO = tbase + 256u + (uint32_t)(t * D);
        const uint64_t vd = dV0 + kTileStep * (uint64_t)vs;
        // k-steps of 16 bf16 (32 e4m3) keys: 8 TMEM columns of P, 16 (32) rows of V
#pragma unroll
        for (int kk = 0; kk < (F8 ? 4 : 8); ++kk) {
          if constexpr (F8)
            mma_ts_f8(tO, tS + (uint32_t)(kk * 8), vd + (uint64_t)(kk * 256), id_o, (!first || kk > 0) ? 1u : 0u);
          else
            mma_ts(tO, tS + (uint32_t)(kk * 8), vd + (uint64_t)(kk * 128), id_o, (!first || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars[C::B_ODONE + t]);
        if (t) ++npv1;
        else ++npv0;
        return true;
      };
      for (; ok; ++ui) {
        const int us = ui & 1;
        ok = mbar_wait(&bars[C::B_UFULL + us], (ui >> 1) & 1u, abort_flag, p.err);
        if (!ok || hdr_at(us, UH_END)) break;
        const int n = hdr_at(us, UH_N), T = hdr_at(us, UH_T);
        mbar_arrive(&bars[C::B_UEMPTY + us]);
        if (n <= 0) continue;
        ok = mbar_wait(&bars[C::B_QFULL], uq & 1u, abort_flag, p.err);
        tc_fence_after();
        uint32_t pslot = 0;
        // S of one head into its TMEM columns (the tensor core runs it after
        // that head's PV, issued just before, which reads the same columns).
        // The head loop below is written out (two heads known at compile
        // time): with a runtime head loop the issue ran measurably behind
        // the tensor core on long unmasked units.
        auto issue_s = [&](int t, int slot, int sb) {
          const uint32_t tS = tbase + (uint32_t)(sb * 128);  // into S buffer sb
          const uint64_t qd = dQ0 + kTileStep * (uint64_t)t, kd = dK0 + kTileStep * (uint64_t)slot;
          // k-steps of 32 bytes (16 bf16 / 32 e4m3), four per 128-byte swizzled row
#pragma unroll
          for (int kk = 0; kk < D * C::ES / 32; ++kk) {
            const uint64_t off = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);
            if constexpr (F8)
              mma_ss_f8(tS, qd + off, kd + off, id_s, kk > 0 ? 1u : 0u);
            else
              mma_ss(tS, qd + off, kd + off, id_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars[C::B_SFULL + sb]);
        };
        if constexpr (SINGLE) {
          // one head: S(j) goes to buffer jt % 2 ahead of PV(j - 1), which
          // reads P(j - 1) from the other buffer. S(j) overwrites P(j - 2):
          // it is issued only once PV(j - 2) has completed (ODONE, counted
          // one completion at a time in pv_done)
          for (int j = 0; j < n && ok; ++j) {
            const int slot = jt % S;
            ok = mbar_wait(&bars[C::B_KFULL + slot], (jt / S) & 1u, abort_flag, p.err);
            tc_fence_after();
            tc_fence_after();
            if (!ok) break;
            issue_s(0, slot, (int)(jt & 1u));
            mma_commit(&bars[C::B_KEMPTY + slot]);
            if (j == n - 1) mma_commit(&bars[C::B_QFREE]);
            if (j > 0) {
              ok = mbar_wait(&bars[C::B_VFULL + pslot], ((jt - 1) / S) & 1u, abort_flag, p.err);
              tc_fence_after();
              if (ok) ok = issue_pv(0, pslot, j == 1, (int)((jt - 1) & 1u));
              if (ok) mma_commit(&bars[C::B_VEMPTY + pslot]);
            }
            pslot = slot;
            ++jt;
          }
          if (!ok) break;
          ok = mbar_wait(&bars[C::B_VFULL + pslot], ((jt - 1) / S) & 1u, abort_flag, p.err);
          tc_fence_after();
          if (ok) ok = issue_pv(0, pslot, n == 1, (int)((jt - 1) & 1u));
          if (!ok) break;
          mma_commit(&bars[C::B_VEMPTY + pslot]);
          ++uq;
          continue;
        }
        for (int j = 0; j < n && ok; ++j) {
          const int slot = jt % S;
          ok = mbar_wait(&bars[C::B_KFULL + slot], (jt / S) & 1u, abort_flag, p.err);
          tc_fence_after();
          if (ok && j > 0) {
            ok = mbar_wait(&bars[C::B_VFULL + pslot], ((jt - 1) / S) & 1u, abort_flag, p.err);
            tc_fence_after();
          }
          if (!ok) break;
          if (j > 0 && !issue_pv(0, pslot, j == 1, 0)) { ok = false; break; }
          issue_s(0, slot, 0);
          if (T == 2) {
            if (j > 0 && !issue_pv(1, pslot, j == 1, 1)) { ok = false; break; }
            issue_s(1, slot, 1);
          }
          if (j > 0) mma_commit(&bars[C::B_VEMPTY + pslot]);
          mma_commit(&bars[C::B_KEMPTY + slot]);
          if (j == n - 1) mma_commit(&bars[C::B_QFREE]);
          pslot = slot;
          ++jt;
        }
        if (!ok) break;
        // the unit's last PV, before anything of the next unit: the softmax
        // warps' epilogue waits for it
        ok = mbar_wait(&bars[C::B_VFULL + pslot], ((jt - 1) / S) & 1u, abort_flag, p.err);
        tc_fence_after();
        for (int t = 0; t < T && ok; ++t) ok = issue_pv(t, pslot, n == 1, t);
        if (!ok) break;
        mma_commit(&bars[C::B_VEMPTY + pslot]);
        ++uq;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tO = tbase + lane_off + 256u + (uint32_t)(t * D);
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const uint32_t oslot = smem_u32(smem + C::O_OFF + warp * C::O_SLOT);
    const uint32_t sepi = smem_u32(smem + C::EPI_OFF) + 16u * threadIdx.x;
    bool ok = t < tmax;
    uint32_t jh = 0, pidx = 0, ui = 0;  // blocks of this head, partial blocks, units so far
    // Epilogue of a finished unit, deferred: its O stays in TMEM until the
    // next unit's first P is written, so the O loads sit after that block's
    // softmax (the last PV has finished by then) and the stores overlap the
    // tensor core's next PV and S. pend: a unit's O is waiting.
    bool pend = false;
    // O / l of the unit in sepi, 32 columns at a time, through the warp's
    // staging slot (64-byte swizzle: row r's 16-byte chunk c sits at chunk
    // c ^ ((r >> 1) & 3), which keeps the row-per-lane stores conflict-free)
    // to one TMA store of the warp's 32 rows (rows past N are clipped by it),
    // then the row's LSE.
    auto store_o = [&](const uint32_t(&orow)[D]) {
      const int4 st = lds_s32x4(sepi);
      const float l = __int_as_float(st.x), m = __int_as_float(st.y);
      const int bh = st.z, q0e = st.w;
      const int w0e = q0e + ((warp & 3) << 5), ie = q0e + row;
      const float inv = (l > 0.f) ? p.o_scale / l : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        const float* f = reinterpret_cast<const float*>(&orow[c0]);
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) w[c] = pack_bf16x2(f[2 * c] * inv, f[2 * c + 1] * inv);
        if (lane == 0) bulk_wait_group_read0();  // the slot's previous store has read it
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          sts_b32x4(oslot + 64 * lane + 16 * (c ^ ((lane >> 1) & 3)), w[4 * c], w[4 * c + 1], w[4 * c + 2],
                    w[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&to, oslot, c0, w0e, bh);
          bulk_commit_group();
        }
      }
      if (ie < p.N) p.lse[(size_t)bh * p.N + ie] = (l > 0.f) ? (m * kLn2 + logf(l)) : -INFINITY;
    };
    // the pending epilogue with nothing to hide behind: wait for the last PV
    auto flush = [&]() -> bool {
      if (!pend) return true;
      pend = false;
      if (!__all_sync(kFull, mbar_wait(&bars[C::B_ODONE + t], (jh - 1) & 1u, abort_flag, p.err))) return false;
      tc_fence_after();
      uint32_t orow[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32(tO + c0, *reinterpret_cast<uint32_t(*)[32]>(&orow[c0]));
      tmem_ld_wait();
      store_o(orow);
      return true;
    };
    for (; ok; ++ui) {
      const int us = ui & 1;
      ok = __all_sync(kFull, mbar_wait(&bars[C::B_UFULL + us], (ui >> 1) & 1u, abort_flag, p.err));
      if (!ok) break;
      if (hdr_at(us, UH_END)) {
        ok = flush();
        break;
      }
      const int n = hdr_at(us, UH_N), T = hdr_at(us, UH_T);
      const int q0 = hdr_at(us, UH_QB) * 128;
      const int i = q0 + row;
      const int w0 = q0 + ((warp & 3) << 5);  // the warp's first row
      if (n <= 0 || t >= T) {
        ok = flush();
        if (!ok) break;
      }
      if (n <= 0) {
        // No visible key for any row of this unit: O = 0 (the warp's staging
        // slot, zeroed, is the source of all its stores), LSE = -inf.
        if (n < 0 && threadIdx.x == 0) record_error(p.err, FM_DEV_ERR_QUEUE);
        if (t < T) {
          const int bh = hdr_at(us, UH_B) * p.H_q + hdr_at(us, UH_H0) + t;
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) sts_b32x4(oslot + 64 * lane + 16 * c, 0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            for (int c0 = 0; c0 < D; c0 += 32) tma_store_3d(&to, oslot, c0, w0, bh);
            bulk_commit_group();
          }
          if (i < p.N) p.lse[(size_t)bh * p.N + i] = -INFINITY;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_UEMPTY + us]);
        continue;
      }
      if (t >= T) {
        // a single-head unit: the second head's warps only advance the
        // partial-block count (head 0 releases the mask ring for both)
        uint32_t c = 0;
        for (int j0 = 0; j0 < n; j0 += 32) {
          const bool part = (j0 + lane < n) && block_partial(p, queue_at(us, j0 + lane));
          c += __popc(__ballot_sync(kFull, part));
        }
        pidx += c;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_UEMPTY + us]);
        continue;
      }
      const uint32_t mrel = (T < tmax) ? 2u : 1u;  // MEMPTY arrivals per warp
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n; ++j) {
        const int e = queue_at(us, j);
        const int kb = e >> 1;
        const bool part = block_partial(p, e);
        // Partial blocks: masked-row bits of this thread's query row over the
        // block's 128 key columns, built while S is still being computed. Lane
        // c of the warp builds the bits of key column 32k + c over the warp's
        // 32 rows; a bit transpose hands each lane its own row.
        uint32_t rb[4] = {0u, 0u, 0u, 0u};
        if (part) {
          const int ms = pidx % S;
          ok = __all_sync(kFull, mbar_wait(&bars[C::B_MFULL + ms], (pidx / S) & 1u, abort_flag, p.err));
          if (!ok) break;
          const uint32_t sm = smem_u32(smem + C::M_OFF + ms * C::M_BYTES);
          const int kc0 = kb * 128;
          // Values outside [0, N] only need clamping here: fm_classify_tiles,
          // run on the same vectors, flags them.
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int c = 32 * kq + lane;
            uint32_t colbits;
            if constexpr (MI) {
              // masked unless one interval [FMS, FME] holds the row (the
              // places past M hold empty intervals)
              auto iv = [&](int mi) -> uint32_t {
                const int f0 = lds_s32(sm + mi * 1024 + 4 * c), f1 = lds_s32(sm + mi * 1024 + 512 + 4 * c);
                return window_bits(f0, min(f1, p.N) + 1, w0);
              };
              const uint32_t vis = (p.M <= 2) ? (iv(0) | iv(1)) : (iv(0) | iv(1) | iv(2) | iv(3));
              colbits = ~vis | (causal ? window_bits(w0, kc0 + c, w0) : 0u);
            } else {
              const int a0 = lds_s32(sm + 4 * c), a1 = lds_s32(sm + 512 + 4 * c);  // LTS, LTE of key column kc0 + c
              const int u0 = lds_s32(sm + 1024 + 4 * c), u1 = lds_s32(sm + 1536 + 4 * c);  // UTS, UTE
              colbits = window_bits(a0, a1, w0) | window_bits(u0, u1, w0) |
                        (causal ? window_bits(w0, kc0 + c, w0) : 0u);
            }
            rb[kq] = warp_transpose32(colbits, lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_cnt(&bars[C::B_MEMPTY + ms], mrel);
          ++pidx;
        }
        // this block's S buffer (one-head units alternate both buffers)
        const uint32_t sb = SINGLE ? (jh & 1u) : (uint32_t)t;
        ok = __all_sync(kFull, mbar_wait(&bars[C::B_SFULL + sb], (SINGLE ? (jh >> 1) : jh) & 1u, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tbase + lane_off + (sb << 7);
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
          for (int c = 0; c < 128; ++c)
            sr[c] = ((rb[c >> 5] >> (c & 31)) & 1u) ? __float_as_uint(-INFINITY) : sr[c];
        }
        // row max with three-input max, four independent chains
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mx0 = max3f(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          mx1 = max3f(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          mx2 = max3f(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
          mx3 = max3f(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
        }
        const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
        const float m_blk = mx * sl2;
        const float m_new = fmaxf(m_run, m_blk);
        const bool resc = m_new > m_run + 8.0f;
        float factor = 1.f;
        if (resc) {
          factor = ex2_approx(m_run - m_new);
          m_run = m_new;
        }
        const float msafe = (m_run == -INFINITY) ? 0.f : m_run;
        // exponent arguments and the row sum on column pairs (f32x2)
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-msafe, -msafe);
        uint64_t rs0 = f2_pack(0.f, 0.f), rs1 = rs0;
        // P as bf16 pairs (e4m3 quadruples for the FP8 forward), key order low to high
        uint32_t pk[64];
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2x2, nm2), x0, x1);
          const float a = ex2_approx(x0), bb = ex2_approx(x1);
          if (c & 1) rs1 = f2_add(rs1, f2_pack(a, bb));
          else rs0 = f2_add(rs0, f2_pack(a, bb));
          if constexpr (F8) {
            if (c & 1) pk[c >> 1] = pack_e4m3x4(pa, pb, a, bb);
            else {
              pa = a;
              pb = bb;
            }
          } else {
            pk[c] = pack_bf16x2(a, bb);
          }
        }
        float r0a, r0b, r1a, r1b;
        f2_unpack(rs0, r0a, r0b);
        f2_unpack(rs1, r1a, r1b);
        l_run = l_run * factor + ((r0a + r0b) + (r1a + r1b));
        {
          const uint32_t(&p0)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]);
          const uint32_t(&p1)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]);
          tmem_st16(tS + 0, p0);
          tmem_st16(tS + 16, p1);
          if constexpr (!F8) {
            const uint32_t(&p2)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[32]);
            const uint32_t(&p3)[16] = *reinterpret_cast<const uint32_t(*)[16]>(&pk[48]);
            tmem_st16(tS + 32, p2);
            tmem_st16(tS + 48, p3);
          }
          tmem_st_wait();
        }
        if (j > 0 && __any_sync(kFull, resc)) {
          // O holds PV of the unit's earlier blocks: wait for the last of them,
          // then rescale the row.
          ok = __all_sync(kFull, mbar_wait(&bars[C::B_ODONE + t], (jh - 1) & 1u, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
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
        if (j == 0 && pend) {
          // the previous unit's O: its last PV is done once ODONE shows it
          pend = false;
          ok = __all_sync(kFull, mbar_wait(&bars[C::B_ODONE + t], (jh - 1) & 1u, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
          uint32_t orow[D];
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32(tO + c0, *reinterpret_cast<uint32_t(*)[32]>(&orow[c0]));
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&bars[C::B_PREADY + (SINGLE ? sb : (uint32_t)t)]);  // PV of this block may now overwrite O
          store_o(orow);
        } else {
          tc_fence_before();
          mbar_arrive(&bars[C::B_PREADY + (SINGLE ? sb : (uint32_t)t)]);
        }
        ++jh;
      }
      if (!ok) break;
      // defer this unit's epilogue (its O stays in TMEM until the next unit's
      // first P is written); keep what it needs and release the ring slot
      sts_b32x4(sepi, __float_as_uint(l_run), __float_as_uint(m_run),
                (uint32_t)(hdr_at(us, UH_B) * p.H_q + hdr_at(us, UH_H0) + t), (uint32_t)q0);
      pend = true;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_UEMPTY + us]);
    }
  }

  // the staging slots stay valid until the TMA stores have read them
  if (warp < 8 && lane == 0) bulk_wait_group_read0();
  tc_fence_before();
  __syncthreads();
  FM_DEBUG_END(p.err);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tbase);
  }
}


template <int D, bool F8, bool MI = false, bool SINGLE = false>
cudaError_t launch_fwd_d(const fm_problem& P, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdParams& prm, unsigned grid, cudaStream_t s) {
  using C = FwdCfg<D, F8, MI>;
  static_assert(C::SMEM_ALLOC <= 232448, "forward shared memory exceeds an SM's 227 KB");
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd_kernel<D, F8, MI, SINGLE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  {
    KernelTimer timer(s, kTimedFwd);
    fwd_kernel<D, F8, MI, SINGLE><<<grid, 320, C::SMEM_ALLOC, s>>>(tq, tk, tv, to, prm);
  }
  count_launches(prm.order ? 2 : 1);  // [LPT order] + main kernel
  return cudaGetLastError();
}

// Library-owned scratch for fm_attn_fwd_noalloc, laid out like the forward
// workspace: the unit-order table (one int32 per Q block) and the work
// counter. Fixed size, present on every device that loads the library, shared
// by all calls on that device.
static __device__ __align__(256) int32_t g_noalloc_order[FM_NOALLOC_MAX_QBLOCKS + 64];

}  // namespace

int32_t* fwd_noalloc_scratch() {
  // Host code cannot hand g_noalloc_order to a kernel directly (that name is
  // a host-side stand-in); the device address is looked up once per device,
  // with the device current, and cached.
  static std::mutex mu;
  static int32_t* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_order) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int32_t*>(ptr);
  }
  return cached[dev];
}

// Forward workspace: the unit-order table (one int32 per queue row: a Q block
// of a batch entry, or of a (batch entry, head) with per-head masks; padded to
// 256 bytes), then the work counter (256 bytes).
static size_t order_bytes(long long rows) { return ((4 * (size_t)rows) + 255) & ~size_t(255); }
static size_t fwd_order_bytes(const fm_problem& p) {
  return order_bytes((long long)p.B * ((p.N + kTile - 1) / kTile));
}

size_t fwd_ws_bytes(const fm_problem& p) { return fwd_order_bytes(p) + 256; }
size_t fwd_heads_ws_bytes(const fm_problem& p) {
  return order_bytes((long long)p.B * p.H_q * ((p.N + kTile - 1) / kTile)) + 256;
}

// The persistent forward (d = 64, 128; bf16 or, with fp8, e4m3 Q / K / V whose
// values are the stored ones times q_scale, k_scale, v_scale).
static cudaError_t launch_fwd_persistent(const fm_problem& P, const void* q, const void* k, const void* v,
                                         const int32_t* lts, const int32_t* lte, const int32_t* uts,
                                         const int32_t* ute, const int32_t* q_off, const int32_t* q_queue, void* o,
                                         float* lse, void* ws, cudaStream_t s, int* err, bool fp8, float q_scale,
                                         float k_scale, float v_scale, bool per_head = false, int M = 0) {
  const int nQ = (P.N + kTile - 1) / kTile;
  const int G = P.H_q / P.H_kv;
  const int PG = (G + 1) / 2;
  // per-head masks: one unit per (batch, head, Q block), in the queues' row order
  const long long units = per_head ? (long long)P.B * P.H_q * nQ : (long long)P.B * nQ * P.H_kv * PG;
  const long long rows = per_head ? (long long)P.B * P.H_q * nQ : (long long)P.B * nQ;  // queue rows
  if (units > INT_MAX) return cudaErrorInvalidConfiguration;
  // unit order: longest queue first, or natural order for long passes
  // (units that run together then share K / V tiles in L2)
  const bool natural = use_natural_order(units);
  int32_t* order = natural ? nullptr : static_cast<int32_t*>(ws);
  int* next_unit = reinterpret_cast<int*>(static_cast<char*>(ws) + order_bytes(rows));
  {
    cudaError_t e = cudaMemsetAsync(next_unit, 0, sizeof(int), s);
    if (e != cudaSuccess) return e;
  }
  if (!natural) lpt_order_kernel<<<1, 1024, 0, s>>>(q_off, (int)rows, order);
  CUtensorMap tq, tk, tv, to;
  const int Nk = kv_rows(P);
  if (fp8) {
    if (!make_tmap_u8_bhnd(&tq, q, (int64_t)P.B * P.H_q, P.N, P.d) ||
        !make_tmap_u8_bhnd(&tk, k, (int64_t)P.B * P.H_kv, Nk, P.d) ||
        !make_tmap_u8_bhnd(&tv, v, (int64_t)P.B * P.H_kv, Nk, P.d))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_bhnd(&tq, q, (int64_t)P.B * P.H_q, P.N, P.d) ||
             !make_tmap_bhnd(&tk, k, (int64_t)P.B * P.H_kv, Nk, P.d) ||
             !make_tmap_bhnd(&tv, v, (int64_t)P.B * P.H_kv, Nk, P.d)) {
    return cudaErrorInvalidValue;
  }
  if (!make_tmap_bhnd_w32(&to, o, (int64_t)P.B * P.H_q, P.N, P.d)) return cudaErrorInvalidValue;
  FwdParams prm;
  prm.lts = lts;
  prm.lte = lte;
  prm.uts = uts;
  prm.ute = ute;
  prm.q_off = q_off;
  prm.q_queue = q_queue;
  prm.order = order;
  prm.next_unit = next_unit;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.B = P.B;
  prm.H_q = P.H_q;
  prm.H_kv = P.H_kv;
  prm.N = P.N;
  prm.Nk = Nk;
  prm.nQ = nQ;
  prm.nK = (Nk + kTile - 1) / kTile;
  prm.G = G;
  prm.PG = PG;
  prm.causal = P.causal ? 1 : 0;
  prm.units = (int)units;
  prm.per_head = per_head ? 1 : 0;
  prm.M = M;
  prm.scale_log2 = P.scale * q_scale * k_scale * 1.4426950408889634f;
  prm.o_scale = v_scale;
  prm.err = err;
  // persistent: one CTA per SM (the kernel's shared memory and TMEM fill an SM)
  const unsigned grid = (unsigned)std::min<long long>(units, (long long)sm_count());
  if (per_head || G < 2) {
    // every unit has one head: the instantiation that double-buffers S
    if (fp8) return launch_fwd_d<128, true, false, true>(P, tq, tk, tv, to, prm, grid, s);
    if (M > 0) {
      if (P.d == 128) return launch_fwd_d<128, false, true, true>(P, tq, tk, tv, to, prm, grid, s);
      return launch_fwd_d<64, false, true, true>(P, tq, tk, tv, to, prm, grid, s);
    }
    if (P.d == 128) return launch_fwd_d<128, false, false, true>(P, tq, tk, tv, to, prm, grid, s);
    return launch_fwd_d<64, false, false, true>(P, tq, tk, tv, to, prm, grid, s);
  }
  if (fp8) return launch_fwd_d<128, true>(P, tq, tk, tv, to, prm, grid, s);
  if (M > 0) {
    if (P.d == 128) return launch_fwd_d<128, false, true>(P, tq, tk, tv, to, prm, grid, s);
    return launch_fwd_d<64, false, true>(P, tq, tk, tv, to, prm, grid, s);
  }
  if (P.d == 128) return launch_fwd_d<128, false>(P, tq, tk, tv, to, prm, grid, s);
  return launch_fwd_d<64, false>(P, tq, tk, tv, to, prm, grid, s);
}

cudaError_t launch_fwd(const fm_problem& P, const void* q, const void* k, const void* v, const int32_t* lts,
                       const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                       const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err) {
  if (P.d == 256) return launch_fwd256(P, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws, s, err);
  return launch_fwd_persistent(P, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws, s, err, false, 1.f, 1.f,
                               1.f);
}

cudaError_t launch_fwd_heads(const fm_problem& P, const void* q, const void* k, const void* v, const int32_t* lts,
                             const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                             const int32_t* q_queue, void* o, float* lse, void* ws, cudaStream_t s, int* err) {
  if (P.d == 256) return launch_fwd256(P, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws, s, err, true);
  return launch_fwd_persistent(P, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws, s, err, false, 1.f, 1.f,
                               1.f, true);
}

cudaError_t launch_fwd_multi(const fm_problem& P, int M, const void* q, const void* k, const void* v,
                             const int32_t* fms, const int32_t* fme, const int32_t* q_off, const int32_t* q_queue,
                             void* o, float* lse, void* ws, cudaStream_t s, int* err) {
  if (P.d == 256)
    return launch_fwd256(P, q, k, v, fms, fme, nullptr, nullptr, q_off, q_queue, o, lse, ws, s, err, false, M);
  return launch_fwd_persistent(P, q, k, v, fms, fme, nullptr, nullptr, q_off, q_queue, o, lse, ws, s, err, false,
                               1.f, 1.f, 1.f, false, M);
}

cudaError_t launch_fwd_fp8(const fm_problem& P, const void* q, const void* k, const void* v, float q_scale,
                           float k_scale, float v_scale, const int32_t* lts, const int32_t* lte, const int32_t* uts,
                           const int32_t* ute, const int32_t* q_off, const int32_t* q_queue, void* o, float* lse,
                           void* ws, cudaStream_t s, int* err) {
  return launch_fwd_persistent(P, q, k, v, lts, lte, uts, ute, q_off, q_queue, o, lse, ws, s, err, true, q_scale,
                               k_scale, v_scale);
}

}  // namespace fm
