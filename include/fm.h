/* fm.h — C ABI of the GB300 (sm_103a) FlashMask column-wise masked attention library.
 *
 * The library computes exact scaled-dot-product attention, forward and backward,
 * under the FlashMask column-wise mask (FlashMask-3 project page, "Overview"):
 * for key column j the masked query rows are the half-open intervals
 * [LTS_j, LTE_j) and [UTS_j, UTE_j), plus rows i < j when causal is set.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless a comment says otherwise.
 *     The caller allocates and owns all memory, including workspaces sized by
 *     the *_workspace_bytes queries; the library never allocates or frees.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every compute entry point only enqueues work on that stream and returns;
 *     it never synchronizes, except fm_device_status.
 *   - Layouts: Q, O, dO, dQ are contiguous (B, H_q, N, d) bf16; K, V, dK, dV are
 *     contiguous (B, H_kv, N_kv, d) bf16 (N_kv = N unless fm_problem says
 *     otherwise); LSE is (B, H_q, N) fp32; the four mask vectors are (B, N_kv)
 *     int32, one entry per key column, shared by every head (the *_heads entry
 *     points take one set per query head, (B, H_q, N_kv); the *_multi ones
 *     take visible intervals instead), holding query-row boundaries in [0, N].
 *     Tensor base addresses must be 16-byte aligned.
 *   - GQA: query head h reads kv head h / (H_q / H_kv) (contiguous groups).
 *   - Errors: arguments are validated on the host and a bad call returns an
 *     error status without launching anything. Problems found on the device
 *     (a mask value outside [0, N], a bounded wait that expired) never trap:
 *     they set bits in a device error word that fm_device_status reads.
 */
#ifndef FM_H_
#define FM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: adds the per-head (fm_attn_*_heads) and multi-interval (fm_attn_*_multi)
 * entry points; the earlier ones are unchanged. */
#define FM_ABI_VERSION 3

typedef enum fm_status {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misaligned tensor */
  FM_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. a head dim without a kernel) */
  FM_ERR_WORKSPACE = 3,   /* workspace pointer null or smaller than required */
  FM_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
  FM_ERR_TIMEOUT = 5,     /* device error word: a bounded on-device wait expired */
  FM_ERR_DEVICE = 6       /* device error word: bad mask values or queue entries */
} fm_status;

/* Device error word bits (fm_device_status). */
#define FM_DEVERR_TIMEOUT 1
#define FM_DEVERR_RANGE 2
#define FM_DEVERR_QUEUE 4
#define FM_DEVERR_DEBUG 8 /* debug build only: a range check on a shared-memory / TMEM address or TMA coordinate failed */

/* Problem shape. N query rows against N_kv key / value rows; N_kv = 0 means
 * N_kv = N (the square problem). A rectangular problem is what one rank of a
 * context-parallel split computes: its own query rows against every key, with
 * the mask vectors localized to its rows (fm_localize). scale multiplies q.k
 * (usually 1/sqrt(d)); causal != 0 adds i < j with i and j counted in the
 * problem's own rows and keys (a split that needs the global diagonal folds it
 * into the vectors instead: UTS_j = 0, UTE_j = j before localizing). */
typedef struct fm_problem {
  int32_t B, H_q, H_kv, N, d;
  float scale;
  int32_t causal;
  int32_t N_kv;
} fm_problem;

/* Tile geometry for classification: block_m query rows x block_n key columns.
 * Each must be one of 32, 64, 128, 256. The attention kernels need the tiling
 * returned by fm_attn_tiling. */
typedef struct fm_tiling {
  int32_t block_m, block_n;
} fm_tiling;

/* ABI version (FM_ABI_VERSION of the built library). */
int32_t fm_abi_version(void);

/* Static, human-readable name of a status code. */
const char* fm_status_string(fm_status s);

/* The tiling the attention kernels were built for (128 x 128). */
fm_status fm_attn_tiling(fm_tiling* out);

/* Number of Q blocks ceil(N / block_m) and KV blocks ceil(N_kv / block_n). */
fm_status fm_tile_counts(const fm_problem* p, const fm_tiling* t, int32_t* n_qblocks, int32_t* n_kblocks);

/* ---------------------------------------------------------------------------
 * Tile classification and queue construction.
 *
 * FlashMask-3 project page, §3.1 ("A third warp role that reads the mask"):
 * block-wise min/max of the boundary vectors classify every (Q-block, KV-block)
 * tile as fully-masked (skipped), partial (masked element-wise) or unmasked,
 * and each Q block gets a queue of its valid KV blocks tagged partial or
 * unmasked, visited right to left. The rule, for tile rows [q0, q1) and key
 * columns [k0, k1) (the last block of an axis may be short when N or N_kv is
 * not a multiple of the tile):
 *   skip     iff (q0 >= max LTS and q1 <= min LTE) or (q0 >= max UTS and q1 <= min UTE)
 *                or (causal and q1 <= k0)
 *   unmasked iff (q1 <= min LTS or q0 >= max LTE) and (q1 <= min UTS or q0 >= max UTE)
 *                and (not causal or q0 >= k1 - 1)
 *   partial  otherwise.
 * With LTE = N and UTS = 0 this is exactly the printed rule plus the causal term.
 *
 * Outputs (device, caller-allocated):
 *   tile_class  (B, nQ, nK) uint8: 0 = skip, 1 = partial, 2 = unmasked.
 *   q_off       B*nQ + 1 int32: CSR offsets; row (b, qb) is entry b*nQ + qb.
 *   q_queue     capacity B*nQ*nK int32: for each row, the non-skipped KV blocks in
 *               DESCENDING kb order, entry = (kb << 1) | is_partial.
 *   k_off       B*nK + 1 int32; k_queue capacity B*nQ*nK int32: for each (b, kb),
 *               the non-skipped Q blocks in ASCENDING qb order, entry =
 *               (qb << 1) | is_partial (the backward pass walks these).
 * Mask values outside [0, N] (N = query rows) are clamped for classification and flagged
 * (FM_DEVERR_RANGE). Workspace: fm_classify_workspace_bytes.
 * ------------------------------------------------------------------------- */
size_t fm_classify_workspace_bytes(const fm_problem* p, const fm_tiling* t);
fm_status fm_classify_tiles(const fm_problem* p, const fm_tiling* t, const int32_t* lts, const int32_t* lte,
                            const int32_t* uts, const int32_t* ute, uint8_t* tile_class, int32_t* q_off,
                            int32_t* q_queue, int32_t* k_off, int32_t* k_queue, void* ws, size_t ws_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------
 * Forward: O = softmax(scale * Q K^T + M) V and LSE = log sum_j exp(scale q.k_j)
 * over visible j (natural log), where M is 0 or -inf from the mask.
 *
 * FlashMask-3 project page, §3.1 (KV Loader: loads only queued KV blocks;
 * MMA Consumer: score, softmax and output, row-interval mask applied only on
 * partial blocks); the online-softmax recurrence (running max m and sum l,
 * rescaling O) is the one in "Flash MSA Attention Kernel Implementation",
 * "The Flash Core: Tiling Over the Memory Hierarchy".
 * A query row with no visible key gets O = 0 and LSE = -inf.
 *
 * q_off / q_queue must come from fm_classify_tiles with the fm_attn_tiling
 * tiling and the same problem and mask. d must be 64, 128 or 256 (256: the
 * FlashMask Guide's usage example, "Complete PyTorch Implementation",
 * dim = 256). Mask values
 * outside [0, N] are clamped; the forward does not flag them again
 * (fm_classify_tiles on the same vectors does).
 * Workspace: fm_attn_fwd_workspace_bytes (the unit-order table and a work
 * counter; every call rewrites what it uses, so it needs no clearing).
 * ------------------------------------------------------------------------- */
size_t fm_attn_fwd_workspace_bytes(const fm_problem* p);
fm_status fm_attn_fwd(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                      const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                      const int32_t* q_queue, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 forward: the same computation as fm_attn_fwd on e4m3 inputs
 * ("Flash MSA Attention Kernel Implementation", "Optimization Tricks That
 * Actually Matter": FP8 matrix products inside the tile, softmax in FP32).
 *
 * q, k, v hold e4m3 (OCP E4M3, finite range +-448) values, contiguous
 * (B, H, N, d) one byte per element; the attention inputs they stand for are
 * stored value x q_scale (k_scale, v_scale), scales finite and > 0.
 * S = Q K^T runs on e4m3 operands with fp32 accumulation (exact products);
 * the softmax, running max and sums are fp32; P is rounded to e4m3 for
 * O = P V (fp32 accumulation); O is bf16, LSE fp32, in the units of fm_attn_fwd.
 * P's rounding (3 mantissa bits) puts O about 2.5% (relative L2) from the
 * exact attention of the dequantized inputs; LSE is not affected.
 * d must be 128. Queues, mask vectors, workspace: as fm_attn_fwd. There is no
 * FP8 backward.
 * ------------------------------------------------------------------------- */
fm_status fm_attn_fwd_fp8(const fm_problem* p, const void* q, const void* k, const void* v, float q_scale,
                          float k_scale, float v_scale, const int32_t* lts, const int32_t* lte, const int32_t* uts,
                          const int32_t* ute, const int32_t* q_off, const int32_t* q_queue, void* o, float* lse,
                          void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Backward: given dO, the gradients of sum(O * dO):
 *   P = exp(scale S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
 *   dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q,
 * recomputing P from LSE ("Flash MSA Attention Kernel Implementation",
 * "The Backward Pass: The Real Beast"), skipping the same fully-masked tiles
 * and masking only partial tiles. dK and dV are summed over the query heads
 * of each GQA group. Rows with LSE = -inf contribute nothing.
 *
 * o and lse must be the forward outputs for the same inputs. k_off / k_queue
 * come from fm_classify_tiles with the fm_attn_tiling tiling. d must be 64,
 * 128 or 256.
 * Workspace: fm_attn_bwd_workspace_bytes (fp32 dQ accumulator, row terms D).
 * ------------------------------------------------------------------------- */
size_t fm_attn_bwd_workspace_bytes(const fm_problem* p);
fm_status fm_attn_bwd(const fm_problem* p, const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, const int32_t* lts, const int32_t* lte,
                      const int32_t* uts, const int32_t* ute, const int32_t* k_off, const int32_t* k_queue,
                      void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Per-head mask vectors: one set of four vectors per query head, lts..ute
 * (B, H_q, N_kv) int32 (the FlashMask Guide's operator takes its vectors per
 * sample; a mask that differs by head is the same representation one level
 * finer). Everything else is fm_attn_fwd / fm_attn_bwd, except:
 *   - the queues come from fm_classify_tiles run on the vectors as B * H_q
 *     rows (an fm_problem with B' = B * H_q), so row (b * H_q + h) holds
 *     query head h's tiles;
 *   - every work unit is one head (two heads of a unit would need one queue);
 *   - d is 64, 128 or 256 like fm_attn_fwd, and H_q / H_kv is at most 64
 *     (FM_ERR_UNSUPPORTED otherwise).
 * Workspaces: fm_attn_fwd_heads_workspace_bytes (one order entry per queue
 * row) and fm_attn_bwd_workspace_bytes.
 * ------------------------------------------------------------------------- */
size_t fm_attn_fwd_heads_workspace_bytes(const fm_problem* p);
fm_status fm_attn_fwd_heads(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                            const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                            const int32_t* q_queue, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);
fm_status fm_attn_bwd_heads(const fm_problem* p, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, const int32_t* lts, const int32_t* lte,
                            const int32_t* uts, const int32_t* ute, const int32_t* k_off, const int32_t* k_queue,
                            void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Multi-interval masks (the FlashMask Guide, "The Solution: FlashMask Sparse
 * Mask Representation": up to four visible intervals per key column). Key
 * column j is visible to query row i iff FMS_m,j <= i <= FME_m,j for some
 * interval m (inclusive bounds; an interval with FMS > FME is empty;
 * intervals may overlap), and, with causal set, i >= j. fms, fme are
 * (M, B, N_kv) int32 device arrays, 1 <= M <= 4.
 *
 * fm_classify_tiles_multi first rewrites each column's visible rows as their
 * maximal runs (intervals clipped to [0, N), sorted by start, joined where
 * they overlap or touch; run k in slot k, the other slots empty, written
 * start N and end -1), so the classes depend on the mask only, then gives
 * every tile the most visible of the slots' own classes (the rule of fm_classify_tiles on each slot's masked
 * complement, [0, start) and (end, N), with the causal term): skipped iff no
 * run reaches the tile, unmasked iff one run alone covers it, partial
 * otherwise; its outputs have the layout of fm_classify_tiles for B batch
 * entries. Workspace: fm_classify_multi_workspace_bytes.
 *
 * fm_attn_fwd_multi / fm_attn_bwd_multi are fm_attn_fwd / fm_attn_bwd with
 * these queues: each queued block is computed once, its partial tiles masked
 * by the union of the intervals (rows outside every interval masked).
 * Workspaces: fm_attn_fwd_workspace_bytes, fm_attn_bwd_workspace_bytes.
 * Errors: M outside [1, 4] is FM_ERR_INVALID_ARG; the rest as fm_attn_fwd /
 * fm_attn_bwd.
 * ------------------------------------------------------------------------- */
size_t fm_classify_multi_workspace_bytes(const fm_problem* p, const fm_tiling* t, int32_t M);
fm_status fm_classify_tiles_multi(const fm_problem* p, const fm_tiling* t, int32_t M, const int32_t* fms,
                                  const int32_t* fme, uint8_t* tile_class, int32_t* q_off, int32_t* q_queue,
                                  int32_t* k_off, int32_t* k_queue, void* ws, size_t ws_bytes, void* stream);
fm_status fm_attn_fwd_multi(const fm_problem* p, int32_t M, const void* q, const void* k, const void* v,
                            const int32_t* fms, const int32_t* fme, const int32_t* q_off, const int32_t* q_queue,
                            void* o, float* lse, void* ws, size_t ws_bytes, void* stream);
fm_status fm_attn_bwd_multi(const fm_problem* p, int32_t M, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, const int32_t* fms,
                            const int32_t* fme, const int32_t* k_off, const int32_t* k_queue, void* dq, void* dk,
                            void* dv, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * One forward + backward from HOST buffers. (No counterpart in the pages: an
 * end-to-end convenience over the calls above.)
 *
 * q, k, v, dout, the four mask vectors, and the outputs o, lse, dq, dk, dv are
 * HOST pointers with the layouts above (page-locked memory lets the copies run
 * asynchronously and overlap other work; pageable memory works but each copy
 * then blocks the calling thread). On `stream`, in order: one host-to-device
 * copy per input into the device workspace, fm_classify_tiles (attention
 * tiling), fm_attn_fwd, fm_attn_bwd, one device-to-host copy per output. The
 * call returns once everything is enqueued; synchronize the stream before
 * reading the outputs. ws: DEVICE memory of fm_attn_host_workspace_bytes(p)
 * bytes (the device copies of inputs and outputs, the queues and the kernels'
 * workspaces), owned by the caller; two calls in flight need two workspaces.
 * Errors: as the calls it makes; FM_ERR_CUDA when a copy cannot be enqueued.
 * ------------------------------------------------------------------------- */
size_t fm_attn_host_workspace_bytes(const fm_problem* p);
fm_status fm_attn_fwd_bwd_host(const fm_problem* p, const void* q, const void* k, const void* v, const void* dout,
                               const int32_t* lts, const int32_t* lte, const int32_t* uts, const int32_t* ute,
                               void* o, float* lse, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                               void* stream);

/* ---------------------------------------------------------------------------
 * Forward without a caller-provided workspace. (No counterpart in the pages:
 * this is a convenience of the library, not part of the method.)
 *
 * Same computation, arguments and results as fm_attn_fwd, minus ws/ws_bytes.
 * It is meant for callers that cannot allocate device memory at call time:
 * for example a plugin inside a host framework that owns all device memory and
 * gives its plugins no allocator, or a service that reserves its memory once
 * at start-up and must not call cudaMalloc afterwards. Nothing here calls
 * cudaMalloc, cudaFree or any allocating library routine.
 *
 * The forward's only scratch (its unit-order table, one int32 per Q block, and
 * a work counter) lives instead in a fixed array inside the library,
 * FM_NOALLOC_MAX_QBLOCKS + 64 entries (256 KiB + 256 B) per GPU, held by every
 * GPU that loads the library until the process exits. Problems with B * ceil(N / 128) > FM_NOALLOC_MAX_QBLOCKS are
 * rejected with FM_ERR_WORKSPACE before anything is launched.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.
 * All calls on a device share the one array: calls that can overlap on the GPU
 * (different streams without ordering between them) race on it and must be
 * serialized by the caller. Every call rewrites the entries it uses, so nothing
 * needs clearing between calls.
 * ------------------------------------------------------------------------- */
#define FM_NOALLOC_MAX_QBLOCKS 65536
fm_status fm_attn_fwd_noalloc(const fm_problem* p, const void* q, const void* k, const void* v, const int32_t* lts,
                              const int32_t* lte, const int32_t* uts, const int32_t* ute, const int32_t* q_off,
                              const int32_t* q_queue, void* o, float* lse, void* stream);

/* ---------------------------------------------------------------------------
 * Zero-communication mask localization (FlashMask-3 project page, §3.2):
 *   x_local = max_i [ clip(x - O_i, 0, C) + i*C*1(clip(x - O_i, 0, C) > 0) ]
 * = the number of the rank's rows before global row x, for a rank that owns
 * kappa chunks of C rows starting at global rows chunk_off[0] < chunk_off[1] < ...
 * x_global: n device int32 values (any of the four boundary vectors, any
 * number of them concatenated); chunk_off: kappa device int32 offsets, ascending,
 * 1 <= kappa <= 4096; x_local: n device int32 outputs. C >= 1.
 * ------------------------------------------------------------------------- */
fm_status fm_localize(const int32_t* x_global, int64_t n, const int32_t* chunk_off, int32_t kappa, int32_t C,
                      int32_t* x_local, void* stream);

/* ---------------------------------------------------------------------------
 * The FlashMask Guide's representation ("The Solution: FlashMask Sparse Mask
 * Representation", "Column-Wise Sparse Representation"): key column j is
 * visible exactly to query rows FMS_j <= i <= FME_j (inclusive, one interval;
 * causality is written into FMS, e.g. FMS_j = j). fm_from_fms_fme writes the
 * equivalent four vectors for use with causal = 0: the masked rows [0, FMS_j)
 * and [FME_j + 1, N) become UTS = 0, UTE = clip(FMS), LTS = clip(FME + 1),
 * LTE = N, clipped to [0, N]; FMS_j > FME_j masks the whole column. fms, fme
 * and the four outputs are n_values device int32 values each (any (B, N_kv)
 * layout); N is the number of query rows. Output buffers must not overlap the
 * inputs.
 * ------------------------------------------------------------------------- */
fm_status fm_from_fms_fme(const int32_t* fms, const int32_t* fme, int64_t n_values, int32_t N, int32_t* lts,
                          int32_t* lte, int32_t* uts, int32_t* ute, void* stream);

/* ---------------------------------------------------------------------------
 * Multi-interval masks (FlashMask Guide, after the DPO example: a key column
 * may be visible to up to M disjoint row intervals [FMS^(m)_j, FME^(m)_j]).
 * For one query row the keys visible through different intervals are then
 * disjoint sets, so attention over their union is the log-sum-exp merge of
 * one single-interval attention per interval (fm_from_fms_fme, classify,
 * forward on each), and its gradients are the sums of the parts' backward
 * passes run with the MERGED O and LSE.
 *
 * fm_merge_parts: M (1..8) parts, O_m (rows x d bf16) and LSE_m (rows fp32);
 *   o_parts / lse_parts are HOST arrays of M DEVICE pointers. Writes
 *   LSE = log sum_m exp(LSE_m) and O = sum_m exp(LSE_m - LSE) O_m (bf16,
 *   rounded once), or LSE = -inf and O = 0 where every part is -inf.
 *   rows = B * H_q * N; d a multiple of 8; O pointers 16-byte aligned.
 * fm_sum_parts: out = sum_m parts[m] over n bf16 elements (fp32 sum, rounded
 *   once); parts is a HOST array of M DEVICE pointers.
 * Outputs must not overlap the inputs.
 * ------------------------------------------------------------------------- */
fm_status fm_merge_parts(int32_t M, const void* const* o_parts, const float* const* lse_parts, int64_t rows,
                         int32_t d, void* o, float* lse, void* stream);
fm_status fm_sum_parts(int32_t M, const void* const* parts, int64_t n, void* out, void* stream);

/* ---------------------------------------------------------------------------
 * Sparsity-aware chunk balancing for context parallelism (FlashMask-3 project
 * page, §3.3 "Balance the work, not the length"). HOST functions: every
 * pointer in this section is a host pointer, nothing touches a GPU, and the
 * calls are synchronous and thread-safe (no shared state).
 *
 * The query axis of a problem is cut into chunks of blocks_per_chunk Q blocks;
 * with n = P * kappa chunks, each of P ranks receives exactly kappa of them.
 *
 * fm_chunk_loads: the tile cost model {0, alpha_p, alpha_u}. tile_class is the
 *   (B, nQ, nK) uint8 output of fm_classify_tiles copied to the host; a tile
 *   of class 1 (partial) costs cost_partial, class 2 (unmasked) costs
 *   cost_unmasked, anything else 0. Chunk c holds Q blocks
 *   [c * blocks_per_chunk, (c + 1) * blocks_per_chunk) of every batch entry
 *   (the last chunk may be short); w[c] (ceil(nQ / blocks_per_chunk) int64
 *   outputs) is the sum of its tiles' costs. Costs must be >= 0.
 *
 * fm_balance_chunks: Stage 1 of HCC-IPO on loads w[0..n_chunks): LPT under the
 *   cardinality constraint, then exact pairwise repartition (phases >= 2),
 *   then exact three-rank repartition (phases == 3); owner[i] (n_chunks int32
 *   outputs) is the rank of chunk i. The pages' lower bound LB =
 *   max(ceil(sum w / P), max w) and a stronger one that also uses the
 *   cardinality constraint, LB_kappa >= LB (a pigeonhole bound, defined in
 *   csrc/fm_balance.cpp), certify the result optimal when the makespan
 *   reaches LB_kappa; every phase stops there. Exact
 *   rules (tie-breaking, the order groups are visited in): the header of
 *   csrc/fm_balance.cpp. node_budget caps the branch-and-bound nodes of one
 *   group's repartition (<= 0: 4,000,000); a group whose search exceeds it is
 *   left unchanged and report->budget_exhausted is set. Requires
 *   n_chunks == P * kappa, w[i] >= 0, 2 * kappa <= 64 when the pairwise phase
 *   runs and 3 * kappa <= 64 when the three-rank phase runs
 *   (FM_ERR_UNSUPPORTED otherwise). report may be NULL.
 * ------------------------------------------------------------------------- */
typedef struct fm_balance_report {
  int64_t lower_bound;   /* LB = max(ceil(sum w / P), max w) */
  int64_t lower_bound_kappa; /* LB_kappa >= LB, which also uses kappa chunks per rank */
  int64_t makespan_lpt;  /* max rank load after LPT */
  int64_t makespan_pair; /* after the pairwise phase (= makespan_lpt when it does not run) */
  int64_t makespan;      /* final max rank load */
  int32_t certified;     /* makespan == lower_bound_kappa: the assignment is optimal */
  int32_t pair_moves;    /* pairwise repartitions applied */
  int32_t triple_moves;  /* three-rank repartitions applied */
  int32_t budget_exhausted;
} fm_balance_report;

fm_status fm_chunk_loads(const uint8_t* tile_class, int32_t B, int32_t nQ, int32_t nK, int32_t blocks_per_chunk,
                         int64_t cost_partial, int64_t cost_unmasked, int64_t* w);
fm_status fm_balance_chunks(const int64_t* w, int32_t n_chunks, int32_t P, int32_t kappa, int32_t phases,
                            int64_t node_budget, int32_t* owner, fm_balance_report* report);

/* Mask-aware pruning of the K / V exchange (FlashMask-3 project page, §3.4: a
 * chunk the mask fully hides is never sent). HOST function. Chunks cut both
 * axes alike (blocks_per_chunk Q blocks and as many KV blocks); owner[c] in
 * [0, P) is chunk c's rank. need (P x n_chunks uint8, row-major) gets 1 where
 * some tile between rank r's query blocks and chunk c's key blocks, in any
 * batch entry of tile_class (B, nQ, nK; fm_classify_tiles classes), is not
 * skipped: rank r needs chunk c's K / V rows, and only those. */
fm_status fm_needed_chunks(const uint8_t* tile_class, int32_t B, int32_t nQ, int32_t nK, const int32_t* owner,
                           int32_t n_chunks, int32_t P, int32_t blocks_per_chunk, uint8_t* need);

/* ---------------------------------------------------------------------------
 * Device error word. Synchronizes `stream`, returns the accumulated FM_DEVERR_*
 * bits in *bits (may be NULL) and clears them. Status: FM_OK when no bit is
 * set, FM_ERR_TIMEOUT when FM_DEVERR_TIMEOUT is set, else FM_ERR_DEVICE.
 * The word is per device and shared by all streams of the process.
 * ------------------------------------------------------------------------- */
fm_status fm_device_status(void* stream, int32_t* bits);

/* Self-test of the bounded device wait: launches one CTA that waits on an
 * mbarrier no one arrives at, with a limit of limit_us microseconds
 * (1 .. 10,000,000). The wait expires, the kernel sets FM_DEVERR_TIMEOUT and
 * returns normally; the context stays usable. Used by the tests to check the
 * timeout path without hanging or faulting the GPU. */
fm_status fm_selftest_wait_timeout(int64_t limit_us, void* stream);

/* ---------------------------------------------------------------------------
 * Measurement hooks (no effect on results).
 *
 * fm_profile_enable(1): from now on every launch of the forward main kernel
 * (kind 0) and of the backward main kernel (kind 1) is bracketed by a pair of
 * CUDA events recorded on its launch stream. fm_profile_enable(0) stops it.
 * fm_profile_read synchronizes on the recorded events and returns, per kind,
 * the summed device milliseconds and the number of launches since the last
 * read, then clears the record. Pointers may be NULL. Host-thread safe.
 *
 * fm_launch_count: total number of kernels this library has launched in the
 * process (every compute entry point counts each kernel it enqueues).
 * ------------------------------------------------------------------------- */
fm_status fm_profile_enable(int32_t on);
fm_status fm_profile_read(double* fwd_ms, int32_t* fwd_launches, double* bwd_ms, int32_t* bwd_launches);
int64_t fm_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* FM_H_ */
