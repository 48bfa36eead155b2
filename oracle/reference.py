"""CPU fp64 oracle for FlashMask column-wise masked attention.

TEST INFRASTRUCTURE. Only the tests, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg import this module; the library's product path
never calls it, and it shares no code with the CUDA kernels. It is plain,
slow and written straight from the definitions:

* the mask comes from the four column-wise boundary vectors
  (FlashMask-3 project page, "Overview" and §3.1): element (i, j) is masked iff
  LTS_j <= i < LTE_j or UTS_j <= i < UTE_j, plus i < j in causal mode;
* attention is softmax(scale * Q K^T + M) V with M in {0, -inf}
  (FlashMask Guide, §2 "The O(N^2) Memory Explosion of Dense Mask Matrices",
  the equation S = QK^T/sqrt(d_k) + M);
* gradients are the analytic ones of that expression (Flash MSA Attention
  Kernel Implementation, "The Backward Pass": dV = P^T dO, dP = dO V^T,
  dS = P * (dP - rowsum(P * dP)), dQ = dS K, dK = dS^T Q, each scaled);
* tiles are classified from block-wise min/max of the vectors (FlashMask-3
  project page, §3.1, the tile rule under the 64 x 64 / 8 x 8 figure),
  generalised to intervals that do not reach the sequence edge;
* localization is the clip-shift-max map of FlashMask-3 project page, §3.2;
* the FlashMask Guide's FMS / FME vectors (one inclusive visible interval per
  key column) map onto the four vectors as the complement of that interval;
  its multi-interval masks (up to M visible intervals per key column) are
  evaluated directly (`multi_masked_rows`), and their tiles are classified on
  each column's visible set written as its maximal runs of rows
  (`union_runs`).

Readings where the pages are silent (pinned by tests/test_oracle.py,
tests/test_cp_oracle.py and tests/test_convert_oracle.py):
  - intervals are half-open row ranges; start >= end is an empty interval;
  - causal masks i < j (the diagonal is visible);
  - a fully-masked query row has O = 0 and LSE = -inf and contributes no
    gradient; LSE is the natural log of sum_j exp(scale * q_i . k_j) over
    visible j;
  - GQA groups are contiguous: query head h uses kv head h // (H_q / H_kv);
  - the vectors are (B, N_kv), one entry per key column, shared by every head;
    the query rows may number N != N_kv (one rank of a context-parallel split:
    its own rows against every key, FlashMask-3 project page, §3.2), with
    causal comparing the problem's own row and key indices;
  - a mask may also be given per query head ({"heads": four (B, H_q, N_kv)
    arrays}) or as multi-interval vectors ({"fms", "fme"}: (B, M, N_kv)).

Precision: every input is widened to float64; all arithmetic is float64.
"""
from __future__ import annotations

import numpy as np

SKIP, PARTIAL, UNMASKED = 0, 1, 2


# ------------------------------------------------------------------ mask
def masked_rows(lts, lte, uts, ute, causal: bool, rows) -> np.ndarray:
    """Rows of the dense mask: True where (i, j) is masked, shape (len(rows), N).

    lts..ute are the (N,) boundary vectors of one batch entry.
    """
    rows = np.asarray(rows, dtype=np.int64)
    n = lts.shape[0]
    i = rows[:, None]
    j = np.arange(n, dtype=np.int64)[None, :]
    lower = (lts[None, :].astype(np.int64) <= i) & (i < lte[None, :].astype(np.int64))
    upper = (uts[None, :].astype(np.int64) <= i) & (i < ute[None, :].astype(np.int64))
    m = lower | upper
    if causal:
        m = m | (i < j)
    return m


def multi_masked_rows(fms, fme, rows) -> np.ndarray:
    """Multi-interval masks (FlashMask Guide, after the DPO example: up to M
    visible intervals per key column): key j is visible to row i iff
    FMS^(m)_j <= i <= FME^(m)_j for some m. fms, fme: (M, N_kv) of one batch
    entry. True where masked, shape (len(rows), N_kv)."""
    rows = np.asarray(rows, dtype=np.int64)[:, None]
    vis = np.zeros((rows.shape[0], fms.shape[1]), dtype=bool)
    for m in range(fms.shape[0]):
        vis |= (fms[m][None, :].astype(np.int64) <= rows) & (rows <= fme[m][None, :].astype(np.int64))
    return ~vis


def _mask_rows(vec, causal, b, rows, h=0):
    """Masked rows of batch entry b (query head h) for any mask form: the four
    vectors shared by every head (a tuple of (B, N_kv) arrays), one set per
    query head ({"heads": a tuple of (B, H_q, N_kv) arrays}), or multi-interval
    ({"fms", "fme"}: (B, M, N_kv) arrays)."""
    if isinstance(vec, dict) and "heads" in vec:
        lts, lte, uts, ute = (x[b, h] for x in vec["heads"])
        return masked_rows(lts, lte, uts, ute, causal, rows)
    if isinstance(vec, dict):
        m = multi_masked_rows(vec["fms"][b], vec["fme"][b], rows)
        if causal:  # the causal term masks i < j on top of every mask form
            m = m | (np.asarray(rows, dtype=np.int64)[:, None] < np.arange(m.shape[1], dtype=np.int64)[None, :])
        return m
    lts, lte, uts, ute = (x[b] for x in vec)
    return masked_rows(lts, lte, uts, ute, causal, rows)


def dense_mask(lts, lte, uts, ute, causal: bool) -> np.ndarray:
    """The full N x N boolean mask (True = masked). Small N only."""
    return masked_rows(lts, lte, uts, ute, causal, np.arange(lts.shape[0]))


def masked_cols(lts, lte, uts, ute, causal: bool, cols, n_rows=None) -> np.ndarray:
    """Columns of the dense mask, shape (n_rows, len(cols)): True where masked
    (n_rows defaults to the number of key columns)."""
    cols = np.asarray(cols, dtype=np.int64)
    n = lts.shape[0] if n_rows is None else int(n_rows)
    i = np.arange(n, dtype=np.int64)[:, None]
    j = cols[None, :]
    lower = (lts[cols].astype(np.int64)[None, :] <= i) & (i < lte[cols].astype(np.int64)[None, :])
    upper = (uts[cols].astype(np.int64)[None, :] <= i) & (i < ute[cols].astype(np.int64)[None, :])
    m = lower | upper
    if causal:
        m = m | (i < j)
    return m


# ------------------------------------------------------- tile classes
def block_minmax(vec, bn: int):
    """Per KV block of bn columns: (min, max) of vec over the block's valid columns."""
    n = vec.shape[0]
    nk = -(-n // bn)
    mins = np.empty(nk, dtype=np.int64)
    maxs = np.empty(nk, dtype=np.int64)
    for kb in range(nk):
        blk = vec[kb * bn : min((kb + 1) * bn, n)].astype(np.int64)
        mins[kb] = blk.min()
        maxs[kb] = blk.max()
    return mins, maxs


def classify_tiles(lts, lte, uts, ute, causal: bool, bm: int, bn: int, n_rows=None) -> np.ndarray:
    """Class of every (Q-block, KV-block) tile of one batch entry: (nQ, nK) uint8
    (n_rows query rows, default: as many as key columns).

    Tile rows [q0, q1), columns [k0, k1) (the last block of each axis may be
    short). With block min/max of the four vectors:
      skip      iff (q0 >= max LTS and q1 <= min LTE)
                 or (q0 >= max UTS and q1 <= min UTE)
                 or (causal and q1 <= k0)
      unmasked  iff (q1 <= min LTS or q0 >= max LTE)
                and (q1 <= min UTS or q0 >= max UTE)
                and (not causal or q0 >= k1 - 1)
      partial   otherwise.
    With LTE = N and UTS = 0 this is exactly the printed rule (skip if
    q0 >= max LTS or q1 <= min UTE; unmasked if q1 <= min LTS and
    q0 >= max UTE) plus the causal term.
    """
    n = lts.shape[0]
    nr = n if n_rows is None else int(n_rows)
    nq, nk = -(-nr // bm), -(-n // bn)
    mn_lts, mx_lts = block_minmax(lts, bn)
    mn_lte, mx_lte = block_minmax(lte, bn)
    mn_uts, mx_uts = block_minmax(uts, bn)
    mn_ute, mx_ute = block_minmax(ute, bn)
    cls = np.empty((nq, nk), dtype=np.uint8)
    for qb in range(nq):
        q0, q1 = qb * bm, min((qb + 1) * bm, nr)
        for kb in range(nk):
            k0, k1 = kb * bn, min((kb + 1) * bn, n)
            skip = (
                (q0 >= mx_lts[kb] and q1 <= mn_lte[kb])
                or (q0 >= mx_uts[kb] and q1 <= mn_ute[kb])
                or (causal and q1 <= k0)
            )
            unmasked = (
                (q1 <= mn_lts[kb] or q0 >= mx_lte[kb])
                and (q1 <= mn_uts[kb] or q0 >= mx_ute[kb])
                and ((not causal) or q0 >= k1 - 1)
            )
            cls[qb, kb] = SKIP if skip else (UNMASKED if unmasked else PARTIAL)
    return cls


def union_runs(fms, fme, n_rows: int):
    """Each key column's visible rows under a multi-interval mask (fms, fme:
    (M, N_kv), rows FMS^(m)_j <= i <= FME^(m)_j for some m, within [0, n_rows))
    as that set's maximal runs of consecutive rows, ascending, run k in slot k:
    (starts, ends), both (M, N_kv) inclusive. A slot past the column's last run
    is empty, written start = n_rows, end = -1: its masked complement then has
    its upper interval reaching the last row and its lower one starting at row
    0, so in a tile's block bounds it neither lowers the smallest upper end nor
    raises the largest lower start of the live columns (it masks every row
    either way). Intervals are clipped to the rows, empty ones dropped, the
    rest taken in order of their start and joined where one overlaps or
    touches the run before it."""
    fms = np.asarray(fms, dtype=np.int64)
    fme = np.asarray(fme, dtype=np.int64)
    M, nk = fms.shape
    starts = np.full((M, nk), n_rows, dtype=np.int64)
    ends = np.full((M, nk), -1, dtype=np.int64)
    for j in range(nk):
        pieces = []
        for m in range(M):
            a, b = max(int(fms[m, j]), 0), min(int(fme[m, j]), n_rows - 1)
            if a <= b:
                pieces.append((a, b))
        runs = []
        for a, b in sorted(pieces):
            if runs and a <= runs[-1][1] + 1:
                runs[-1][1] = max(runs[-1][1], b)
            else:
                runs.append([a, b])
        for k, (a, b) in enumerate(runs):
            starts[k, j], ends[k, j] = a, b
    return starts, ends


def classify_tiles_multi(fms, fme, causal: bool, bm: int, bn: int, n_rows: int) -> np.ndarray:
    """Tile classes of a multi-interval mask for one batch entry (fms, fme:
    (M, N_kv), key j visible to rows FMS^(m)_j <= i <= FME^(m)_j for some m,
    plus i >= j when causal). The visible set of every column is first
    rewritten as its runs (`union_runs`: the same mask, overlapping or
    touching intervals joined); a tile's class is then the most visible of the
    run slots' own classes, each from `classify_tiles` on the slot's masked
    complement (`from_fms_fme`) with the causal term. A tile is skipped iff
    every slot skips it, unmasked iff one slot alone leaves it unmasked,
    partial otherwise (class codes 0 < 1 < 2, so the most visible is the
    maximum)."""
    starts, ends = union_runs(fms, fme, n_rows)
    cls = [classify_tiles(*from_fms_fme(starts[m], ends[m], n_rows), causal, bm, bn, n_rows=n_rows)
           for m in range(starts.shape[0])]
    return np.maximum.reduce(cls)


def build_queues(cls_batches):
    """Compacted queues in CSR form from a list of per-batch (nQ, nK) class tables.

    Q-side: for each (b, qb) in order, the non-skipped KV blocks in DESCENDING
    kb order (visited right to left), entry = (kb << 1) | is_partial.
    K-side: for each (b, kb), the non-skipped Q blocks in ASCENDING qb order,
    entry = (qb << 1) | is_partial.
    Returns (q_off, q_queue, k_off, k_queue) as int32 arrays; offsets have
    B*nQ + 1 (resp. B*nK + 1) entries.
    """
    q_off, q_queue, k_off, k_queue = [0], [], [0], []
    for cls in cls_batches:
        nq, nk = cls.shape
        for qb in range(nq):
            for kb in range(nk - 1, -1, -1):
                c = int(cls[qb, kb])
                if c != SKIP:
                    q_queue.append((kb << 1) | (1 if c == PARTIAL else 0))
            q_off.append(len(q_queue))
    for cls in cls_batches:
        nq, nk = cls.shape
        for kb in range(nk):
            for qb in range(nq):
                c = int(cls[qb, kb])
                if c != SKIP:
                    k_queue.append((qb << 1) | (1 if c == PARTIAL else 0))
            k_off.append(len(k_queue))
    as32 = lambda x: np.asarray(x, dtype=np.int32)
    return as32(q_off), as32(q_queue), as32(k_off), as32(k_queue)


# ------------------------------------------------------------- attention
def _kv_head(h: int, hq: int, hkv: int) -> int:
    return h // (hq // hkv)


def row_probs(q, k, vec, causal, scale, b, h, rows):
    """Softmax probabilities P (len(rows), N) and LSE (len(rows),) for one head.

    S = scale * q_i . k_j over all N keys, masked entries set to -inf, then
    P = exp(S - max) / sum. A fully-masked row gets P = 0 and LSE = -inf.
    q: (B, Hq, N, d), k: (B, Hkv, N_kv, d), float64.
    """
    g = _kv_head(h, q.shape[1], k.shape[1])
    m = _mask_rows(vec, causal, b, rows, h)
    s = scale * (q[b, h, rows] @ k[b, g].T)
    s = np.where(m, -np.inf, s)
    r = s.max(axis=1)
    empty = np.isneginf(r)
    r_safe = np.where(empty, 0.0, r)
    e = np.exp(s - r_safe[:, None])
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    lse = np.where(empty, -np.inf, r_safe + np.log(np.where(empty, 1.0, l)))
    return p, lse


def row_probs_visible(q, k, vec, causal, scale, b, h, rows):
    """As `row_probs`, restricted to the key columns that at least one of the
    given rows sees: returns (P over those columns, LSE, the column indices).

    Every other column is masked for every one of these rows, so its weight
    exp(-inf) = 0 contributes exactly nothing to O, LSE or any gradient; only
    the rounding order of the sums changes. This is what lets the oracle reach
    every row of the long workloads."""
    g = _kv_head(h, q.shape[1], k.shape[1])
    m = _mask_rows(vec, causal, b, rows, h)
    vc = np.nonzero(~m.all(axis=0))[0]
    s = scale * (q[b, h, rows] @ k[b, g][vc].T)
    s = np.where(m[:, vc], -np.inf, s)
    r = s.max(axis=1) if vc.size else np.full(len(rows), -np.inf)
    empty = np.isneginf(r)
    r_safe = np.where(empty, 0.0, r)
    e = np.exp(s - r_safe[:, None])
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    lse = np.where(empty, -np.inf, r_safe + np.log(np.where(empty, 1.0, l)))
    return p, lse, vc


def forward(q, k, v, vec, causal: bool, scale: float, heads=None, rows=None, row_chunk: int = 512,
            visible_only: bool = False):
    """O and LSE for the selected heads and rows.

    Returns O of shape (B, len(heads), len(rows), d) and LSE (B, len(heads), len(rows)).
    visible_only: compute each row chunk over the key columns it sees
    (`row_probs_visible`), the same result up to rounding order.
    """
    B, Hq, N, d = q.shape
    heads = list(range(Hq)) if heads is None else list(heads)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    O = np.zeros((B, len(heads), len(rows), d))
    L = np.zeros((B, len(heads), len(rows)))
    for b in range(B):
        for hi, h in enumerate(heads):
            g = _kv_head(h, Hq, k.shape[1])
            for c0 in range(0, len(rows), row_chunk):
                rr = rows[c0 : c0 + row_chunk]
                if visible_only:
                    p, lse, vc = row_probs_visible(q, k, vec, causal, scale, b, h, rr)
                    O[b, hi, c0 : c0 + len(rr)] = p @ v[b, g][vc]
                else:
                    p, lse = row_probs(q, k, vec, causal, scale, b, h, rr)
                    O[b, hi, c0 : c0 + len(rr)] = p @ v[b, g]
                L[b, hi, c0 : c0 + len(rr)] = lse
    return O, L


def backward(q, k, v, do, vec, causal: bool, scale: float, heads=None, rows=None, cols=None, row_chunk=256,
             visible_only: bool = False):
    """Analytic gradients of sum(O * dO).

    dQ is returned for the selected `rows` of the selected `heads`:
    shape (B, len(heads), len(rows), d).
    dK, dV are returned for the selected key `cols` of every kv head,
    summed over the selected query heads only (so a head subset gives the
    gradient of that subset): shape (B, Hkv, len(cols), d).
    Per row i (one query head): P from `row_probs`; dP_ij = dO_i . v_j;
    D_i = sum_j P_ij dP_ij; dS_ij = P_ij (dP_ij - D_i);
    dQ_i = scale sum_j dS_ij k_j; dV_j += P_ij dO_i; dK_j += scale dS_ij q_i.
    visible_only: each row chunk over the key columns it sees
    (`row_probs_visible`); P = dS = 0 on the others.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    heads = list(range(Hq)) if heads is None else list(heads)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    cols = np.arange(k.shape[2]) if cols is None else np.asarray(cols)
    dQ = np.zeros((B, len(heads), len(rows), d))
    dK = np.zeros((B, Hkv, len(cols), d))
    dV = np.zeros((B, Hkv, len(cols), d))
    per_head = isinstance(vec, dict) and "heads" in vec

    def feed(b, h):
        # rows that see at least one selected column: only they feed dK/dV there
        if isinstance(vec, dict):
            mc = _mask_rows(vec, causal, b, np.arange(N), h)[:, cols]
        else:
            lts, lte, uts, ute = (x[b] for x in vec)
            mc = masked_cols(lts, lte, uts, ute, causal, cols, n_rows=N)
        return np.nonzero(~mc.all(axis=1))[0]

    for b in range(B):
        row_pos = {int(r): t for t, r in enumerate(rows)}
        shared = None if per_head else feed(b, 0)
        for hi, h in enumerate(heads):
            feed_rows = feed(b, h) if per_head else shared
            need = np.union1d(rows, feed_rows)
            want_q = np.isin(need, rows)
            want_kv = np.isin(need, feed_rows)
            g = _kv_head(h, Hq, Hkv)
            for c0 in range(0, len(need), row_chunk):
                rr = need[c0 : c0 + row_chunk]
                if visible_only:
                    p, _, vc = row_probs_visible(q, k, vec, causal, scale, b, h, rr)
                else:
                    p, _ = row_probs(q, k, vec, causal, scale, b, h, rr)
                    vc = np.arange(k.shape[2])
                dp = do[b, h, rr] @ v[b, g][vc].T
                D = (p * dp).sum(axis=1)
                ds = p * (dp - D[:, None])
                wq = want_q[c0 : c0 + len(rr)]
                if wq.any():
                    dq_rows = scale * (ds[wq] @ k[b, g][vc])
                    for t, r in enumerate(rr[wq]):
                        dQ[b, hi, row_pos[int(r)]] = dq_rows[t]
                wk = want_kv[c0 : c0 + len(rr)]
                if wk.any():
                    # the selected columns among the computed ones (others: P = dS = 0)
                    pos = np.minimum(np.searchsorted(vc, cols), max(len(vc) - 1, 0))
                    hit = (vc[pos] == cols) if len(vc) else np.zeros(len(cols), dtype=bool)
                    p_c = np.zeros((int(wk.sum()), len(cols)))
                    ds_c = np.zeros_like(p_c)
                    p_c[:, hit] = p[wk][:, pos[hit]]
                    ds_c[:, hit] = ds[wk][:, pos[hit]]
                    dV[b, g] += p_c.T @ do[b, h, rr[wk]]
                    dK[b, g] += scale * (ds_c.T @ q[b, h, rr[wk]])
    return dQ, dK, dV


def unmasked_pairs(vec_b, causal: bool, row_chunk: int = 4096) -> int:
    """Number of visible (i, j) pairs of one batch entry's mask."""
    lts, lte, uts, ute = vec_b
    n = lts.shape[0]
    tot = 0
    for r0 in range(0, n, row_chunk):
        m = masked_rows(lts, lte, uts, ute, causal, np.arange(r0, min(r0 + row_chunk, n)))
        tot += int((~m).sum())
    return tot


# ------------------------------------------------ FMS / FME conversion
def from_fms_fme(fms, fme, n_rows: int):
    """The FlashMask Guide's representation ("Column-Wise Sparse Representation"
    under "The Solution: FlashMask Sparse Mask Representation"): key column j
    is visible exactly to rows FMS_j <= i <= FME_j (inclusive), one interval,
    with causality written into FMS. As the four vectors (used with causal
    off): the masked rows of column j are [0, FMS_j) and [FME_j + 1, N), so
    UTS = 0, UTE = FMS, LTS = FME + 1, LTE = N, each clipped to [0, N]. An
    empty interval (FMS_j > FME_j) masks the whole column.
    """
    n = int(n_rows)
    fms = np.asarray(fms, dtype=np.int64)
    fme = np.asarray(fme, dtype=np.int64)
    lts = np.clip(fme + 1, 0, n)
    lte = np.full_like(fms, n)
    uts = np.zeros_like(fms)
    ute = np.clip(fms, 0, n)
    return tuple(x.astype(np.int32) for x in (lts, lte, uts, ute))


# ---------------------------------------------------------- localization
def localize(x, offsets, C: int) -> np.ndarray:
    """Rank-local row boundaries, the clip-shift-max form.

    x^(r) = max_i [ clip(x - O_i, 0, C) + i*C*1(clip(x - O_i, 0, C) > 0) ],
    with O_i the global start of the rank's i-th chunk (ascending) and C the
    chunk length; the max over an all-zero set is 0.
    """
    x = np.asarray(x, dtype=np.int64)
    out = np.zeros_like(x)
    for i, o in enumerate(offsets):
        c = np.clip(x - int(o), 0, C)
        out = np.maximum(out, c + i * C * (c > 0))
    return out.astype(np.int32)


def localize_count(x, offsets, C: int) -> np.ndarray:
    """The same map as a plain count: number of the rank's rows before global row x."""
    x = np.asarray(x, dtype=np.int64)
    out = np.zeros_like(x)
    for o in offsets:
        out += np.clip(x - int(o), 0, C)
    return out.astype(np.int32)
