"""CPU oracle of the sparsity-aware chunk balancer (HCC-IPO Stage 1).

TEST INFRASTRUCTURE. Only the tests and the benchmark's CPU legs import this
module; the library never calls it and shares no code with it. Plain,
exhaustive Python, written from FlashMask-3 project page, §3.3 ("Balance the
work, not the length") and the "IPO phase ablation" table of §4:

* the query axis is cut into n = P * kappa chunks and every rank receives
  exactly kappa of them (the cardinality constraint);
* tile cost model: a skipped tile costs 0, a partial tile alpha_p, an
  unmasked tile alpha_u; the load w_i of a chunk is the sum over its tiles;
* the load of rank j is L_j = sum of its chunks' loads, the makespan is
  Phi = max_j L_j, and LB = max(ceil(sum w / P), max w) is a lower bound:
  an assignment with Phi == LB is optimal (the certificate);
* Stage 1 runs LPT, then exact pairwise repartition (P2), then exact
  three-rank repartition (P3);
* the K / V exchange sends a rank only the chunks its rows can see (§3.4).

A second lower bound uses the cardinality constraint that LB ignores (a
pigeonhole argument, not on the pages): the m lightest chunks are held by at
most m ranks, so at least P - m ranks hold none of them and carry at least the
(P - m) * kappa lightest of the others; and the rank with the heaviest chunk
holds kappa - 1 more. LB_kappa (>= LB) is the largest of these bounds; the
certificate is makespan == LB_kappa and every phase stops there.

Readings where the pages are silent (the library follows the same ones):
  - LPT: chunks in order of load descending, ties by chunk index; each goes to
    the least-loaded rank still holding fewer than kappa chunks, ties to the
    lowest rank index.
  - A repartition of a group of k ranks (k = 2 in P2, 3 in P3) pools their
    k * kappa chunks and deals them out again, kappa each, so that the
    group's largest load is as small as possible; it is applied only when
    that is strictly below the group's current largest load. Among the best
    deals the first in this order is taken: the pool sorted by chunk index,
    the first rank's set running over the kappa-combinations of the pool in
    lexicographic order, the second rank's over those of the rest, the last
    rank taking what is left.
  - Only groups that hold a rank whose load equals the current makespan are
    visited (no other group can lower it), in lexicographic order of their
    rank indices; one sweep visits every such group once and applies each
    improvement as it is found.
  - P2 repeats sweeps over pairs until one applies nothing. P3 alternates one
    sweep over triples with P2 run to its end, until a triple sweep applies
    nothing. Every phase stops as soon as Phi == LB_kappa.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

SKIP, PARTIAL, UNMASKED = 0, 1, 2


def chunk_loads(tile_class, blocks_per_chunk: int, cost_partial: int, cost_unmasked: int) -> np.ndarray:
    """Load of every chunk: tile_class is (B, nQ, nK); chunk c holds Q blocks
    [c * blocks_per_chunk, (c + 1) * blocks_per_chunk) of every batch entry
    (the last chunk may be short)."""
    tile_class = np.asarray(tile_class)
    B, nq, nk = tile_class.shape
    n = -(-nq // blocks_per_chunk)
    w = np.zeros(n, dtype=np.int64)
    for b in range(B):
        for qb in range(nq):
            c = qb // blocks_per_chunk
            for kb in range(nk):
                t = tile_class[b, qb, kb]
                if t == PARTIAL:
                    w[c] += cost_partial
                elif t == UNMASKED:
                    w[c] += cost_unmasked
    return w


def needed_chunks(tile_class, owner, P: int, blocks_per_chunk: int) -> np.ndarray:
    """Mask-aware pruning of the K / V exchange (FlashMask-3 project page,
    §3.4: a chunk the mask fully hides is never sent): need[r, c] = 1 iff some
    tile between the query blocks of rank r's chunks and the key blocks of
    chunk c, in any batch entry, is not skipped. Chunks cut both axes alike
    (a chunk is a range of tokens: its query rows and its keys)."""
    tile_class = np.asarray(tile_class)
    B, nq, nk = tile_class.shape
    n = len(owner)
    need = np.zeros((P, n), dtype=np.uint8)
    for b in range(B):
        for qb in range(nq):
            r = owner[qb // blocks_per_chunk]
            for kb in range(nk):
                if tile_class[b, qb, kb] != SKIP:
                    need[r, kb // blocks_per_chunk] = 1
    return need


def lower_bound(w, P: int) -> int:
    w = [int(x) for x in w]
    return max(-(-sum(w) // P), max(w))


def lower_bound_kappa(w, P: int, kappa: int) -> int:
    ws = sorted(int(x) for x in w)
    bounds = [ws[-1] + sum(ws[: kappa - 1])]
    for m in range(P):
        held = ws[m : m + (P - m) * kappa]  # the lightest chunks a rank outside the first m can hold
        bounds.append(-(-sum(held) // (P - m)))
    return max(bounds)


def rank_loads(w, owner, P: int):
    L = [0] * P
    for i, r in enumerate(owner):
        L[r] += int(w[i])
    return L


def lpt(w, P: int, kappa: int):
    """Longest-processing-time-first under the cardinality constraint."""
    n = len(w)
    order = sorted(range(n), key=lambda i: (-int(w[i]), i))
    load = [0] * P
    count = [0] * P
    owner = [-1] * n
    for i in order:
        best = None
        for r in range(P):
            if count[r] < kappa and (best is None or load[r] < load[best]):
                best = r
        owner[i] = best
        load[best] += int(w[i])
        count[best] += 1
    return owner


def _deals(pool, k: int, kappa: int):
    """Every deal of `pool` (sorted) into k sets of kappa, in the stated order."""
    if k == 1:
        yield (tuple(pool),)
        return
    for first in itertools.combinations(pool, kappa):
        rest = [c for c in pool if c not in first]
        for tail in _deals(rest, k - 1, kappa):
            yield (first,) + tail


def best_deal(w, pool, k: int, kappa: int, bar: int):
    """The first deal whose largest set load is minimal and below `bar`, or None."""
    best, best_val = None, bar
    for deal in _deals(sorted(pool), k, kappa):
        val = max(sum(int(w[c]) for c in s) for s in deal)
        if val < best_val:
            best, best_val = deal, val
    return best


def _sweep(w, owner, P: int, kappa: int, k: int, lb: int) -> int:
    """One sweep over the groups of k ranks; returns the number of moves."""
    moves = 0
    for group in itertools.combinations(range(P), k):
        L = rank_loads(w, owner, P)
        phi = max(L)
        if phi == lb:
            break
        if all(L[r] != phi for r in group):
            continue
        pool = [i for i in range(len(w)) if owner[i] in group]
        deal = best_deal(w, pool, k, kappa, max(L[r] for r in group))
        if deal is not None:
            for r, s in zip(group, deal):
                for c in s:
                    owner[c] = r
            moves += 1
    return moves


def ipo(w, P: int, kappa: int, phases: int = 3):
    """Stage 1 of HCC-IPO: returns (owner list, report dict)."""
    n = len(w)
    assert n == P * kappa
    lb = lower_bound_kappa(w, P, kappa)
    owner = lpt(w, P, kappa)
    rep = dict(lower_bound=lower_bound(w, P), lower_bound_kappa=lb, makespan_lpt=max(rank_loads(w, owner, P)),
               pair_moves=0, triple_moves=0)

    def pair_phase():
        while max(rank_loads(w, owner, P)) > lb:
            m = _sweep(w, owner, P, kappa, 2, lb)
            rep["pair_moves"] += m
            if m == 0:
                break

    if phases >= 2 and P >= 2:
        pair_phase()
    rep["makespan_pair"] = max(rank_loads(w, owner, P))
    if phases >= 3 and P >= 3:
        while max(rank_loads(w, owner, P)) > lb:
            m = _sweep(w, owner, P, kappa, 3, lb)
            rep["triple_moves"] += m
            if m == 0:
                break
            pair_phase()
    rep["makespan"] = max(rank_loads(w, owner, P))
    rep["certified"] = int(rep["makespan"] == lb)
    return owner, rep


def optimum(w, P: int, kappa: int) -> int:
    """Smallest makespan over every assignment (exhaustive; tiny instances only)."""
    best = math.inf
    for deal in _deals(list(range(len(w))), P, kappa):
        best = min(best, max(sum(int(w[c]) for c in s) for s in deal))
    return int(best)

