"""Pins of the oracle's FMS / FME conversion (FlashMask Guide, "The Solution:
FlashMask Sparse Mask Representation" and "Real-World Attention Mask
Topologies"): the Guide's own closed forms for causal, document and DPO masks
give its printed matrices and the masks of the workload encoders, and the
converted vectors mask exactly the rows outside [FMS_j, FME_j]."""
import os

import numpy as np
import pytest

import oracle
from oracle import reference
from workloads import masks

from test_oracle import GOLDEN, _read_golden


def visible(fms, fme, n):
    return ~oracle.dense_mask(*oracle.from_fms_fme(fms, fme, n), False)


def test_guide_causal_closed_form_matches_printed_matrix():
    n = 8
    g = _read_golden(os.path.join(GOLDEN, "p3_mask_topologies.txt"))["causal"]
    fms, fme = np.arange(n), np.full(n, n - 1)  # FMS_j = j, FME_j = N - 1
    assert np.array_equal(visible(fms, fme, n)[: g.shape[0]], g)


def test_guide_document_closed_form_matches_printed_matrix():
    n = 8
    g = _read_golden(os.path.join(GOLDEN, "p3_mask_topologies.txt"))["document_packing"]
    ends = np.repeat([1, 3, 5, 7], 2)  # documents of two tokens: FME_j = inclusive end
    assert np.array_equal(visible(np.arange(n), ends, n)[: g.shape[0]], g)


def test_guide_dpo_closed_form_equals_share_question_encoder():
    P, Cc, R = 5, 3, 4
    n = P + Cc + R
    fms = np.arange(n)
    fme = np.empty(n, np.int64)
    fme[:P] = n - 1             # prompt keys: every later row
    fme[P:P + Cc] = P + Cc - 1  # chosen keys: chosen rows only
    fme[P + Cc:] = n - 1        # rejected keys: rejected rows only
    ours = ~oracle.dense_mask(*masks.share_question([(P, Cc, R)], n), True)
    assert np.array_equal(visible(fms, fme, n), ours)


def test_conversion_brute_force():
    rng = np.random.default_rng(0)
    n = 37
    for _ in range(20):
        fms = rng.integers(-3, n + 4, size=n)
        fme = rng.integers(-3, n + 4, size=n)
        i = np.arange(n)[:, None]
        want = (fms[None, :] <= i) & (i <= fme[None, :])
        assert np.array_equal(visible(fms, fme, n), want)
        v = oracle.from_fms_fme(fms, fme, n)
        assert all(((x >= 0) & (x <= n)).all() for x in v)


def test_multi_interval_mask_brute_force():
    rng = np.random.default_rng(1)
    n, M = 23, 3
    fms = rng.integers(-2, n + 2, size=(M, n))
    fme = rng.integers(-2, n + 2, size=(M, n))
    got = oracle.multi_masked_rows(fms, fme, np.arange(n))
    for i in range(n):
        for j in range(n):
            vis = any(fms[m, j] <= i <= fme[m, j] for m in range(M))
            assert got[i, j] == (not vis)
    # one interval is the single-interval form
    one = oracle.multi_masked_rows(fms[:1], fme[:1], np.arange(n))
    assert np.array_equal(one, oracle.dense_mask(*oracle.from_fms_fme(fms[0], fme[0], n), False))


def test_multi_interval_mask_with_causal_brute_force():
    # the causal term (i < j masked) applies on top of the visible intervals,
    # as it does on top of the four-vector form
    rng = np.random.default_rng(2)
    n, M = 19, 3
    fms = rng.integers(-2, n + 2, size=(1, M, n))
    fme = rng.integers(-2, n + 2, size=(1, M, n))
    got = reference._mask_rows({"fms": fms, "fme": fme}, True, 0, np.arange(n))
    for i in range(n):
        for j in range(n):
            vis = any(fms[0, m, j] <= i <= fme[0, m, j] for m in range(M)) and i >= j
            assert got[i, j] == (not vis)
    assert np.array_equal(reference._mask_rows({"fms": fms, "fme": fme}, False, 0, np.arange(n)),
                          oracle.multi_masked_rows(fms[0], fme[0], np.arange(n)))


@pytest.mark.parametrize("causal", [False, True])
def test_multi_interval_tile_rule_is_sound_and_exact_at_1x1(causal):
    # the union rule (the most visible per-interval class) against the dense
    # multi-interval mask: skip => every element masked, unmasked => every
    # element visible, on overlapping and empty random intervals; at 1 x 1
    # tiles each interval's rule is exact, so the union's is too
    rng = np.random.default_rng(11 + causal)
    for n, nk, M, bm, bn in ((24, 24, 3, 4, 4), (20, 28, 2, 8, 4), (16, 16, 4, 1, 1), (9, 13, 2, 1, 1)):
        fms = rng.integers(-2, n + 2, size=(1, M, nk))
        fme = rng.integers(-2, n + 2, size=(1, M, nk))
        cls = oracle.classify_tiles_multi(fms[0], fme[0], causal, bm, bn, n)
        dense = reference._mask_rows({"fms": fms, "fme": fme}, causal, 0, np.arange(n))
        for qb in range(cls.shape[0]):
            for kb in range(cls.shape[1]):
                t = dense[qb * bm:(qb + 1) * bm, kb * bn:(kb + 1) * bn]
                if cls[qb, kb] == 0:
                    assert t.all()
                elif cls[qb, kb] == 2:
                    assert not t.any()
                elif bm == 1 and bn == 1:
                    raise AssertionError("a 1 x 1 tile is never partial")
    # one interval is the single-interval rule on its complement
    fms = rng.integers(0, 30, size=(1, 30))
    fme = rng.integers(0, 30, size=(1, 30))
    one = oracle.classify_tiles_multi(fms, fme, causal, 8, 8, 30)
    assert np.array_equal(one, oracle.classify_tiles(*oracle.from_fms_fme(fms[0], fme[0], 30), causal, 8, 8,
                                                      n_rows=30))


def test_union_runs_are_the_maximal_runs_of_the_visible_rows():
    # brute force: the runs cover exactly the rows some interval holds (within
    # [0, n)), are ascending with a gap of at least one row between them (so
    # maximal), and fill the first slots; empty, reversed, out-of-range,
    # overlapping and touching intervals all occur
    rng = np.random.default_rng(21)
    for n, nk, M in ((17, 40, 2), (30, 60, 3), (12, 50, 4), (1, 9, 3)):
        fms = rng.integers(-3, n + 3, size=(M, nk))
        fme = rng.integers(-3, n + 3, size=(M, nk))
        starts, ends = oracle.union_runs(fms, fme, n)
        for j in range(nk):
            want = {i for m in range(M) for i in range(n) if fms[m, j] <= i <= fme[m, j]}
            runs = [(int(a), int(b)) for a, b in zip(starts[:, j], ends[:, j]) if a <= b]
            assert all(a >= b + 2 for (_, b), (a, _) in zip(runs, runs[1:]))
            assert [int(a) <= int(b) for a, b in zip(starts[:, j], ends[:, j])] == [True] * len(runs) + [False] * (
                M - len(runs))
            assert {i for a, b in runs for i in range(a, b + 1)} == want
    # two touching pieces are one run; so are nested ones
    starts, ends = oracle.union_runs(np.array([[4], [0]]), np.array([[9], [3]]), 20)
    assert (starts[:, 0].tolist(), ends[:, 0].tolist()) == ([0, 20], [9, -1])
    starts, ends = oracle.union_runs(np.array([[2], [5]]), np.array([[15], [7]]), 20)
    assert (starts[:, 0].tolist(), ends[:, 0].tolist()) == ([2, 20], [15, -1])


@pytest.mark.parametrize("causal", [False, True])
def test_multi_interval_classes_do_not_depend_on_how_the_union_is_cut(causal):
    # the tile classes are a function of the mask: a column's single visible
    # interval cut into touching or overlapping pieces, in any slot order,
    # classifies exactly like the interval itself
    rng = np.random.default_rng(31 + causal)
    n = 96
    a = rng.integers(0, n, size=n)
    b = np.minimum(a + rng.integers(0, n, size=n), n - 1)
    one = oracle.classify_tiles(*oracle.from_fms_fme(a, b, n), causal, 16, 16, n_rows=n)
    cut = a + (b - a) // 3
    over = np.minimum(cut + 4, b)
    for fms, fme in ((np.stack([a, cut + 1]), np.stack([cut, b])),           # touching halves
                     (np.stack([cut + 1, a]), np.stack([b, cut])),           # swapped slots
                     (np.stack([a, a, cut]), np.stack([over, b, b]))):       # overlapping, nested
        assert np.array_equal(oracle.classify_tiles_multi(fms, fme, causal, 16, 16, n), one)


@pytest.mark.parametrize("causal", [False, True])
def test_multi_interval_tile_that_no_run_reaches_is_skipped(causal):
    # blocks whose columns hold one run each (cut into pieces) or none (fully
    # masked columns mixed in): a tile wholly above every live run of its
    # block, or wholly below, has no visible element and must be skipped
    rng = np.random.default_rng(41 + causal)
    n, nk, bm, bn = 64, 64, 8, 8
    for _ in range(20):
        a = rng.integers(0, n, size=nk)
        b = np.minimum(a + rng.integers(0, 24, size=nk), n - 1)
        dead = rng.random(nk) < 0.3
        a, b = np.where(dead, 5, a), np.where(dead, 2, b)          # empty interval
        cut = a + (b - a) // 2
        fms, fme = np.stack([a, cut + 1]), np.stack([cut, b])
        cls = oracle.classify_tiles_multi(fms, fme, causal, bm, bn, n)
        dense = reference._mask_rows({"fms": fms[None], "fme": fme[None]}, causal, 0, np.arange(n))
        for kb in range(nk // bn):
            live = ~dead[kb * bn:(kb + 1) * bn]
            lo = a[kb * bn:(kb + 1) * bn][live].min() if live.any() else n
            hi = b[kb * bn:(kb + 1) * bn][live].max() if live.any() else -1
            for qb in range(n // bm):
                if (qb + 1) * bm <= lo or qb * bm > hi:
                    assert dense[qb * bm:(qb + 1) * bm, kb * bn:(kb + 1) * bn].all()
                    assert cls[qb, kb] == 0, (qb, kb)


def test_multi_interval_attention_is_the_lse_merge_of_its_parts():
    # With disjoint intervals per column, a row's visible keys split into
    # disjoint sets, one per interval: the attention over their union is the
    # LSE-weighted merge of the per-interval attentions, and its gradients
    # are the sums of the per-interval backward passes taken with the merged
    # output and LSE (the row term D then belongs to the merged output).
    rng = np.random.default_rng(2)
    n, d, M = 48, 8, 3
    cuts = np.sort(rng.integers(0, n, size=(2 * M, n)), axis=0)  # disjoint, ascending per column
    fms, fme = cuts[0::2], cuts[1::2] - 1
    q, k, v, do = (rng.standard_normal((1, 2, n, d)) for _ in range(4))
    k, v = k[:, :1], v[:, :1]
    spec = {"fms": fms[None], "fme": fme[None]}
    O, L = oracle.forward(q, k, v, spec, False, 0.3)
    parts = [oracle.forward(q, k, v, tuple(x[None] for x in oracle.from_fms_fme(fms[m], fme[m], n)), False, 0.3)
             for m in range(M)]
    Ls = np.stack([p[1] for p in parts])
    with np.errstate(invalid="ignore", divide="ignore"):
        top = np.max(Ls, axis=0)
        Lm = np.where(np.isneginf(top), -np.inf, top + np.log(np.sum(np.exp(Ls - np.where(np.isneginf(top), 0, top)), axis=0)))
        w = np.where(np.isneginf(Ls), 0.0, np.exp(Ls - np.where(np.isneginf(Lm), 0, Lm)))
    Om = sum(w[m][..., None] * parts[m][0] for m in range(M))
    assert np.array_equal(np.isneginf(Lm), np.isneginf(L))
    fin = ~np.isneginf(L)
    assert np.allclose(Lm[fin], L[fin], atol=1e-12) and np.allclose(Om, O, atol=1e-12)


def test_per_head_masks_reduce_to_one_head_problems():
    # one set of vectors per query head: each head's output is that of a
    # one-head problem with its own vectors, and each kv head's key gradients
    # are the sum over its query heads of those problems' gradients
    rng = np.random.default_rng(3)
    B, hq, hkv, n, d = 2, 4, 2, 40, 8
    G = hq // hkv
    a = rng.integers(0, n + 1, size=(2, B, hq, n))
    c = rng.integers(0, n + 1, size=(2, B, hq, n))
    heads = (a.min(0), a.max(0), c.min(0), c.max(0))
    q, do = (rng.standard_normal((B, hq, n, d)) for _ in range(2))
    k, v = (rng.standard_normal((B, hkv, n, d)) for _ in range(2))
    spec = {"heads": heads}
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, spec, causal, 0.4)
        dQ, dK, dV = oracle.backward(q, k, v, do, spec, causal, 0.4)
        dK_sum, dV_sum = np.zeros_like(dK), np.zeros_like(dV)
        for h in range(hq):
            g = h // G
            one = tuple(x[:, h] for x in heads)
            sl, gl = slice(h, h + 1), slice(g, g + 1)
            O1, L1 = oracle.forward(q[:, sl], k[:, gl], v[:, gl], one, causal, 0.4)
            assert np.allclose(O1, O[:, sl], atol=1e-12)
            assert np.array_equal(np.isneginf(L1), np.isneginf(L[:, sl]))
            dq1, dk1, dv1 = oracle.backward(q[:, sl], k[:, gl], v[:, gl], do[:, sl], one, causal, 0.4)
            assert np.allclose(dq1, dQ[:, sl], atol=1e-12)
            dK_sum[:, gl] += dk1
            dV_sum[:, gl] += dv1
        assert np.allclose(dK_sum, dK, atol=1e-10) and np.allclose(dV_sum, dV, atol=1e-10)
