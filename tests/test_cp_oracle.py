"""Zero-communication localization, end to end, in the oracle (FlashMask-3
project page, §3.2, Theorem 1): a rank that holds some chunks of the query
rows and every key, with the four vectors localized to its rows, computes for
each of its rows exactly the mask, output and gradients of that row in the
whole problem; the ranks' key gradients add up to the whole problem's."""
import numpy as np
import pytest

import oracle
from workloads import masks


def fold_causal(vec, n):
    """Causal masking moved into the upper interval: UTS_j = 0, UTE_j = j
    (rows i < j masked), valid where the upper interval is otherwise empty."""
    lts, lte, uts, ute = vec
    assert not ((uts < ute).any())
    return lts, lte, np.zeros(n, np.int32), np.arange(n, dtype=np.int32)


def rank_rows(owner, r, C):
    return np.concatenate([np.arange(c * C, (c + 1) * C) for c in np.nonzero(np.asarray(owner) == r)[0]])


def cases(n):
    rng = np.random.default_rng(0)
    doc = masks.causal_documents([n // 4 + 40, n // 3, n - n // 4 - 40 - n // 3], n)
    pre = masks.prefix_lm_documents([n // 2 + 64, n - n // 2 - 64], n)
    a = rng.integers(0, n + 1, size=(2, n))
    c = rng.integers(0, n + 1, size=(2, n))
    gen = (a.min(0), a.max(0), c.min(0), c.max(0))
    return {"doc_causal_folded": fold_causal(doc, n), "prefix_lm": pre, "general": gen}


@pytest.mark.parametrize("name", ["doc_causal_folded", "prefix_lm", "general"])
def test_localized_rank_equals_whole_problem(name):
    n, C, P, kappa, d = 256, 32, 4, 2, 16
    vec = tuple(np.asarray(x, np.int32) for x in cases(n)[name])
    rng = np.random.default_rng(1)
    owner = rng.permutation(np.repeat(np.arange(P), kappa))  # chunk -> rank, kappa each
    q, k, v, do = (rng.standard_normal((1, 2, n, d)) for _ in range(4))
    k, v = k[:, :1], v[:, :1]  # GQA: two query heads on one kv head
    scale = d ** -0.5
    vb = tuple(x[None] for x in vec)
    O, L = oracle.forward(q, k, v, vb, False, scale)
    dQ, dK, dV = oracle.backward(q, k, v, do, vb, False, scale)
    dK_sum, dV_sum = np.zeros_like(dK), np.zeros_like(dV)
    for r in range(P):
        rows = rank_rows(owner, r, C)
        offsets = np.sort(np.nonzero(owner == r)[0]) * C
        loc = tuple(oracle.localize(x, offsets, C)[None] for x in vec)
        # the localized mask of the rank's rows is the global mask of those rows
        m_loc = oracle.masked_rows(*(x[0] for x in loc), False, np.arange(len(rows)))
        m_glob = oracle.masked_rows(*vec, False, rows)
        assert np.array_equal(m_loc, m_glob)
        O_r, L_r = oracle.forward(q[:, :, rows], k, v, loc, False, scale)
        assert np.allclose(O_r, O[:, :, rows], rtol=1e-12, atol=1e-12)
        assert np.array_equal(np.isneginf(L_r), np.isneginf(L[:, :, rows]))
        fin = ~np.isneginf(L_r)
        assert np.allclose(L_r[fin], L[:, :, rows][fin], rtol=1e-12, atol=1e-12)
        dQ_r, dK_r, dV_r = oracle.backward(q[:, :, rows], k, v, do[:, :, rows], loc, False, scale)
        assert np.allclose(dQ_r, dQ[:, :, rows], rtol=1e-10, atol=1e-12)
        dK_sum += dK_r
        dV_sum += dV_r
    assert np.allclose(dK_sum, dK, rtol=1e-10, atol=1e-12)
    assert np.allclose(dV_sum, dV, rtol=1e-10, atol=1e-12)


def test_causal_fold_is_the_causal_mask():
    n = 96
    doc = masks.causal_documents([30, 40, 26], n)
    folded = fold_causal(doc, n)
    assert np.array_equal(oracle.dense_mask(*folded, False), oracle.dense_mask(*doc, True))


def test_rectangular_classes_cover_the_mask():
    # tile classes of a rank's (rows x all keys) problem: skipped tiles hold
    # only masked pairs, unmasked tiles only visible ones
    n, C = 512, 64
    vec = cases(n)["general"]
    offsets = np.array([64, 320])
    loc = tuple(oracle.localize(x, offsets, C) for x in vec)
    nr = 2 * C
    cls = oracle.classify_tiles(*loc, False, 32, 64, n_rows=nr)
    assert cls.shape == (nr // 32, n // 64)
    m = oracle.masked_rows(*loc, False, np.arange(nr))
    for qb in range(cls.shape[0]):
        for kb in range(cls.shape[1]):
            t = m[qb * 32:(qb + 1) * 32, kb * 64:(kb + 1) * 64]
            if cls[qb, kb] == oracle.SKIP:
                assert t.all()
            elif cls[qb, kb] == oracle.UNMASKED:
                assert not t.any()
