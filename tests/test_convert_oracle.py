"""Pins of the oracle's FMS / FME conversion (FlashMask Guide, "The Solution:
FlashMask Sparse Mask Representation" and "Real-World Attention Mask
Topologies"): the Guide's own closed forms for causal, document and DPO masks
give its printed matrices and the masks of this build's encoders, and the
converted vectors mask exactly the rows outside [FMS_j, FME_j]."""
import os

import numpy as np

import oracle
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
