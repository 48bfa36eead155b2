"""The FP8 forward's tolerance, pinned on the CPU: the only rounding the FP8
path adds beyond its (dequantized) inputs is P -> e4m3 before O = P V. With
P rounded to e4m3 by torch's own conversion (round to nearest even), the
oracle's O moves from the exact O by about the relative RMS rounding error of
a 3-mantissa-bit format, ~2.5% in relative L2, and element-wise by at most
2^-4 max|V|; the GPU test's bounds (rel-L2 4e-2, max-abs 2^-4 max|V| + 1e-2) must hold with
margin for every mask family, and a coarser format (a planted
2-mantissa-bit rounding) must show about twice the error, so the measure
tracks the format's precision."""
import numpy as np
import pytest
import torch

import oracle
from workloads import masks

FP8_O_REL_L2, FP8_P_REL = 4e-2, 2.0 ** -4


def _o_with_rounded_p(q, k, v, vec, causal, scale, rnd):
    """O with P (normalised to its row max, the kernel's P <= 1 case) rounded by rnd."""
    n = q.shape[2]
    p, lse = oracle.row_probs(q, k, vec, causal, scale, 0, 0, np.arange(n))
    live = ~np.isneginf(lse)
    mx = np.where(live, p.max(axis=1), 1.0)[:, None]
    pn = p / mx                          # exp(S - max): what the kernel exponentiates
    l = pn.sum(axis=1, keepdims=True)    # the kernel's row sum, unrounded
    pr = rnd(pn)
    return np.where(live[:, None], (pr @ v[0, 0]) / np.where(live[:, None], l, 1.0), 0.0), live


def _e4m3(x):
    return torch.from_numpy(x).float().to(torch.float8_e4m3fn).double().numpy()


def _two_mantissa_bits(x):
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 8) / 8, e)


@pytest.mark.parametrize("kind", ["docs", "prefix_lm", "window", "eviction", "dense"])
def test_fp8_tolerance_model(kind):
    rng = np.random.default_rng(3)
    n, d = 1024, 128
    if kind == "docs":
        v, causal = masks.causal_documents(masks.draw_fill(rng, n, 50, 400), n), True
    elif kind == "prefix_lm":
        v, causal = masks.prefix_lm_documents(masks.draw_fill(rng, n, 100, 500), n), False
    elif kind == "window":
        v, causal = masks.sliding_window(n, 200, 4), True
    elif kind == "eviction":
        v, causal = masks.random_eviction(n, 1 / 128, rng), True
    else:
        v, causal = masks._empty(n), False
    vec = tuple(x[None] for x in v)
    q, k, vv = (rng.standard_normal((1, 1, n, d)) for _ in range(3))
    scale = d ** -0.5
    O, _ = oracle.forward(q, k, vv, vec, causal, scale)
    Oq, live = _o_with_rounded_p(q, k, vv, vec, causal, scale, _e4m3)
    rel = np.linalg.norm(Oq - O[0, 0]) / np.linalg.norm(O[0, 0])
    mx = np.abs(Oq - O[0, 0]).max()
    assert 0.005 < rel < FP8_O_REL_L2 / 1.3 and mx < FP8_P_REL * np.abs(vv).max(), (rel, mx)
    # one mantissa bit fewer doubles the error: the measure tracks the format
    Oc, _ = _o_with_rounded_p(q, k, vv, vec, causal, scale, _two_mantissa_bits)
    assert np.linalg.norm(Oc - O[0, 0]) / np.linalg.norm(O[0, 0]) > 1.6 * rel
