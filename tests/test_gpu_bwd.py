"""GPU backward parity against the fp64 oracle (dQ, dK, dV rel-L2 <= 1e-2)."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, masks, tensors

from helpers import assert_grad, f64, random_vectors

pytestmark = pytest.mark.gpu


def _run(vec, B, hq, hkv, n, d, causal, scale=None):
    scale = d ** -0.5 if scale is None else scale
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d)
    q, k, v, do = tensors.make_qkvdo(cfg)
    dv_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv_, causal=causal)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *dv_, qs, scale=scale, causal=causal)
    dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *dv_, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec, causal, scale)
    return (f64(dq), f64(dk), f64(dv)), ref


def _assert_all(got, ref):
    for name, a, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_grad(a, r, name)


def test_bwd_tiny_config():
    cfg = configs.make("tiny")
    vec = tuple(cfg[x] for x in ("lts", "lte", "uts", "ute"))
    got, ref = _run(vec, cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], cfg["d"], True)
    _assert_all(got, ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_random_masks(d, hq, hkv, causal):
    rng = np.random.default_rng(d + 10 * hq + 100 * hkv + causal)
    for n in (128, 384):
        vec = random_vectors(rng, 1, n, "general")
        got, ref = _run(vec, 1, hq, hkv, n, d, causal)
        _assert_all(got, ref)


@pytest.mark.parametrize("n", [1, 100, 200, 300])
def test_bwd_ragged_n(n):
    rng = np.random.default_rng(n)
    vec = random_vectors(rng, 2, n, "lower")
    got, ref = _run(vec, 2, 4, 2, n, 128, True)
    _assert_all(got, ref)


@pytest.mark.parametrize("kind", ["docs", "share_question", "prefix_lm", "window", "eviction"])
def test_bwd_mask_families_2k(kind):
    rng = np.random.default_rng(7)
    n = 2048
    if kind == "docs":
        v, causal = masks.causal_documents(masks.draw_fill(rng, n, 100, 700), n), True
    elif kind == "share_question":
        v, causal = masks.share_question([(300, 150, 200), (257, 90, 300), (111, 64, 65)], n), True
    elif kind == "prefix_lm":
        v, causal = masks.prefix_lm_documents(masks.draw_fill(rng, n, 200, 900), n), False
    elif kind == "window":
        v, causal = masks.sliding_window(n, 300, 4), True
    else:
        v, causal = masks.random_eviction(n, 1 / 256, rng), True
    vec = tuple(x[None] for x in v)
    got, ref = _run(vec, 1, 4, 2, n, 128, causal)
    _assert_all(got, ref)


def test_bwd_everything_masked_gives_zero():
    n = 256
    vec = tuple(x[None] for x in masks.share_question([], n))
    (dq, dk, dv), _ = _run(vec, 1, 2, 1, n, 128, True)
    assert (dq == 0).all() and (dk == 0).all() and (dv == 0).all()


def test_bwd_no_mask_dense():
    n = 512
    vec = tuple(x[None] for x in masks._empty(n))
    got, ref = _run(vec, 1, 4, 1, n, 128, False)
    _assert_all(got, ref)


def test_bwd_gqa_group_of_64_heads():
    # the random-eviction family's head layout (H_kv = 1) at a small N
    rng = np.random.default_rng(11)
    n = 256
    vec = tuple(x[None] for x in masks.random_eviction(n, 1 / 64, rng))
    got, ref = _run(vec, 1, 64, 1, n, 128, True)
    _assert_all(got, ref)
