"""Head dimension 256 (the FlashMask Guide's usage example, "Complete PyTorch
Implementation", runs the operator at dim = 256): GPU parity against the fp64
oracle with the same tolerances as every other head size (O rel-L2 <= 5e-3,
max-abs <= 2e-2; LSE max-abs <= 1e-3; fully-masked rows exactly O = 0,
LSE = -inf; dQ, dK, dV rel-L2 <= 1e-2)."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, masks, tensors

from helpers import assert_grad, assert_lse, assert_out, f64, random_vectors

pytestmark = pytest.mark.gpu

D = 256


def _fwd(vec, B, hq, hkv, n, causal, seed_scale=None):
    scale = D ** -0.5 if seed_scale is None else seed_scale
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=D)
    q, k, v, do = tensors.make_qkvdo(cfg)
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv, causal=causal)
    o, lse = fm.fm_attn_fwd(q.cuda(), k.cuda(), v.cuda(), *dv, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vec, causal, scale)
    return f64(o), f64(lse), O_ref, L_ref


def _families(kind, n, rng):
    if kind == "docs":
        return masks.causal_documents(masks.draw_fill(rng, n, 100, 700), n), True
    if kind == "share_question":
        return masks.share_question([(300, 150, 200), (257, 90, 300), (111, 64, 65)], n), True
    if kind == "prefix_lm":
        return masks.prefix_lm_documents(masks.draw_fill(rng, n, 200, 900), n), False
    if kind == "window":
        return masks.sliding_window(n, 300, 4), True
    return masks.random_eviction(n, 1 / 256, rng), True


def test_fwd256_tiny_config():
    cfg = configs.make("tiny", d=D)
    vec = tuple(cfg[x] for x in ("lts", "lte", "uts", "ute"))
    o, lse, O, L = _fwd(vec, cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], True)
    assert_out(o, O)
    assert_lse(lse, L)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 2), (3, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd256_random_masks(hq, hkv, causal):
    rng = np.random.default_rng(256 + 10 * hq + 100 * hkv + causal)
    for n in (128, 384):
        vec = random_vectors(rng, 1, n, "general")
        o, lse, O, L = _fwd(vec, 1, hq, hkv, n, causal)
        assert_out(o, O)
        assert_lse(lse, L)


@pytest.mark.parametrize("n", [1, 100, 300, 389])
def test_fwd256_ragged_n(n):
    # B = 2 and n = 389: the second entry's vectors are not 16-byte aligned
    rng = np.random.default_rng(n + 256)
    vec = random_vectors(rng, 2, n, "lower")
    o, lse, O, L = _fwd(vec, 2, 2, 1, n, True)
    assert_out(o, O)
    assert_lse(lse, L)


@pytest.mark.parametrize("kind", ["docs", "share_question", "prefix_lm", "window", "eviction"])
def test_fwd256_mask_families_2k(kind):
    rng = np.random.default_rng(11)
    v, causal = _families(kind, 2048, rng)
    o, lse, O, L = _fwd(tuple(x[None] for x in v), 1, 2, 1, 2048, causal)
    assert_out(o, O)
    assert_lse(lse, L)


def test_fwd256_fully_masked_and_deterministic():
    n = 384
    vec = tuple(x[None] for x in masks.share_question([(100, 40, 50)], n))  # rows from 190 on see nothing
    a = _fwd(vec, 1, 2, 1, n, True)
    b = _fwd(vec, 1, 2, 1, n, True)
    assert_out(a[0], a[2])
    assert_lse(a[1], a[3])
    assert (a[0][:, :, 190:] == 0).all() and np.isneginf(a[1][:, :, 190:]).all()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fwd256_long_pass_natural_order():
    # more than eight waves of CTAs: units run in natural order
    rng = np.random.default_rng(5)
    n = 8192
    vec = tuple(x[None] for x in masks.causal_documents(masks.draw_fill(rng, n, 256, 2048), n))
    cfg = dict(B=1, H_q=16, H_kv=4, N=n, d=D)
    q, k, v, _ = tensors.make_qkvdo(cfg, device="cuda")
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv, causal=True)
    o, lse = fm.fm_attn_fwd(q, k, v, *dv, qs, scale=D ** -0.5, causal=True)
    assert fm.fm_device_status()[0] == fm.FM_OK
    rows = np.sort(np.random.default_rng(1).choice(n, 256, replace=False))
    for h in (0, 13):
        g = h // 4
        O_ref, L_ref = oracle.forward(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]), vec, True,
                                      D ** -0.5, rows=rows)
        tr = torch.as_tensor(rows, device="cuda")
        assert_out(f64(o[:, h:h + 1, tr]), O_ref)
        assert_lse(f64(lse[:, h:h + 1, tr]), L_ref)


# ---------------------------------------------------------------- backward
def _bwd(vec, B, hq, hkv, n, causal):
    scale = D ** -0.5
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=D)
    q, k, v, do = tensors.make_qkvdo(cfg)
    dv_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv_, causal=causal)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *dv_, qs, scale=scale, causal=causal)
    dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *dv_, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec, causal, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


def test_bwd256_tiny_config():
    cfg = configs.make("tiny", d=D)
    _bwd(tuple(cfg[x] for x in ("lts", "lte", "uts", "ute")), cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], True)


@pytest.mark.parametrize("hq,hkv", [(1, 1), (4, 2), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd256_random_masks(hq, hkv, causal):
    rng = np.random.default_rng(512 + 10 * hq + hkv + causal)
    for n in (128, 384):
        _bwd(random_vectors(rng, 1, n, "general"), 1, hq, hkv, n, causal)


@pytest.mark.parametrize("n", [1, 100, 300, 389])
def test_bwd256_ragged_n(n):
    rng = np.random.default_rng(n + 512)
    _bwd(random_vectors(rng, 2, n, "lower"), 2, 2, 1, n, True)


@pytest.mark.parametrize("kind", ["docs", "share_question", "prefix_lm", "window", "eviction"])
def test_bwd256_mask_families_2k(kind):
    rng = np.random.default_rng(13)
    v, causal = _families(kind, 2048, rng)
    _bwd(tuple(x[None] for x in v), 1, 4, 2, 2048, causal)
