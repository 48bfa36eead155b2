"""GPU forward parity against the fp64 oracle (O rel-L2 <= 5e-3, max-abs <= 2e-2;
LSE max-abs <= 1e-3; fully-masked rows exactly O = 0, LSE = -inf)."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, masks, tensors

from helpers import assert_lse, assert_out, f64, random_vectors

pytestmark = pytest.mark.gpu


def _run(vec, B, hq, hkv, n, d, causal, scale=None, seed=1):
    scale = d ** -0.5 if scale is None else scale
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d)
    q, k, v, _ = tensors.make_qkvdo(cfg)
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv, causal=causal)
    o, lse = fm.fm_attn_fwd(q.cuda(), k.cuda(), v.cuda(), *dv, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vec, causal, scale)
    return f64(o), f64(lse), O_ref, L_ref


def test_fwd_tiny_config():
    cfg = configs.make("tiny")
    vec = tuple(cfg[x] for x in ("lts", "lte", "uts", "ute"))
    o, lse, O, L = _run(vec, cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], cfg["d"], True)
    assert_out(o, O)
    assert_lse(lse, L)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 2), (8, 1), (6, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_random_masks(d, hq, hkv, causal):
    rng = np.random.default_rng(d + 10 * hq + 100 * hkv + causal)
    for n in (128, 384):
        vec = random_vectors(rng, 1, n, "general")
        o, lse, O, L = _run(vec, 1, hq, hkv, n, d, causal)
        assert_out(o, O)
        assert_lse(lse, L)


@pytest.mark.parametrize("n", [1, 100, 200, 300, 389])
def test_fwd_ragged_n(n):
    # n = 389 with B = 2: the second batch entry's mask vectors are not 16-byte
    # aligned, so the kernel takes its element-wise mask path
    rng = np.random.default_rng(n)
    vec = random_vectors(rng, 2, n, "lower")
    o, lse, O, L = _run(vec, 2, 4, 2, n, 128, True)
    assert_out(o, O)
    assert_lse(lse, L)


@pytest.mark.parametrize("kind", ["docs", "share_question", "prefix_lm", "window", "eviction"])
def test_fwd_mask_families_2k(kind):
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
    o, lse, O, L = _run(vec, 1, 4, 2, n, 128, causal)
    assert_out(o, O)
    assert_lse(lse, L)


def test_fwd_fully_masked_everything():
    n = 256
    vec = tuple(x[None] for x in masks.share_question([], n))  # every row padding
    o, lse, O, L = _run(vec, 1, 2, 1, n, 128, True)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_fwd_no_mask_is_dense_attention():
    n = 512
    vec = tuple(x[None] for x in masks._empty(n))
    o, lse, O, L = _run(vec, 1, 2, 2, n, 128, False)
    assert_out(o, O)
    assert_lse(lse, L)


def test_fwd_deterministic():
    rng = np.random.default_rng(3)
    vec = random_vectors(rng, 1, 384, "general")
    a = _run(vec, 1, 4, 1, 384, 128, True)
    b = _run(vec, 1, 4, 1, 384, 128, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
