"""FP8 forward ("Flash MSA Attention Kernel Implementation", "Optimization Tricks
That Actually Matter": FP8 products inside the tile, softmax in FP32) against
the fp64 oracle run on the DEQUANTIZED inputs (stored e4m3 value x scale).

Tolerances (derived in the library's design notes, pinned on the CPU by
tests/test_fp8_tolerance.py): the kernel rounds P to e4m3 before O = P V,
whose relative rounding error (3 mantissa bits) averages to about 2.5% of O
in relative L2 norm: O rel-L2 <= 4e-2. Element-wise, every rounded P_j is
within 2^-4 P_j of the exact one (e4m3's worst relative rounding) and the
row sum is at least 1 (the exponent base is within 8 of the row max, in log2
units), so |O - O_exact| <= 2^-4 max|V| (+ 1e-2 for subnormal P and the bf16
output). S = Q K^T is exact
up to fp32 accumulation (products of e4m3 values are exact in fp32), so LSE
keeps the bf16 path's bound, max-abs <= 1e-3. Fully-masked rows: exactly
O = 0 and LSE = -inf.
"""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, masks, tensors

from helpers import f64, random_vectors, rel_l2

pytestmark = pytest.mark.gpu

FP8_O_REL_L2, FP8_LSE_MAX_ABS = 4e-2, 1e-3
FP8_P_REL = 2.0 ** -4  # worst relative rounding of a normal e4m3 value
E4 = torch.float8_e4m3fn


def quantize(x):
    """Per-tensor e4m3 quantization: (stored tensor, scale) with value = stored x scale."""
    amax = float(x.float().abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    return (x.float() / scale).to(E4), scale


def _run(vec, B, hq, hkv, n, causal, d=128):
    scale = d ** -0.5
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d)
    q, k, v, _ = tensors.make_qkvdo(cfg)
    (q8, sq), (k8, sk), (v8, sv) = quantize(q), quantize(k), quantize(v)
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv, causal=causal)
    o, lse = fm.fm_attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), *dv, qs, q_scale=sq, k_scale=sk, v_scale=sv,
                                scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    deq = lambda t, s: t.double().numpy() * s
    vdq = deq(v8, sv)
    O_ref, L_ref = oracle.forward(deq(q8, sq), deq(k8, sk), vdq, vec, causal, scale)
    return f64(o), f64(lse), O_ref, L_ref, FP8_P_REL * float(np.abs(vdq).max()) + 1e-2


def _check(o, lse, O, L, max_abs):
    inf = np.isneginf(L)
    assert np.array_equal(np.isneginf(lse), inf), "fully-masked rows differ"
    assert (o[np.broadcast_to(inf[..., None], o.shape)] == 0).all()
    if (~inf).any():
        assert np.abs(lse[~inf] - L[~inf]).max() <= FP8_LSE_MAX_ABS
    r = rel_l2(o, O)
    m = float(np.abs(o - O).max())
    assert r <= FP8_O_REL_L2 and m <= max_abs, f"O rel-L2 {r:.3e} max-abs {m:.3e} (bound {max_abs:.3e})"


def test_fp8_tiny_workload_at_d128():
    cfg = configs.make("tiny", d=128)
    _check(*_run(tuple(cfg[x] for x in ("lts", "lte", "uts", "ute")), 1, 2, 2, cfg["N"], True))


@pytest.mark.parametrize("hq,hkv", [(1, 1), (2, 1), (4, 2), (6, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_random_masks(hq, hkv, causal):
    rng = np.random.default_rng(800 + 10 * hq + hkv + causal)
    for n in (128, 384):
        _check(*_run(random_vectors(rng, 1, n, "general"), 1, hq, hkv, n, causal))


@pytest.mark.parametrize("n", [1, 100, 300, 389])
def test_fp8_ragged_n(n):
    rng = np.random.default_rng(n + 800)
    _check(*_run(random_vectors(rng, 2, n, "lower"), 2, 4, 2, n, True))


@pytest.mark.parametrize("kind", ["docs", "share_question", "prefix_lm", "window", "eviction"])
def test_fp8_mask_families_2k(kind):
    rng = np.random.default_rng(17)
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
    _check(*_run(tuple(x[None] for x in v), 1, 4, 2, n, causal))


def test_fp8_rejects_other_head_dims_and_bad_scales():
    cfg = dict(B=1, H_q=2, H_kv=1, N=128, d=64)
    q, k, v, _ = tensors.make_qkvdo(cfg)
    vec = [torch.zeros(1, 128, dtype=torch.int32, device="cuda") for _ in range(4)]
    qs = fm.fm_classify_tiles(*vec, causal=True)
    q8, k8, v8 = (quantize(x)[0].cuda() for x in (q, k, v))
    with pytest.raises(fm.FMError):
        fm.fm_attn_fwd_fp8(q8, k8, v8, *vec, qs, q_scale=1.0, k_scale=1.0, v_scale=1.0, scale=0.1, causal=True)
    cfg["d"] = 128
    q, k, v, _ = tensors.make_qkvdo(cfg)
    q8, k8, v8 = (quantize(x)[0].cuda() for x in (q, k, v))
    with pytest.raises(fm.FMError):
        fm.fm_attn_fwd_fp8(q8, k8, v8, *vec, qs, q_scale=0.0, k_scale=1.0, v_scale=1.0, scale=0.1, causal=True)
