"""Per-head mask vectors (B, H_q, N_kv) through the native per-head entry
points (fm_attn_fwd_heads / fm_attn_bwd_heads) against the fp64 oracle run
with one set of vectors per query head.

The FlashMask Guide ("The Solution: FlashMask Sparse Mask Representation")
defines the four vectors per sample; a mask that differs by head is the same
column-wise representation one level finer, and every head's attention is
that head's own masked softmax: the oracle evaluates exactly that.
"""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import masks, tensors

from helpers import assert_grad, assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu


def _general_heads(rng, B, hq, n):
    a = rng.integers(0, n + 1, size=(2, B, hq, n))
    c = rng.integers(0, n + 1, size=(2, B, hq, n))
    return tuple(x.astype(np.int32) for x in (a.min(0), a.max(0), c.min(0), c.max(0)))


def _family_heads(rng, B, hq, n):
    """A different mask family per head: documents, share-question, window,
    eviction, fully visible (empty vectors), and a head whose every row is
    masked (LTS = 0, LTE = N)."""
    fams = []
    for h in range(hq):
        kind = h % 6
        if kind == 0:
            v = masks.causal_documents(masks.draw_fill(rng, n, 40, 300), n)
        elif kind == 1:
            v = masks.share_question([(n // 5, n // 10, n // 8), (n // 4, n // 7, n // 6)], n)
        elif kind == 2:
            v = masks.sliding_window(n, 97, 3)
        elif kind == 3:
            v = masks.random_eviction(n, 1 / 32, rng)
        elif kind == 4:
            v = masks._empty(n)
        else:
            v = (np.zeros(n, np.int32), np.full(n, n, np.int32), np.zeros(n, np.int32), np.zeros(n, np.int32))
        fams.append(tuple(np.asarray(x, np.int32) for x in v))
    one = tuple(np.stack([f[i] for f in fams]) for i in range(4))   # (hq, n)
    return tuple(np.ascontiguousarray(np.broadcast_to(x[None], (B,) + x.shape)) for x in one)


def _run(heads, B, hq, hkv, n, d, causal, backward=True):
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d)
    q, k, v, do = tensors.make_qkvdo(cfg)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    vec = [torch.from_numpy(x).cuda() for x in heads]
    scale = d ** -0.5
    out = fm.fm_attn_per_head(qd, kd, vd, *vec, causal=causal, scale=scale, do=dod if backward else None)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"heads": heads}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, causal, scale)
    assert_out(f64(out[0]), O_ref)
    assert_lse(f64(out[1]), L_ref)
    if backward:
        ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, causal, scale)
        for name, x, r in zip(("dQ", "dK", "dV"), out[2:], ref):
            assert_grad(f64(x), r, name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,hq,hkv,n,d", [(2, 4, 2, 700, 128), (1, 1, 1, 300, 64), (1, 6, 2, 389, 128),
                                          (2, 8, 1, 1000, 64), (1, 4, 2, 389, 256), (2, 2, 1, 600, 256)])
def test_per_head_random_masks(B, hq, hkv, n, d, causal):
    rng = np.random.default_rng(9 + hq + n)
    _run(_general_heads(rng, B, hq, n), B, hq, hkv, n, d, causal)


@pytest.mark.parametrize("hq,hkv,d", [(6, 1, 128), (6, 3, 128), (6, 2, 256)])
def test_per_head_mask_families(hq, hkv, d):
    rng = np.random.default_rng(31)
    n = 1500
    _run(_family_heads(rng, 2, hq, n), 2, hq, hkv, n, d, True)


def test_per_head_group_of_64_overflows_the_staged_queue():
    # 64 query heads per kv head and 18 Q blocks: a KV block's queues hold up
    # to 64 x 18 = 1152 entries, more than the 1024 staged in shared memory
    rng = np.random.default_rng(64)
    n = 2200
    heads = _general_heads(rng, 1, 64, n)
    heads = (heads[0] // 4, heads[1] // 4, heads[2], heads[2])  # mostly visible, upper interval empty
    _run(heads, 1, 64, 1, n, 64, True)


def test_per_head_d256_overflows_the_staged_queue():
    # d = 256 stages 128 queue entries per KV block: 8 query heads per kv head
    # and 18 Q blocks give up to 8 x 18 = 144
    rng = np.random.default_rng(256)
    n = 2200
    heads = _general_heads(rng, 1, 8, n)
    heads = (heads[0] // 4, heads[1] // 4, heads[2], heads[2])
    _run(heads, 1, 8, 1, n, 256, True)


@pytest.mark.parametrize("d", [128, 256])
def test_repeated_vectors_match_the_shared_path(d):
    # per-head vectors that repeat one mask: each head's arithmetic is the
    # shared path's (same tiles, same order), so O, LSE, dK and dV agree bit for
    # bit; dQ is summed with fp32 reduce-adds whose order between CTAs is free
    rng = np.random.default_rng(77)
    B, hq, hkv, n = 2, 4, 2, 1100
    v1 = masks.causal_documents(masks.draw_fill(rng, n, 100, 500), n)
    shared = [torch.from_numpy(np.ascontiguousarray(np.broadcast_to(np.asarray(x, np.int32), (B, n)))).cuda()
              for x in v1]
    per = [x[:, None].expand(B, hq, n).contiguous() for x in shared]
    q, k, v, do = (x.cuda() for x in tensors.make_qkvdo(dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d)))
    s = d ** -0.5
    qs = fm.fm_classify_tiles(*shared, causal=True)
    o1, l1 = fm.fm_attn_fwd(q, k, v, *shared, qs, scale=s, causal=True)
    dq1, dk1, dv1 = fm.fm_attn_bwd(q, k, v, o1, l1, do, *shared, qs, scale=s, causal=True)
    o2, l2, dq2, dk2, dv2 = fm.fm_attn_per_head(q, k, v, *per, causal=True, scale=s, do=do)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 2e-2 * dq1.float().abs().max().item()


def test_per_head_refuses_unsupported_shapes():
    n = 128
    vec = [torch.zeros(1, 65, n, dtype=torch.int32, device="cuda") for _ in range(4)]
    q = torch.zeros(1, 65, n, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, n, 64, dtype=torch.bfloat16, device="cuda")
    do, o = torch.zeros_like(q), torch.zeros_like(q)
    lse = torch.zeros(1, 65, n, dtype=torch.float32, device="cuda")
    # at most 64 query heads per kv head (the backward stages one queue per head)
    qs = fm.fm_classify_tiles_heads(*vec, causal=True)
    with pytest.raises(fm.FMError):
        fm.fm_attn_fwd_heads(q, k, k, *vec, qs, scale=0.125, causal=True)
    with pytest.raises(fm.FMError):
        fm.fm_attn_bwd_heads(q, k, k, o, lse, do, *vec, qs, scale=0.125, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits


@pytest.mark.parametrize("n,nk,d,hq,hkv,causal", [(600, 900, 128, 4, 2, False), (900, 384, 64, 2, 1, True),
                                                  (700, 500, 256, 2, 1, True)])
def test_per_head_rectangular(n, nk, d, hq, hkv, causal):
    # N query rows against N_kv keys (the shape of one context-parallel rank),
    # with per-head vectors of N_kv entries and values in [0, N]
    rng = np.random.default_rng(n + nk)
    B = 2
    a = rng.integers(0, n + 1, size=(2, B, hq, nk))
    c = rng.integers(0, n + 1, size=(2, B, hq, nk))
    heads = tuple(x.astype(np.int32) for x in (a.min(0), a.max(0), c.min(0), c.max(0)))
    q = tensors.randn_bf16((B, hq, n, d), 41)
    k = tensors.randn_bf16((B, hkv, nk, d), 42)
    v = tensors.randn_bf16((B, hkv, nk, d), 43)
    do = tensors.randn_bf16((B, hq, n, d), 44)
    vec = [torch.from_numpy(x).cuda() for x in heads]
    scale = d ** -0.5
    o, lse, dq, dk, dv = fm.fm_attn_per_head(q.cuda(), k.cuda(), v.cuda(), *vec, causal=causal, scale=scale,
                                             do=do.cuda())
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"heads": heads}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, causal, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, causal, scale)
    for name, x, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(x), r, name)
