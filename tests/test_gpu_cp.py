"""Rectangular problems (N query rows against N_kv keys) against the oracle,
and a context-parallel split emulated on one GPU (FlashMask-3 project page,
§3.2-3.4): the balancer deals the query chunks to ranks, each rank's vectors
are localized to its rows by fm_localize, each rank gets only the K / V chunks
its rows can see (the others zero) and runs the forward and backward on its own
rows against the keys, and the ranks' outputs and summed key gradients match
the whole problem."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import tensors

from helpers import assert_grad, assert_lse, assert_out, f64
from test_cp_oracle import cases

pytestmark = pytest.mark.gpu


def inputs(B, hq, hkv, n, nk, d, seed=20):
    q = tensors.randn_bf16((B, hq, n, d), seed)
    k = tensors.randn_bf16((B, hkv, nk, d), seed + 1)
    v = tensors.randn_bf16((B, hkv, nk, d), seed + 2)
    do = tensors.randn_bf16((B, hq, n, d), seed + 3)
    return q, k, v, do


def rect_vectors(rng, B, n_rows, n_keys):
    out = []
    for _ in range(B):
        a = rng.integers(0, n_rows + 1, size=(2, n_keys))
        c = rng.integers(0, n_rows + 1, size=(2, n_keys))
        out.append((a.min(0), a.max(0), c.min(0), c.max(0)))
    return tuple(np.stack(x).astype(np.int32) for x in zip(*out))


@pytest.mark.parametrize("n,nk,d,hq,hkv,causal", [
    (640, 1000, 128, 4, 2, False),
    (1300, 384, 64, 2, 1, True),
    (384, 1300, 128, 2, 2, True),
    (200, 2048, 128, 4, 1, False),
])
def test_rectangular_matches_oracle(n, nk, d, hq, hkv, causal):
    rng = np.random.default_rng(n + nk)
    B = 2
    vec = rect_vectors(rng, B, n, nk)
    q, k, v, do = inputs(B, hq, hkv, n, nk, d)
    dv_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv_, causal=causal, n_rows=n)
    cls_ref = np.stack([oracle.classify_tiles(*(x[b] for x in vec), causal, 128, 128, n_rows=n) for b in range(B)])
    assert np.array_equal(qs.tile_class.cpu().numpy(), cls_ref)
    scale = d ** -0.5
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *dv_, qs, scale=scale, causal=causal)
    dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *dv_, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vec, causal, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec, causal, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


@pytest.mark.parametrize("name", ["doc_causal_folded", "prefix_lm", "general"])
def test_cp_split_on_one_gpu(name):
    n, C, P, kappa, d, hq, hkv = 4096, 512, 4, 2, 128, 4, 2
    vec = tuple(np.asarray(x, np.int32) for x in cases(n)[name])
    vb = tuple(x[None] for x in vec)
    q, k, v, do = inputs(1, hq, hkv, n, n, d, seed=30)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    scale = d ** -0.5
    gvec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vb]
    qs = fm.fm_classify_tiles(*gvec, causal=False)
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *gvec, qs, scale=scale, causal=False)
    dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *gvec, qs, scale=scale, causal=False)
    # deal the chunks of C rows (C / 128 Q blocks each) to P ranks, kappa each
    w = fm.fm_chunk_loads(qs.tile_class, C // 128, 13, 10)
    owner, rep = fm.fm_balance_chunks(w, P, kappa)
    assert np.bincount(owner, minlength=P).tolist() == [kappa] * P
    # each rank receives only the K / V chunks its rows can see (mask-aware
    # pruning of the exchange); the chunks it does not receive stay zero
    need = fm.fm_needed_chunks(qs.tile_class, owner, P, C // 128)
    flat = torch.cat([x.reshape(-1) for x in gvec])
    dk_sum = torch.zeros_like(dk, dtype=torch.float32)
    dv_sum = torch.zeros_like(dv, dtype=torch.float32)
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vb, False, scale)
    dQ_ref, dK_ref, dV_ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vb, False, scale)
    same = 0
    for r in range(P):
        chunks = np.sort(np.nonzero(owner == r)[0])
        rows = np.concatenate([np.arange(c * C, (c + 1) * C) for c in chunks])
        off = torch.from_numpy((chunks * C).astype(np.int32)).cuda()
        loc = fm.fm_localize(flat, off, C).view(4, 1, n)
        lvec = [loc[i].contiguous() for i in range(4)]
        tr = torch.from_numpy(rows).cuda()
        q_r = qd[:, :, tr].contiguous()
        do_r = dod[:, :, tr].contiguous()
        keep = torch.from_numpy(np.repeat(need[r].astype(bool), C)).cuda()
        k_r = torch.where(keep[None, None, :, None], kd, torch.zeros_like(kd))
        v_r = torch.where(keep[None, None, :, None], vd, torch.zeros_like(vd))
        qs_r = fm.fm_classify_tiles(*lvec, causal=False, n_rows=len(rows))
        o_r, lse_r = fm.fm_attn_fwd(q_r, k_r, v_r, *lvec, qs_r, scale=scale, causal=False)
        dq_r, dk_r, dv_r = fm.fm_attn_bwd(q_r, k_r, v_r, o_r, lse_r, do_r, *lvec, qs_r, scale=scale, causal=False)
        st, bits = fm.fm_device_status()
        assert st == fm.FM_OK, bits
        assert_out(f64(o_r), O_ref[:, :, rows])
        assert_lse(f64(lse_r), L_ref[:, :, rows])
        assert_grad(f64(dq_r), dQ_ref[:, :, rows], "dQ")
        # the rank's tiles are the whole run's tiles of the same rows, and any
        # tile only one of the two classifications skips is fully masked (it
        # adds exact zeros), so O matches bit for bit
        same += int(torch.equal(o_r, o[:, :, tr]))
        dk_sum += dk_r.float()
        dv_sum += dv_r.float()
    assert_grad(f64(dk_sum), dK_ref, "dK")
    assert_grad(f64(dv_sum), dV_ref, "dV")
    assert same == P


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("n,nk", [(1, 1), (1, 300), (300, 1), (129, 1), (1, 129), (2, 257)])
def test_extreme_rectangular_shapes(n, nk, d):
    # one query row or one key, and blocks of a single row or key on either axis
    rng = np.random.default_rng(7 * n + nk + d)
    B, hq, hkv = 2, 2, 1
    for causal in (False, True):
        vec = rect_vectors(rng, B, n, nk)
        q, k, v, do = inputs(B, hq, hkv, n, nk, d, seed=30)
        dv_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
        qs = fm.fm_classify_tiles(*dv_, causal=causal, n_rows=n)
        scale = d ** -0.5
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        o, lse = fm.fm_attn_fwd(qd, kd, vd, *dv_, qs, scale=scale, causal=causal)
        dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *dv_, qs, scale=scale, causal=causal)
        st, bits = fm.fm_device_status()
        assert st == fm.FM_OK, bits
        O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vec, causal, scale)
        assert_out(f64(o), O_ref)
        assert_lse(f64(lse), L_ref)
        ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec, causal, scale)
        for name, x, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert_grad(f64(x), r, name)
