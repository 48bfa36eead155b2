"""fm_from_fms_fme against the oracle, bit for bit, and the FlashMask Guide's
DPO mask through the whole path (FlashMask Guide, "The Solution: FlashMask
Sparse Mask Representation" and "Real-World Attention Mask Topologies")."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import tensors

from helpers import assert_grad, assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,offset", [((2, 1003), 0), ((3, 512), 1), ((1, 7), 0)])
def test_from_fms_fme_matches_oracle(shape, offset):
    rng = np.random.default_rng(shape[1] + offset)
    n = shape[1]
    m = int(np.prod(shape))
    fms = rng.integers(-3, n + 4, size=m + offset).astype(np.int32)
    fme = rng.integers(-3, n + 4, size=m + offset).astype(np.int32)
    # offset 1: inputs that are not 16-byte aligned take the element-wise path
    a = torch.from_numpy(fms).cuda()[offset:].view(shape)
    b = torch.from_numpy(fme).cuda()[offset:].view(shape)
    got = fm.fm_from_fms_fme(a, b, n_rows=n)
    ref = oracle.from_fms_fme(fms[offset:], fme[offset:], n)
    for g, r in zip(got, ref):
        assert np.array_equal(g.cpu().numpy().reshape(-1), r)


def test_guide_dpo_mask_end_to_end():
    # one DPO sample as the Guide writes it: prompt keys visible to every later
    # row, chosen keys to chosen rows, rejected keys to rejected rows
    P, Cc, R = 700, 500, 848
    n, d, hq, hkv = P + Cc + R, 128, 4, 2
    fms = np.arange(n)
    fme = np.empty(n, np.int64)
    fme[:P] = n - 1
    fme[P:P + Cc] = P + Cc - 1
    fme[P + Cc:] = n - 1
    t = lambda x: torch.from_numpy(x.astype(np.int32)[None]).cuda()  # noqa: E731
    vec = fm.fm_from_fms_fme(t(fms), t(fme))
    vec_np = oracle.from_fms_fme(fms[None], fme[None], n)
    cfg = dict(B=1, H_q=hq, H_kv=hkv, N=n, d=d)
    q, k, v, do = tensors.make_qkvdo(cfg)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    scale = d ** -0.5
    qs = fm.fm_classify_tiles(*vec, causal=False)
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *vec, qs, scale=scale, causal=False)
    dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *vec, qs, scale=scale, causal=False)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), vec_np, False, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec_np, False, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


def disjoint_intervals(rng, M, B, n_rows, n_keys):
    """(M, B, N_kv) inclusive intervals, disjoint and ascending per column
    (some empty: end < start)."""
    cuts = np.sort(rng.integers(0, n_rows + 1, size=(2 * M, B, n_keys)), axis=0)
    return cuts[0::2].astype(np.int32), (cuts[1::2] - 1).astype(np.int32)


@pytest.mark.parametrize("M,n,nk,d,hq,hkv,B", [
    (3, 1000, 1000, 128, 4, 2, 2), (2, 640, 1300, 64, 2, 1, 2), (4, 512, 512, 128, 2, 2, 2),
    (2, 700, 700, 256, 4, 2, 2), (4, 389, 389, 256, 2, 1, 2), (1, 600, 600, 128, 2, 1, 2),
    # past the staged queues: the forward's unit ring holds 512 entries (M x nK
    # = 4 x 133), the backward stages 1024 per KV block at d <= 128 (4 x 258)
    # and 128 at d = 256 (4 x 36)
    (4, 300, 17000, 64, 1, 1, 1), (4, 33000, 256, 64, 1, 1, 1), (4, 4500, 300, 256, 1, 1, 1)])
def test_multi_interval_matches_oracle(M, n, nk, d, hq, hkv, B):
    # one forward and one backward launch over every interval (each block
    # masked with its own interval's vectors) against the oracle's direct
    # evaluation of the union of the intervals
    rng = np.random.default_rng(M * 1000 + n)
    fms, fme = disjoint_intervals(rng, M, B, n, nk)
    q = tensors.randn_bf16((B, hq, n, d), 40)
    k = tensors.randn_bf16((B, hkv, nk, d), 41)
    v = tensors.randn_bf16((B, hkv, nk, d), 42)
    do = tensors.randn_bf16((B, hq, n, d), 43)
    scale = d ** -0.5
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse, dq, dk, dv = fm.fm_attn_multi_interval(qd, kd, vd, torch.from_numpy(fms).cuda(),
                                                   torch.from_numpy(fme).cuda(), scale=scale, do=dod)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"fms": fms.transpose(1, 0, 2), "fme": fme.transpose(1, 0, 2)}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, False, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, False, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


def test_merge_and_sum_of_one_part_are_identities():
    rng = np.random.default_rng(5)
    o = torch.from_numpy(rng.standard_normal((3, 77, 64)).astype(np.float32)).to(torch.bfloat16).cuda()
    lse = torch.from_numpy(rng.standard_normal((3, 77)).astype(np.float32)).cuda()
    lse[0, :5] = -float("inf")
    om, lm = fm.fm_merge_parts([o], [lse])
    assert torch.equal(lm, lse)
    assert torch.equal(om[lse != -float("inf")], o[lse != -float("inf")])
    assert (om[lse == -float("inf")] == 0).all()
    x = torch.from_numpy(rng.standard_normal(1001).astype(np.float32)).to(torch.bfloat16).cuda()
    assert torch.equal(fm.fm_sum_parts([x]), x)
    assert torch.equal(fm.fm_sum_parts([x[1:], x[1:]]), (2 * x[1:].float()).to(torch.bfloat16))


@pytest.mark.parametrize("d", [128, 256])
def test_multi_interval_entry_points_with_causal(d):
    # fm_classify_tiles_multi / fm_attn_fwd_multi / fm_attn_bwd_multi called
    # directly with the causal flag: the causal term masks i < j on top of the
    # intervals (the oracle applies it the same way)
    rng = np.random.default_rng(d + 3)
    M, B, hq, hkv, n = 3, 2, 4, 2, 700
    fms, fme = disjoint_intervals(rng, M, B, n, n)
    q = tensors.randn_bf16((B, hq, n, d), 50)
    k = tensors.randn_bf16((B, hkv, n, d), 51)
    v = tensors.randn_bf16((B, hkv, n, d), 52)
    do = tensors.randn_bf16((B, hq, n, d), 53)
    scale = d ** -0.5
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    fms_t, fme_t = torch.from_numpy(fms).cuda(), torch.from_numpy(fme).cuda()
    qs = fm.fm_classify_tiles_multi(fms_t, fme_t, causal=True, n_rows=n)
    o, lse = fm.fm_attn_fwd_multi(qd, kd, vd, fms_t, fme_t, qs, scale=scale, causal=True)
    dq, dk, dv = fm.fm_attn_bwd_multi(qd, kd, vd, o, lse, dod, fms_t, fme_t, qs, scale=scale, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"fms": fms.transpose(1, 0, 2), "fme": fme.transpose(1, 0, 2)}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, True, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, True, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("M,n,nk", [(1, 700, 700), (3, 1000, 640), (4, 389, 1300)])
def test_multi_interval_classification_matches_oracle(M, n, nk, causal):
    # union classes (the most visible of the run slots' own classes) and both
    # queues, bit for bit, on overlapping, empty and out-of-range intervals
    rng = np.random.default_rng(M * 31 + n + causal)
    B = 2
    fms = rng.integers(-3, n + 3, size=(M, B, nk)).astype(np.int32)
    fme = rng.integers(-3, n + 3, size=(M, B, nk)).astype(np.int32)
    qs = fm.fm_classify_tiles_multi(torch.from_numpy(fms).cuda(), torch.from_numpy(fme).cuda(), causal=causal,
                                    n_rows=n)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    cls_ref = [oracle.classify_tiles_multi(fms[:, b], fme[:, b], causal, 128, 128, n) for b in range(B)]
    assert np.array_equal(qs.tile_class.cpu().numpy(), np.stack(cls_ref))
    q_off, q_queue, k_off, k_queue = oracle.build_queues(cls_ref)
    assert np.array_equal(qs.q_off.cpu().numpy(), q_off)
    assert np.array_equal(qs.k_off.cpu().numpy(), k_off)
    assert np.array_equal(qs.q_queue.cpu().numpy()[:len(q_queue)], q_queue)
    assert np.array_equal(qs.k_queue.cpu().numpy()[:len(k_queue)], k_queue)


@pytest.mark.parametrize("causal", [False, True])
def test_multi_interval_classes_of_a_cut_interval(causal):
    # one visible interval per column [j, L_j] (a causal-document-like mask)
    # cut into touching, swapped and overlapping pieces: the kernel's classes
    # and queues equal the oracle's, which equal the uncut interval's
    rng = np.random.default_rng(77 + causal)
    B, n = 2, 1500
    j = np.arange(n)[None, :]
    ends = np.minimum(j + rng.integers(0, 600, size=(B, 1)) + (j % 97), n - 1)
    mid = (j + ends) // 2
    one = [oracle.classify_tiles(*oracle.from_fms_fme(np.broadcast_to(j, (B, n))[b], ends[b], n), causal, 128, 128,
                                 n_rows=n) for b in range(B)]
    for fms, fme in ((np.stack([np.broadcast_to(j, (B, n)), mid + 1]), np.stack([mid, ends])),
                     (np.stack([mid + 1, np.broadcast_to(j, (B, n))]), np.stack([ends, mid])),
                     (np.stack([np.broadcast_to(j, (B, n)), np.maximum(mid - 5, j), mid]),
                      np.stack([mid, ends, np.minimum(mid + 3, ends)]))):
        fms, fme = np.ascontiguousarray(fms, np.int32), np.ascontiguousarray(fme, np.int32)
        qs = fm.fm_classify_tiles_multi(torch.from_numpy(fms).cuda(), torch.from_numpy(fme).cuda(), causal=causal,
                                        n_rows=n)
        st, bits = fm.fm_device_status()
        assert st == fm.FM_OK, bits
        cls_ref = [oracle.classify_tiles_multi(fms[:, b], fme[:, b], causal, 128, 128, n) for b in range(B)]
        assert all(np.array_equal(c, o) for c, o in zip(cls_ref, one))
        assert np.array_equal(qs.tile_class.cpu().numpy(), np.stack(cls_ref))
        q_off, q_queue, k_off, k_queue = oracle.build_queues(cls_ref)
        assert np.array_equal(qs.q_off.cpu().numpy(), q_off)
        assert np.array_equal(qs.q_queue.cpu().numpy()[:len(q_queue)], q_queue)
        assert np.array_equal(qs.k_queue.cpu().numpy()[:len(k_queue)], k_queue)


@pytest.mark.parametrize("d,causal", [(128, False), (64, True), (256, False)])
def test_multi_interval_overlapping_intervals(d, causal):
    # overlapping visible intervals: a key is visible to the union of its
    # intervals (each block computed once, masked by the union)
    rng = np.random.default_rng(d + 7 + causal)
    M, B, hq, hkv, n = 3, 2, 4, 2, 650
    a = rng.integers(0, n, size=(M, B, n))
    w = rng.integers(0, n // 2, size=(M, B, n))
    fms, fme = a.astype(np.int32), np.minimum(a + w, n - 1).astype(np.int32)
    q = tensors.randn_bf16((B, hq, n, d), 60)
    k = tensors.randn_bf16((B, hkv, n, d), 61)
    v = tensors.randn_bf16((B, hkv, n, d), 62)
    do = tensors.randn_bf16((B, hq, n, d), 63)
    scale = d ** -0.5
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse, dq, dk, dv = fm.fm_attn_multi_interval(qd, kd, vd, torch.from_numpy(fms).cuda(),
                                                   torch.from_numpy(fme).cuda(), scale=scale, do=dod, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"fms": fms.transpose(1, 0, 2), "fme": fme.transpose(1, 0, 2)}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, causal, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, causal, scale)
    for name, a_, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a_), r, name)
