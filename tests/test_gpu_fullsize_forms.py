"""Per-head and multi-interval masks at the full share-question / DPO 32K size
(B = 1, H_q = 32, H_kv = 8, N = 32768, d = 128), in the launch configuration
of the benchmark's compositions, checked the way the shared-vector full-size
test checks its workloads (tests/test_gpu_fullsize.py):
  * O, LSE and dQ on every row of two seeded query heads;
  * dK and dV of a <= 4-head group slice (the same kernels on the same N, mask
    and data with the query heads cut to the slice) on every key column of the
    two KV blocks with the longest backward queues.
Per-head vectors: every query head packs its own eight samples (prompt and
response lengths drawn per head), so the heads' masks and queues differ.
Multi-interval: the workload's own mask with each key column's visible rows
[j, LTS_j) written as two inclusive intervals split at their midpoint.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, masks, tensors

from helpers import assert_grad, assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu
_POOL = 16


def _rows(qh, kh, vh, doh, spec, causal, scale, rows):
    segs = [s for s in np.array_split(rows, _POOL) if len(s)]

    def one(r):
        O, L = oracle.forward(qh, kh, vh, spec, causal, scale, rows=r, visible_only=True)
        dQ, _, _ = oracle.backward(qh, kh, vh, doh, spec, causal, scale, rows=r, cols=np.array([], dtype=np.int64),
                                   visible_only=True)
        return O, L, dQ

    with ThreadPoolExecutor(len(segs)) as ex:
        parts = list(ex.map(one, segs))
    return tuple(np.concatenate([p[i] for p in parts], axis=2) for i in range(3))


def _key_grads(q, k, v, do, spec_of_head, causal, scale, cols):
    """dK, dV of `cols` summed over the heads of q (spec_of_head(h): that head's mask)."""
    def one(h):
        _, dK, dV = oracle.backward(q[:, h:h + 1], k, v, do[:, h:h + 1], spec_of_head(h), causal, scale,
                                    rows=np.array([], dtype=np.int64), cols=cols, visible_only=True)
        return dK, dV

    with ThreadPoolExecutor(q.shape[1]) as ex:
        parts = list(ex.map(one, range(q.shape[1])))
    return sum(p[0] for p in parts), sum(p[1] for p in parts)


def _heavy_columns(k_off, rows_per_kb, nK, n, count=2):
    """Every key column of the `count` KV blocks whose queues (summed over the
    queue rows that feed one CTA) are longest."""
    lens = np.diff(k_off.cpu().numpy().astype(np.int64)).reshape(rows_per_kb, nK).sum(0)
    top = np.sort(np.argsort(-lens, kind="stable")[:count])
    return np.concatenate([np.arange(kb * 128, min((kb + 1) * 128, n)) for kb in top]), lens[top]


def test_full_size_per_head():
    cfg = configs.make("share_question32k")
    B, Hq, Hkv, N, d = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], cfg["d"]
    G = Hq // Hkv
    scale, causal = cfg["scale"], cfg["causal"]
    per = []
    for h in range(Hq):
        v_h = masks.share_question(masks.draw_share_question(np.random.default_rng(1000 + h)), N)
        per.append(tuple(np.asarray(x, np.int32) for x in v_h))
    vec_np = tuple(np.stack([p[i] for p in per])[None] for i in range(4))  # (1, H_q, N)
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device="cuda")
    o, lse, dq, dk, dv = fm.fm_attn_per_head(q, k, v, *vec, causal=causal, scale=scale, do=do)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    rng = np.random.default_rng(321)
    rows = np.arange(N)
    for h in sorted(rng.choice(Hq, size=2, replace=False).tolist()):
        g = h // G
        spec = {"heads": tuple(x[:, h:h + 1] for x in vec_np)}
        O_ref, L_ref, dQ_ref = _rows(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]),
                                     f64(do[:, h:h + 1]), spec, causal, scale, rows)
        assert_out(f64(o[:, h:h + 1]), O_ref)
        assert_lse(f64(lse[:, h:h + 1]), L_ref)
        assert_grad(f64(dq[:, h:h + 1]), dQ_ref, f"dQ[per-head h{h}]")
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    # group slice
    g0 = int(rng.integers(Hkv))
    hsel = g0 * G + np.sort(rng.choice(G, size=min(4, G), replace=False))
    th = torch.as_tensor(hsel, device="cuda")
    qs_, dos_ = q[:, th].contiguous(), do[:, th].contiguous()
    ks_, vs_ = k[:, g0:g0 + 1].contiguous(), v[:, g0:g0 + 1].contiguous()
    vsub = [x[:, th].contiguous() for x in vec]
    queues = fm.fm_classify_tiles_heads(*vsub, causal=causal)
    o_s, lse_s = fm.fm_attn_fwd_heads(qs_, ks_, vs_, *vsub, queues, scale=scale, causal=causal)
    _, dk_s, dv_s = fm.fm_attn_bwd_heads(qs_, ks_, vs_, o_s, lse_s, dos_, *vsub, queues, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    nK = N // 128
    cols, qlen = _heavy_columns(queues.k_off, len(hsel), nK, N)
    vsub_np = tuple(x[:, hsel] for x in vec_np)
    dK_ref, dV_ref = _key_grads(f64(qs_), f64(ks_), f64(vs_), f64(dos_),
                                lambda h: {"heads": tuple(x[:, h:h + 1] for x in vsub_np)}, causal, scale, cols)
    tc = torch.as_tensor(cols, device="cuda")
    assert_grad(f64(dk_s[:, :, tc]), dK_ref, f"dK[per-head, KV blocks with queues of {qlen.tolist()} units]")
    assert_grad(f64(dv_s[:, :, tc]), dV_ref, f"dV[per-head, KV blocks with queues of {qlen.tolist()} units]")


def test_full_size_multi_interval():
    cfg = configs.make("share_question32k")
    B, Hq, Hkv, N = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"]
    G = Hq // Hkv
    scale = cfg["scale"]
    lts = cfg["lts"].astype(np.int64)
    assert cfg["causal"] and (cfg["lte"] == N).all() and (cfg["uts"] >= cfg["ute"]).all()
    j = np.arange(N, dtype=np.int64)[None, :]
    last = np.maximum(lts - 1, j - 1)            # visible rows [j, LTS_j) -> inclusive [j, last]
    mid = (j + last) // 2
    fms = np.stack([np.broadcast_to(j, lts.shape), mid + 1]).astype(np.int32)   # (2, B, N)
    fme = np.stack([mid, last]).astype(np.int32)
    q, k, v, do = tensors.make_qkvdo(cfg, device="cuda")
    o, lse, dq, dk, dv = fm.fm_attn_multi_interval(q, k, v, torch.from_numpy(fms).cuda(),
                                                   torch.from_numpy(fme).cuda(), scale=scale, do=do)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"fms": fms.transpose(1, 0, 2), "fme": fme.transpose(1, 0, 2)}
    rng = np.random.default_rng(654)
    rows = np.arange(N)
    for h in sorted(rng.choice(Hq, size=2, replace=False).tolist()):
        g = h // G
        O_ref, L_ref, dQ_ref = _rows(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]),
                                     f64(do[:, h:h + 1]), spec, False, scale, rows)
        assert_out(f64(o[:, h:h + 1]), O_ref)
        assert_lse(f64(lse[:, h:h + 1]), L_ref)
        assert_grad(f64(dq[:, h:h + 1]), dQ_ref, f"dQ[multi-interval h{h}]")
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    g0 = int(rng.integers(Hkv))
    hsel = g0 * G + np.sort(rng.choice(G, size=min(4, G), replace=False))
    th = torch.as_tensor(hsel, device="cuda")
    qs_, dos_ = q[:, th].contiguous(), do[:, th].contiguous()
    ks_, vs_ = k[:, g0:g0 + 1].contiguous(), v[:, g0:g0 + 1].contiguous()
    queues = fm.fm_classify_tiles_multi(torch.from_numpy(fms).cuda(), torch.from_numpy(fme).cuda(), causal=False,
                                        n_rows=N)
    o_s, lse_s, _, dk_s, dv_s = fm.fm_attn_multi_interval(qs_, ks_, vs_, torch.from_numpy(fms).cuda(),
                                                          torch.from_numpy(fme).cuda(), scale=scale, do=dos_)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    cols, qlen = _heavy_columns(queues.k_off, B, N // 128, N)
    dK_ref, dV_ref = _key_grads(f64(qs_), f64(ks_), f64(vs_), f64(dos_), lambda h: spec, False, scale, cols)
    tc = torch.as_tensor(cols, device="cuda")
    assert_grad(f64(dk_s[:, :, tc]), dK_ref, f"dK[multi-interval, KV blocks with queues of {qlen.tolist()} units]")
    assert_grad(f64(dv_s[:, :, tc]), dV_ref, f"dV[multi-interval, KV blocks with queues of {qlen.tolist()} units]")
