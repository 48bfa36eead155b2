"""Launch-order paths of the forward and backward passes.

Both passes choose a launch order on the device: longest queue first (a rank
sort up to 1024 work units, a bitonic sort up to 4096) for passes of a few
waves, natural order for long passes. Every path must visit every work unit
exactly once, so a batched call must reproduce the per-batch-entry calls
(which take other order paths): bit for bit where each output element is
written by one CTA (O, LSE, dK, dV), within the dQ tolerance where the fp32
accumulation order differs (dQ).
"""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
from workloads import masks, tensors

from helpers import GRAD_REL_L2, f64, rel_l2

pytestmark = pytest.mark.gpu


def _vectors(B, n, seed):
    rng = np.random.default_rng(seed)
    vs = [masks.causal_documents(masks.draw_fill(rng, n, 256, 1024), n) for _ in range(B)]
    return tuple(np.stack([v[i] for v in vs]).astype(np.int32) for i in range(4))


def _run(vec_np, cfg, q, k, v, do):
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    qs = fm.fm_classify_tiles(*vec, causal=True)
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=cfg["scale"], causal=True)
    dq, dk, dv = fm.fm_attn_bwd(q, k, v, o, lse, do, *vec, qs, scale=cfg["scale"], causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    return o, lse, dq, dk, dv


def test_batched_bitonic_order_matches_per_entry_calls():
    # B * nQ = 1152 work units (above the rank-sort limit), 1152 CTAs per pass
    # (below eight waves): both passes sort with the bitonic network
    B, n = 9, 16384
    cfg = dict(B=B, H_q=2, H_kv=1, N=n, d=128, scale=128 ** -0.5)
    q, k, v, do = (t.cuda() for t in tensors.make_qkvdo(cfg))
    vec_np = _vectors(B, n, 21)
    o, lse, dq, dk, dv = _run(vec_np, cfg, q, k, v, do)
    for b in range(B):
        one = dict(cfg, B=1)
        sl = slice(b, b + 1)
        ob, lseb, dqb, dkb, dvb = _run(tuple(x[sl] for x in vec_np), one, q[sl].contiguous(), k[sl].contiguous(),
                                       v[sl].contiguous(), do[sl].contiguous())
        assert torch.equal(o[sl], ob) and torch.equal(lse[sl], lseb)
        assert torch.equal(dk[sl], dkb) and torch.equal(dv[sl], dvb)
        assert rel_l2(f64(dq[sl]), f64(dqb)) <= GRAD_REL_L2
