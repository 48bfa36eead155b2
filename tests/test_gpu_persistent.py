"""The persistent forward's unit hand-out at scale.

With many more work units than SMs, each forward CTA walks a long sequence of
units taken from the work counter: runs of empty units (query blocks that see
no key) between non-empty ones, and for an odd GQA group single-head units
next to two-head ones. Those sequences only arise when units far outnumber
the SMs, which the small parity tests never reach. Each case checks the device
status (a stuck hand-off would end in a bounded-wait timeout), O and LSE on
sampled rows against the oracle, the exact zero / -inf output of every empty
row of every head, and that a second call reproduces the first bit for bit
(the work counter starts from zero on every call).
"""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import tensors

from helpers import assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu


def dead_zone_vectors(n, a, b):
    """Causal mask whose rows [a, b) see no key (FlashMask column intervals).

    Key columns j < a mask rows [a, b) with their upper interval; columns j in
    [a, b) mask rows [j, b) with their lower interval (rows above j are masked
    by causality). Rows from b on see every earlier column."""
    j = np.arange(n)
    lts = np.full(n, n, np.int32)
    lte = np.full(n, n, np.int32)
    uts = np.zeros(n, np.int32)
    ute = np.zeros(n, np.int32)
    before = j < a
    uts[before], ute[before] = a, b
    inside = (j >= a) & (j < b)
    lts[inside], lte[inside] = j[inside], b
    return tuple(x[None, :] for x in (lts, lte, uts, ute))


CASES = [
    # (H_q, H_kv, N, d, dead zone rows): 2048 units in natural order, 480 of them empty
    (32, 8, 16384, 128, (4096, 4096 + 30 * 128)),
    # odd group (G = 3: two-head and single-head units), d = 64, 1024 units in
    # longest-queue-first order, the empty ones last
    (24, 8, 8192, 64, (2048, 2048 + 20 * 128)),
]


@pytest.mark.parametrize("hq,hkv,n,d,zone", CASES)
def test_persistent_forward_unit_sequences(hq, hkv, n, d, zone):
    cfg = dict(B=1, H_q=hq, H_kv=hkv, N=n, d=d, causal=True)
    scale = 1.0 / np.sqrt(d)
    a, b = zone
    vec_np = dead_zone_vectors(n, a, b)
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device="cuda")
    qs = fm.fm_classify_tiles(*vec, causal=True)
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=scale, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits

    # every empty row of every head: O = 0, LSE = -inf
    assert torch.all(o[:, :, a:b] == 0).item()
    assert torch.all(torch.isneginf(lse[:, :, a:b])).item()
    assert not torch.isneginf(lse[:, :, b:]).any().item()

    # sampled rows against the oracle (around and inside the dead zone), two heads;
    # with G = 3 head 2 of a group is a single-head unit
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(n, size=48, replace=False), [0, a - 1, a, b - 1, b, n - 1]]))
    trows = torch.as_tensor(rows, device="cuda")
    G = hq // hkv
    for h in sorted({1, hq - 1}):
        g = h // G
        O_ref, L_ref = oracle.forward(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]), vec_np, True,
                                      scale, rows=rows)
        assert_out(f64(o[:, h:h + 1, trows]), O_ref)
        assert_lse(f64(lse[:, h:h + 1, trows]), L_ref)

    # a second call: same work, same bits
    o2, lse2 = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=scale, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    assert torch.equal(o, o2) and torch.equal(lse, lse2)

    # the backward on the same problem: no error, dQ of empty rows is zero
    dq, dk, dv = fm.fm_attn_bwd(q, k, v, o, lse, do, *vec, qs, scale=scale, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    assert torch.all(dq[:, :, a:b] == 0).item()


def test_persistent_forward_batches():
    """Three batch entries, each with its own dead zone: units of different
    batch entries interleave in every CTA's sequence (natural order, 1536 units)."""
    B, hq, hkv, n, d = 3, 16, 4, 8192, 128
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d, causal=True)
    scale = 1.0 / np.sqrt(d)
    zones = [(1024, 1024 + 8 * 128), (4096, 4096 + 12 * 128), (0, 5 * 128)]
    per = [dead_zone_vectors(n, a, b) for a, b in zones]
    vec_np = tuple(np.concatenate([p[i] for p in per]) for i in range(4))
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device="cuda")
    qs = fm.fm_classify_tiles(*vec, causal=True)
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=scale, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    rng = np.random.default_rng(11)
    G = hq // hkv
    for bi, (a, b) in enumerate(zones):
        assert torch.all(o[bi, :, a:b] == 0).item()
        assert torch.all(torch.isneginf(lse[bi, :, a:b])).item()
        rows = np.unique(np.concatenate([rng.choice(n, size=24, replace=False), [a, b - 1, min(b, n - 1)]]))
        trows = torch.as_tensor(rows, device="cuda")
        h = int(rng.integers(hq))
        g = h // G
        O_ref, L_ref = oracle.forward(f64(q[bi:bi + 1, h:h + 1]), f64(k[bi:bi + 1, g:g + 1]), f64(v[bi:bi + 1, g:g + 1]),
                                      tuple(x[bi:bi + 1] for x in vec_np), True, scale, rows=rows)
        assert_out(f64(o[bi:bi + 1, h:h + 1, trows]), O_ref)
        assert_lse(f64(lse[bi:bi + 1, h:h + 1, trows]), L_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_persistent_forward_general_masks(causal):
    """Random two-interval masks: nearly every tile partial, many units per CTA."""
    from helpers import random_vectors
    B, hq, hkv, n, d = 1, 32, 8, 4096, 128
    cfg = dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d, causal=causal)
    scale = 1.0 / np.sqrt(d)
    rng = np.random.default_rng(5)
    vec_np = random_vectors(rng, B, n, "general")
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device="cuda")
    qs = fm.fm_classify_tiles(*vec, causal=causal)
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=scale, causal=causal)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    # every row of two heads: a unit's output is written by four row groups
    # at different times, and the last unit of each CTA takes its own path
    G = hq // hkv
    for h in (0, hq - 1):
        g = h // G
        O_ref, L_ref = oracle.forward(f64(q[:, h:h + 1]), f64(k[:, g:g + 1]), f64(v[:, g:g + 1]), vec_np, causal,
                                      scale)
        og = f64(o[:, h:h + 1])
        for q0 in range(0, n, 128):
            assert_out(og[:, :, q0:q0 + 128], O_ref[:, :, q0:q0 + 128])
        assert_lse(f64(lse[:, h:h + 1]), L_ref)
