"""Seeded random problems over the joint space the other GPU tests cover one
axis at a time: head dim 64 / 128 / 256, GQA groups of 1 to 4, one or two
batch entries, square and rectangular (N query rows against N_kv keys) shapes
with ragged tails, causal on and off, shared or per-head mask vectors. The
masks are piecewise constant over runs of key columns (each run fully
visible, fully masked, a lower interval, an upper interval or both), so the
tiles fall in all three classes (skipped, unmasked, partial) rather than all
partial as with independent random columns. Every output is compared with the
fp64 oracle (the column-wise representation of the FlashMask Guide, "The
Solution: FlashMask Sparse Mask Representation"; tile skipping of the
FlashMask-3 project page §3.1)."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import tensors

from helpers import assert_grad, assert_lse, assert_out, f64

SEEDS = list(range(24))


def run_vectors(rng, n_rows, n_keys):
    """One set of (N_kv,) vectors, piecewise constant over runs of columns."""
    lts = np.zeros(n_keys, np.int64)
    lte = np.zeros(n_keys, np.int64)
    uts = np.zeros(n_keys, np.int64)
    ute = np.zeros(n_keys, np.int64)
    j = 0
    while j < n_keys:
        r = int(min(n_keys - j, rng.integers(1, 300)))
        kind = int(rng.integers(0, 5))
        a = np.sort(rng.integers(0, n_rows + 1, size=2))
        c = np.sort(rng.integers(0, n_rows + 1, size=2))
        s = slice(j, j + r)
        if kind == 1:      # every row masked
            lte[s] = n_rows
        elif kind == 2:    # lower interval [a0, N)
            lts[s], lte[s] = a[0], n_rows
        elif kind == 3:    # upper interval
            uts[s], ute[s] = c
        elif kind == 4:    # both intervals
            lts[s], lte[s] = a
            uts[s], ute[s] = c
        j += r             # kind 0: fully visible (empty intervals)
    return lts, lte, uts, ute


def draw(seed):
    rng = np.random.default_rng(7000 + seed)
    d = int(rng.choice([64, 128, 256]))
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.integers(1, 5))
    B = int(rng.integers(1, 3))
    n = int(rng.integers(1, 700))
    nk = n if rng.random() < 0.5 else int(rng.integers(1, 700))
    causal = bool(rng.random() < 0.5)
    per_head = bool(rng.random() < 0.35)
    rows = B * hq if per_head else B
    sets = [run_vectors(rng, n, nk) for _ in range(rows)]
    vec = tuple(np.stack([s[i] for s in sets]).astype(np.int32) for i in range(4))
    if per_head:
        vec = tuple(x.reshape(B, hq, nk) for x in vec)
    return dict(d=d, hkv=hkv, hq=hq, B=B, n=n, nk=nk, causal=causal, per_head=per_head, vec=vec)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", SEEDS)
def test_fuzz_against_oracle(seed):
    c = draw(seed)
    B, hq, hkv, n, nk, d = c["B"], c["hq"], c["hkv"], c["n"], c["nk"], c["d"]
    q = tensors.randn_bf16((B, hq, n, d), 100 + seed)
    k = tensors.randn_bf16((B, hkv, nk, d), 200 + seed)
    v = tensors.randn_bf16((B, hkv, nk, d), 300 + seed)
    do = tensors.randn_bf16((B, hq, n, d), 400 + seed)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    vd_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in c["vec"]]
    scale = d ** -0.5
    if c["per_head"]:
        o, lse, dq, dk, dv = fm.fm_attn_per_head(qd, kd, vd, *vd_, causal=c["causal"], scale=scale, do=dod)
        spec = {"heads": c["vec"]}
    else:
        qs = fm.fm_classify_tiles(*vd_, causal=c["causal"], n_rows=n)
        o, lse = fm.fm_attn_fwd(qd, kd, vd, *vd_, qs, scale=scale, causal=c["causal"])
        dq, dk, dv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *vd_, qs, scale=scale, causal=c["causal"])
        spec = c["vec"]
        # the classes the kernels ran on are the oracle's, bit for bit
        cls_ref = np.stack([oracle.classify_tiles(*(x[b] for x in c["vec"]), c["causal"], 128, 128, n_rows=n)
                            for b in range(B)])
        assert np.array_equal(qs.tile_class.cpu().numpy(), cls_ref)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, c["causal"], scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, c["causal"], scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


def test_fuzz_draws_cover_the_space():
    # the seeds above reach every head dim, both GQA and MHA, rectangular and
    # square shapes, both causal settings, shared and per-head vectors, and
    # masks with all three tile classes
    draws = [draw(s) for s in SEEDS]
    assert {c["d"] for c in draws} == {64, 128, 256}
    assert any(c["hq"] > c["hkv"] for c in draws) and any(c["hq"] == c["hkv"] for c in draws)
    assert any(c["n"] != c["nk"] for c in draws) and any(c["n"] == c["nk"] for c in draws)
    assert {c["causal"] for c in draws} == {False, True}
    assert {c["per_head"] for c in draws} == {False, True}
    classes = set()
    for c in draws:
        vec = c["vec"] if not c["per_head"] else tuple(x.reshape(-1, c["nk"]) for x in c["vec"])
        for b in range(vec[0].shape[0]):
            cls = oracle.classify_tiles(*(x[b] for x in vec), c["causal"], 128, 128, n_rows=c["n"])
            classes |= set(np.unique(cls).tolist())
    assert classes == {0, 1, 2}


MULTI_SEEDS = list(range(8))


def draw_multi(seed):
    """A random multi-interval problem: M = 2..4 disjoint inclusive visible
    intervals per key column, piecewise constant over runs of columns (runs
    with every interval empty, runs covering every row, random cuts)."""
    rng = np.random.default_rng(9000 + seed)
    d = int(rng.choice([64, 128, 256]))
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.integers(1, 5))
    B = int(rng.integers(1, 3))
    n = int(rng.integers(1, 700))
    nk = n if rng.random() < 0.5 else int(rng.integers(1, 700))
    M = int(rng.integers(2, 5))
    fms = np.zeros((M, B, nk), np.int64)
    fme = np.full((M, B, nk), -1, np.int64)   # empty: end < start
    for b in range(B):
        j = 0
        while j < nk:
            r = int(min(nk - j, rng.integers(1, 300)))
            kind = int(rng.integers(0, 3))
            if kind == 1:      # one interval covers every row
                fms[0, b, j:j + r], fme[0, b, j:j + r] = 0, n - 1
            elif kind == 2:    # M random disjoint intervals
                cuts = np.sort(rng.integers(0, n + 1, size=2 * M))
                fms[:, b, j:j + r] = cuts[0::2, None]
                fme[:, b, j:j + r] = cuts[1::2, None] - 1
            j += r             # kind 0: nothing visible
    return dict(d=d, hkv=hkv, hq=hq, B=B, n=n, nk=nk, M=M, fms=fms.astype(np.int32), fme=fme.astype(np.int32))


@pytest.mark.gpu
@pytest.mark.parametrize("seed", MULTI_SEEDS)
def test_fuzz_multi_interval_against_oracle(seed):
    c = draw_multi(seed)
    B, hq, hkv, n, nk, d = c["B"], c["hq"], c["hkv"], c["n"], c["nk"], c["d"]
    q = tensors.randn_bf16((B, hq, n, d), 500 + seed)
    k = tensors.randn_bf16((B, hkv, nk, d), 600 + seed)
    v = tensors.randn_bf16((B, hkv, nk, d), 700 + seed)
    do = tensors.randn_bf16((B, hq, n, d), 800 + seed)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    scale = d ** -0.5
    o, lse, dq, dk, dv = fm.fm_attn_multi_interval(qd, kd, vd, torch.from_numpy(c["fms"]).cuda(),
                                                   torch.from_numpy(c["fme"]).cuda(), scale=scale, do=dod)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    spec = {"fms": c["fms"].transpose(1, 0, 2), "fme": c["fme"].transpose(1, 0, 2)}
    O_ref, L_ref = oracle.forward(f64(q), f64(k), f64(v), spec, False, scale)
    assert_out(f64(o), O_ref)
    assert_lse(f64(lse), L_ref)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, False, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad(f64(a), r, name)


def test_fuzz_multi_draws_cover_the_space():
    draws = [draw_multi(s) for s in MULTI_SEEDS]
    assert {c["M"] for c in draws} == {2, 3, 4}
    assert {c["d"] for c in draws} == {64, 128, 256}
    assert any(c["n"] != c["nk"] for c in draws)
