"""Pins for the CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something fixed outside it: the mask
matrices printed on the FlashMask Guide page, closed forms, brute force
from a plain-language description of each mask family, torch's own
scaled_dot_product_attention and autograd in float64, central finite
differences, and Theorem 1 of the FlashMask-3 project page (§3.2).
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from workloads import configs, masks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(path):
    out, cur = {}, None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("["):
            cur = line.strip("[]")
            out[cur] = []
            continue
        out[cur].append([int(t) for t in line.split()])
    return {k: np.array(v, dtype=bool) for k, v in out.items()}


def _random_vectors(rng, n, general=True):
    """Random boundary vectors; `general` lets LTE < N, UTS > 0 and empty intervals."""
    if general:
        a = rng.integers(0, n + 1, size=(2, n))
        b = rng.integers(0, n + 1, size=(2, n))
        lts, lte = a.min(0), a.max(0)
        uts, ute = b.min(0), b.max(0)
        # some explicitly empty / reversed intervals
        flip = rng.random(n) < 0.1
        lts[flip], lte[flip] = lte[flip], lts[flip]
    else:
        lts = rng.integers(0, n + 1, size=n)
        lte = np.full(n, n)
        uts = np.zeros(n, dtype=np.int64)
        ute = rng.integers(0, n + 1, size=n)
    return tuple(x.astype(np.int32) for x in (lts, lte, uts, ute))


def _structured_vectors(rng, n, t):
    """One of the mask families with random parameters (gives unmasked tiles too)."""
    kind = t % 4
    if kind == 0:
        return masks.causal_documents(masks.draw_fill(rng, n, 4, 30), n)
    if kind == 1:
        return masks.prefix_lm_documents(masks.draw_fill(rng, n, 6, 40), n)
    if kind == 2:
        return masks.sliding_window(n, int(rng.integers(4, 40)), int(rng.integers(0, 5)))
    return masks.random_eviction(n, 1 / 12, rng)


# ------------------------------------------------------------ mask pins
def test_golden_p3_causal():
    g = _read_golden(os.path.join(GOLDEN, "p3_mask_topologies.txt"))["causal"]
    n = 8
    lts, lte, uts, ute = masks._empty(n)
    vis = ~oracle.dense_mask(lts, lte, uts, ute, True)
    assert np.array_equal(vis[: g.shape[0]], g)


def test_golden_p3_document_packing():
    g = _read_golden(os.path.join(GOLDEN, "p3_mask_topologies.txt"))["document_packing"]
    lts, lte, uts, ute = masks.causal_documents([2, 2, 2, 2], 8)
    vis = ~oracle.dense_mask(lts, lte, uts, ute, True)
    assert np.array_equal(vis[: g.shape[0]], g)


def _brute_docs(lens, n):
    doc = np.repeat(np.arange(len(lens)), lens)[:n]
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    return (doc[i] == doc[j]) & (j <= i)


def test_encoder_causal_documents():
    lens = [5, 1, 9, 3, 14]
    n = sum(lens)
    vis = ~oracle.dense_mask(*masks.causal_documents(lens, n), True)
    assert np.array_equal(vis, _brute_docs(lens, n))


def test_encoder_share_question():
    samples = [(4, 3, 2), (2, 1, 5), (3, 3, 3)]
    n = sum(map(sum, samples)) + 4  # 4 tokens of padding
    vis = ~oracle.dense_mask(*masks.share_question(samples, n), True)
    # brute force from the description: same sample, causal, responses see
    # the prompt and themselves but not the sibling; padding sees nothing.
    seg = np.full(n, -1)
    part = np.full(n, -1)  # 0 prompt, 1 resp a, 2 resp b
    s = 0
    for t, (p, a, b) in enumerate(samples):
        for off, (ln, kind) in enumerate([(p, 0), (a, 1), (b, 2)]):
            seg[s : s + ln] = t
            part[s : s + ln] = kind
            s += ln
    exp = np.zeros((n, n), dtype=bool)
    for i in range(n):
        for j in range(n):
            if seg[i] < 0 or seg[j] < 0 or seg[i] != seg[j] or j > i:
                continue
            if part[j] == 0 or part[j] == part[i]:
                exp[i, j] = True
    assert np.array_equal(vis, exp)
    assert (~vis[-4:]).all()  # padding rows fully masked


def test_encoder_prefix_lm():
    lens = [8, 12, 7]
    n = sum(lens)
    vis = ~oracle.dense_mask(*masks.prefix_lm_documents(lens, n), False)
    exp = np.zeros((n, n), dtype=bool)
    s = 0
    for L in lens:
        p = L // 4
        for i in range(s, s + L):
            for j in range(s, s + L):
                exp[i, j] = (j < s + p) or (j <= i)
        s += L
    assert np.array_equal(vis, exp)


def test_encoder_sliding_window():
    n, w, k = 40, 6, 2
    vis = ~oracle.dense_mask(*masks.sliding_window(n, w, k), True)
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    exp = (j <= i) & ((i < j + w) | (j < k))
    assert np.array_equal(vis, exp)


def test_encoder_random_eviction_diagonal_visible():
    n = 300
    rng = np.random.default_rng(3)
    vec = masks.random_eviction(n, 1 / 16, rng)
    vis = ~oracle.dense_mask(*vec, True)
    assert vis.diagonal().all()
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    assert np.array_equal(vis, (j <= i) & (i < vec[0][j]))


def test_closed_form_causal_document_pairs():
    lens = [163, 54, 39]
    cfg = configs.make("tiny")
    assert cfg["docs"] == lens
    vec_b = tuple(x[0] for x in (cfg["lts"], cfg["lte"], cfg["uts"], cfg["ute"]))
    got = oracle.unmasked_pairs(vec_b, True)
    assert got == sum(L * (L + 1) // 2 for L in lens) == 15631


# ------------------------------------------------------------ tile rule
def _true_class(vis_tile):
    if not vis_tile.any():
        return oracle.SKIP
    if vis_tile.all():
        return oracle.UNMASKED
    return oracle.PARTIAL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("general", [False, True])
def test_tile_rule_exhaustive_64_8x8(causal, general):
    """The worked geometry of FlashMask-3 §3.1: a 64 x 64 mask with 8 x 8 tiles."""
    rng = np.random.default_rng(11 + causal + 2 * general)
    n, bt = 64, 8
    seen = set()
    for trial in range(60):
        vec = _random_vectors(rng, n, general) if trial % 2 else _structured_vectors(rng, n, trial // 2)
        vis = ~oracle.dense_mask(*vec, causal)
        cls = oracle.classify_tiles(*vec, causal, bt, bt)
        for qb in range(n // bt):
            for kb in range(n // bt):
                t = vis[qb * bt : (qb + 1) * bt, kb * bt : (kb + 1) * bt]
                c = cls[qb, kb]
                seen.add(int(c))
                if c == oracle.SKIP:
                    assert not t.any()
                if c == oracle.UNMASKED:
                    assert t.all()
    assert seen == {0, 1, 2}


def test_tile_rule_reduces_to_printed_rule():
    """With LTE = N and UTS = 0 (non-causal) the class is the printed rule exactly."""
    rng = np.random.default_rng(5)
    n, bt = 64, 8
    for trial in range(40):
        lts, lte, uts, ute = _random_vectors(rng, n, general=False)
        cls = oracle.classify_tiles(lts, lte, uts, ute, False, bt, bt)
        for qb in range(n // bt):
            q0, q1 = qb * bt, (qb + 1) * bt
            for kb in range(n // bt):
                blk = slice(kb * bt, (kb + 1) * bt)
                if q0 >= lts[blk].max() or q1 <= ute[blk].min():
                    want = oracle.SKIP
                elif q1 <= lts[blk].min() and q0 >= ute[blk].max():
                    want = oracle.UNMASKED
                else:
                    want = oracle.PARTIAL
                assert cls[qb, kb] == want


def test_tile_rule_causal_document_tight():
    """Document-aligned tiles of a causal document mask classify exactly."""
    lens = [16, 32, 16]
    vec = masks.causal_documents(lens, 64)
    cls = oracle.classify_tiles(*vec, True, 8, 8)
    vis = ~oracle.dense_mask(*vec, True)
    for qb in range(8):
        for kb in range(8):
            t = vis[qb * 8 : (qb + 1) * 8, kb * 8 : (kb + 1) * 8]
            assert cls[qb, kb] == _true_class(t)


def test_tile_rule_ragged_edge():
    rng = np.random.default_rng(9)
    n, bm, bn = 50, 16, 8  # ragged on both axes
    for causal in (False, True):
        for trial in range(30):
            vec = _random_vectors(rng, n, True)
            vis = ~oracle.dense_mask(*vec, causal)
            cls = oracle.classify_tiles(*vec, causal, bm, bn)
            assert cls.shape == (4, 7)
            for qb in range(4):
                for kb in range(7):
                    t = vis[qb * bm : (qb + 1) * bm, kb * bn : (kb + 1) * bn]
                    if cls[qb, kb] == oracle.SKIP:
                        assert not t.any()
                    if cls[qb, kb] == oracle.UNMASKED:
                        assert t.all()


# At 1 x 1 tiles the block min and max are the column's own values, so the
# generalised rule must reproduce the dense mask element for element: skip
# exactly where masked, unmasked exactly where visible. Soundness pins alone
# ("skip => all masked", "unmasked => all visible") cannot see a clause written
# too conservatively; exactness can.
def _rule_exact_at_1x1(classify, seed=21, n=40, trials=30):
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        for trial in range(trials):
            vec = _random_vectors(rng, n, general=True)
            if trial % 3 == 0:  # reversed / empty intervals in both pairs
                lts, lte, uts, ute = (x.copy() for x in vec)
                uts[::4], ute[::4] = ute[::4].copy(), uts[::4].copy()
                vec = (lts, lte, uts, ute)
            cls = classify(*vec, causal, 1, 1)
            vis = ~oracle.dense_mask(*vec, causal)
            want = np.where(vis, oracle.UNMASKED, oracle.SKIP)
            if not np.array_equal(cls, want):
                return False
    return True


def _uniform_block_vectors(rng, n, bt):
    """Vectors whose columns share their four values within each bt-wide block."""
    nb = n // bt
    a = rng.integers(0, n + 1, size=(2, nb))
    c = rng.integers(0, n + 1, size=(2, nb))
    lts, lte = a.min(0), a.max(0)
    uts, ute = c.min(0), c.max(0)
    flip = rng.random(nb) < 0.15
    lts[flip], lte[flip] = lte[flip], lts[flip]
    return tuple(np.repeat(x, bt).astype(np.int32) for x in (lts, lte, uts, ute))


def _rule_exact_on_uniform_blocks(classify, seed=23, n=64, bt=8, trials=60):
    """Uniform blocks: the rule's class equals the tile's true class, except in
    the two places where the rule is conservative by construction: only the
    union of the masked sets covers the tile (no single term does; the rule
    tests each term alone), or an empty interval's endpoints straddle the
    tile's rows (the rule reads an interval by its endpoints). Both then give
    partial."""
    rng = np.random.default_rng(seed)
    for causal in (False, True):
        for _ in range(trials):
            vec = _uniform_block_vectors(rng, n, bt)
            cls = classify(*vec, causal, bt, bt)
            vis = ~oracle.dense_mask(*vec, causal)
            for qb in range(n // bt):
                q0, q1 = qb * bt, (qb + 1) * bt
                for kb in range(n // bt):
                    k0, k1 = kb * bt, (kb + 1) * bt
                    truth = _true_class(vis[q0:q1, k0:k1])
                    if cls[qb, kb] == truth:
                        continue
                    a0, a1, u0, u1 = (int(x[k0]) for x in vec)
                    one_term_covers = ((a0 <= q0 and q1 <= a1) or (u0 <= q0 and q1 <= u1)
                                       or (causal and q1 <= k0))
                    if truth == oracle.SKIP and cls[qb, kb] == oracle.PARTIAL and not one_term_covers:
                        continue
                    # an empty interval (start >= end) is judged by its endpoints
                    # too: one that straddles the tile's rows makes it partial
                    straddles_empty = any(s >= e and not (q1 <= s or q0 >= e) for s, e in ((a0, a1), (u0, u1)))
                    if truth == oracle.UNMASKED and cls[qb, kb] == oracle.PARTIAL and straddles_empty:
                        continue
                    return False
    return True


def test_tile_rule_exact_at_1x1_tiles():
    assert _rule_exact_at_1x1(oracle.classify_tiles)


def test_tile_rule_exact_on_uniform_blocks():
    assert _rule_exact_on_uniform_blocks(oracle.classify_tiles)


# Conservative slips: each keeps every soundness pin green (the tile is only
# called partial more often), so only the exactness pins above can catch them.
_CONSERVATIVE_SLIPS = [
    ("q1 <= mn_lts[kb] or q0 >= mx_lte[kb]", "q1 <= mn_lts[kb]"),
    ("q1 <= mn_uts[kb] or q0 >= mx_ute[kb]", "q0 >= mx_ute[kb]"),
    ("q1 <= mn_uts[kb] or q0 >= mx_ute[kb]", "q1 <= mn_uts[kb]"),
    ("or (q0 >= mx_uts[kb] and q1 <= mn_ute[kb])", ""),
    ("(not causal) or q0 >= k1 - 1", "(not causal) or q0 >= k1"),
]


@pytest.mark.parametrize("old,new", _CONSERVATIVE_SLIPS)
def test_tile_rule_exactness_pins_catch_conservative_slips(old, new):
    """Plant each slip in a copy of the oracle's classifier (CPU, test-local)."""
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(oracle.classify_tiles))
    assert old in src
    ns = dict(vars(oracle.reference))
    exec(src.replace(old, new), ns)
    slipped = ns["classify_tiles"]
    caught = not _rule_exact_at_1x1(slipped) or not _rule_exact_on_uniform_blocks(slipped)
    assert caught, f"slip not caught: {old!r} -> {new!r}"


def test_tiny_tile_counts():
    cfg = configs.make("tiny")
    vec = tuple(x[0] for x in (cfg["lts"], cfg["lte"], cfg["uts"], cfg["ute"]))
    cls = oracle.classify_tiles(*vec, True, 64, 64)
    counts = [int((cls == c).sum()) for c in (0, 1, 2)]
    assert counts == [8, 7, 1]


def test_queues_cover_tiles_in_order():
    rng = np.random.default_rng(2)
    tabs = [rng.integers(0, 3, size=(5, 7)).astype(np.uint8) for _ in range(2)]
    q_off, q_q, k_off, k_q = oracle.build_queues(tabs)
    assert len(q_off) == 11 and len(k_off) == 15
    for b, cls in enumerate(tabs):
        for qb in range(5):
            ent = q_q[q_off[b * 5 + qb] : q_off[b * 5 + qb + 1]]
            kbs = ent >> 1
            assert list(kbs) == sorted(kbs, reverse=True)  # right to left
            assert set(kbs) == set(np.nonzero(cls[qb])[0])
            assert all((e & 1) == (cls[qb, e >> 1] == 1) for e in ent)
        for kb in range(7):
            ent = k_q[k_off[b * 7 + kb] : k_off[b * 7 + kb + 1]]
            qbs = ent >> 1
            assert list(qbs) == sorted(qbs)
            assert set(qbs) == set(np.nonzero(cls[:, kb])[0])


# ------------------------------------------------------------ attention
def _rand_problem(rng, B, hq, hkv, n, d, seed=0):
    g = torch.Generator().manual_seed(seed)
    mk = lambda h: torch.randn(B, h, n, d, generator=g, dtype=torch.float64)
    return mk(hq), mk(hkv), mk(hkv), mk(hq)


def _stack_vec(vecs):
    return tuple(np.stack(x) for x in zip(*vecs))


def _torch_sdpa(q, k, v, vis, scale):
    """Reference by torch: boolean mask (True = attend), GQA by repeat."""
    rep = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(rep, dim=1)
    vv = v.repeat_interleave(rep, dim=1)
    return F.scaled_dot_product_attention(q, kk, vv, attn_mask=torch.as_tensor(vis)[:, None], scale=scale)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_matches_torch_sdpa(causal):
    rng = np.random.default_rng(1)
    B, hq, hkv, n, d = 2, 4, 2, 48, 16
    q, k, v, _ = _rand_problem(rng, B, hq, hkv, n, d)
    vecs = [_random_vectors(rng, n, True) for _ in range(B)]
    vec = _stack_vec(vecs)
    vis = np.stack([~oracle.dense_mask(*vb, causal) for vb in vecs])
    scale = 0.37
    O, L = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, causal, scale)
    ref = _torch_sdpa(q, k, v, vis, scale).numpy()
    ok_rows = vis.any(axis=2)  # (B, n) rows with at least one visible key
    for b in range(B):
        assert np.allclose(O[b][:, ok_rows[b]], ref[b][:, ok_rows[b]], atol=1e-12, rtol=1e-10)
        # fully masked rows: exactly zero output and -inf LSE
        assert (O[b][:, ~ok_rows[b]] == 0).all()
        assert np.isneginf(L[b][:, ~ok_rows[b]]).all()
    # LSE against scipy's logsumexp of the visible scaled scores
    for b in range(B):
        for h in range(hq):
            s = scale * (q[b, h].numpy() @ k[b, h // 2].numpy().T)
            s = np.where(vis[b], s, -np.inf)
            want = logsumexp(s, axis=1)
            assert np.allclose(L[b, h][ok_rows[b]], want[ok_rows[b]], atol=1e-12)


def test_unmasked_rows_sum_to_one():
    rng = np.random.default_rng(4)
    q, k, v, _ = _rand_problem(rng, 1, 2, 1, 40, 8)
    vec = _stack_vec([_random_vectors(rng, 40, True)])
    p, lse = oracle.row_probs(q.numpy(), k.numpy(), vec, True, 0.5, 0, 1, np.arange(40))
    live = ~np.isneginf(lse)
    assert np.abs(p[live].sum(1) - 1).max() < 1e-12
    assert (p[~live] == 0).all()


def test_all_visible_is_plain_sdpa_and_causal_is_causal_sdpa():
    rng = np.random.default_rng(6)
    n = 33
    q, k, v, _ = _rand_problem(rng, 1, 2, 2, n, 8)
    none = masks._empty(n)
    vec = _stack_vec([none])
    O, _ = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, False, 0.3)
    ref = F.scaled_dot_product_attention(q, k, v, scale=0.3).numpy()
    assert np.allclose(O, ref, atol=1e-12)
    O, _ = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, True, 0.3)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.3).numpy()
    assert np.allclose(O, ref, atol=1e-12)


def test_causal_document_equals_per_document_attention():
    rng = np.random.default_rng(8)
    lens = [7, 19, 4, 12]
    n = sum(lens)
    q, k, v, _ = _rand_problem(rng, 1, 2, 1, n, 8)
    vec = _stack_vec([masks.causal_documents(lens, n)])
    O, L = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, True, 0.25)
    s = 0
    for ln in lens:
        sl = slice(s, s + ln)
        ref = F.scaled_dot_product_attention(
            q[:, :, sl], k[:, :, sl].repeat_interleave(2, 1), v[:, :, sl].repeat_interleave(2, 1),
            is_causal=True, scale=0.25).numpy()
        assert np.allclose(O[:, :, sl], ref, atol=1e-12)
        s += ln


# ------------------------------------------------------------ backward
def test_backward_finite_differences():
    rng = np.random.default_rng(12)
    B, hq, hkv, n, d = 1, 4, 2, 20, 6
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, B, hq, hkv, n, d, seed=3))
    vec = _stack_vec([_random_vectors(rng, n, True)])
    scale, causal = 0.45, True
    dQ, dK, dV = oracle.backward(q, k, v, do, vec, causal, scale)

    def loss(qq, kk, vv):
        O, _ = oracle.forward(qq, kk, vv, vec, causal, scale)
        return float((O * do).sum())

    eps = 1e-6
    picks = [(0, 1, 3, 2), (0, 3, 17, 5), (0, 0, 9, 0), (0, 2, 19, 4)]
    for (b, h, i, c) in picks:
        for name, arr, grad, hh in (("q", q, dQ, h), ("k", k, dK, h // 2), ("v", v, dV, h // 2)):
            plus, minus = arr.copy(), arr.copy()
            plus[b, hh, i, c] += eps
            minus[b, hh, i, c] -= eps
            args = lambda a: (a, k, v) if name == "q" else ((q, a, v) if name == "k" else (q, k, a))
            fd = (loss(*args(plus)) - loss(*args(minus))) / (2 * eps)
            an = grad[b, hh, i, c]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, b, hh, i, c, fd, an)


def test_backward_matches_torch_autograd():
    rng = np.random.default_rng(13)
    B, hq, hkv, n, d = 2, 4, 2, 40, 8
    q, k, v, do = _rand_problem(rng, B, hq, hkv, n, d, seed=5)
    # masks without fully-masked rows (torch returns NaN there)
    vecs = []
    while len(vecs) < B:
        vb = _random_vectors(rng, n, True)
        if (~oracle.dense_mask(*vb, True)).any(axis=1).all():
            vecs.append(vb)
    vis = np.stack([~oracle.dense_mask(*vb, True) for vb in vecs])
    vec = _stack_vec(vecs)
    scale = 0.3
    dQ, dK, dV = oracle.backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), vec, True, scale)
    qq, kk, vv = (x.clone().requires_grad_() for x in (q, k, v))
    out = _torch_sdpa(qq, kk, vv, vis, scale)
    (out * do).sum().backward()
    assert np.allclose(dQ, qq.grad.numpy(), atol=1e-10)
    assert np.allclose(dK, kk.grad.numpy(), atol=1e-10)
    assert np.allclose(dV, vv.grad.numpy(), atol=1e-10)


def test_backward_fully_masked_rows_contribute_nothing():
    rng = np.random.default_rng(14)
    samples = [(3, 2, 2), (2, 2, 1)]
    n = 16  # 4 padding rows at the end are fully masked
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, 1, 2, 1, n, 4, seed=6))
    vec = _stack_vec([masks.share_question(samples, n)])
    dQ, dK, dV = oracle.backward(q, k, v, do, vec, True, 0.5)
    assert (dQ[:, :, 12:] == 0).all()
    # zeroing dO on the padding rows changes nothing
    do2 = do.copy()
    do2[:, :, 12:] = 0
    _, dK2, dV2 = oracle.backward(q, k, v, do2, vec, True, 0.5)
    assert np.array_equal(dK, dK2) and np.array_equal(dV, dV2)


def test_backward_gqa_equals_replicated_heads():
    rng = np.random.default_rng(15)
    n, d = 24, 4
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, 1, 6, 2, n, d, seed=7))
    vec = _stack_vec([_random_vectors(rng, n, True)])
    dQ, dK, dV = oracle.backward(q, k, v, do, vec, False, 0.7)
    kr, vr = np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1)
    dQr, dKr, dVr = oracle.backward(q, kr, vr, do, vec, False, 0.7)
    assert np.allclose(dQ, dQr, atol=1e-13)
    assert np.allclose(dK, dKr.reshape(1, 2, 3, n, d).sum(2), atol=1e-12)
    assert np.allclose(dV, dVr.reshape(1, 2, 3, n, d).sum(2), atol=1e-12)


def test_backward_subsets_are_slices():
    rng = np.random.default_rng(16)
    n, d = 30, 4
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, 1, 4, 2, n, d, seed=8))
    vec = _stack_vec([_random_vectors(rng, n, True)])
    dQ, dK, dV = oracle.backward(q, k, v, do, vec, True, 0.6)
    rows, cols = np.array([2, 7, 29]), np.array([0, 11, 12, 28])
    dQs, dKs, dVs = oracle.backward(q, k, v, do, vec, True, 0.6, rows=rows, cols=cols)
    assert np.allclose(dQs, dQ[:, :, rows], atol=1e-13)
    assert np.allclose(dKs, dK[:, :, cols], atol=1e-13)
    assert np.allclose(dVs, dV[:, :, cols], atol=1e-13)


# ---------------------------------------------------------- localization
def test_localize_theorem_1_bruteforce():
    """FlashMask-3 §3.2, Theorem 1: for any chunk assignment the rank-local
    intervals equal the global intervals at the corresponding rows."""
    rng = np.random.default_rng(21)
    for trial in range(40):
        P, kappa = int(rng.integers(2, 5)), int(rng.integers(1, 4))
        C = int(rng.integers(1, 6))
        n = P * kappa * C
        lts, lte, uts, ute = _random_vectors(rng, n, True)
        owner = rng.permutation(np.repeat(np.arange(P), kappa))
        for r in range(P):
            chunks = np.sort(np.nonzero(owner == r)[0])
            offs = chunks * C
            loc = [oracle.localize(x, offs, C) for x in (lts, lte, uts, ute)]
            assert all(np.array_equal(a, oracle.localize_count(x, offs, C))
                       for a, x in zip(loc, (lts, lte, uts, ute)))
            grow = np.concatenate([np.arange(o, o + C) for o in offs])  # local row -> global row
            gl = ~oracle.dense_mask(lts, lte, uts, ute, False)[grow]
            n_loc = len(grow)
            l = np.arange(n_loc)[:, None]
            loc_vis = ~(((loc[0][None, :] <= l) & (l < loc[1][None, :])) |
                        ((loc[2][None, :] <= l) & (l < loc[3][None, :])))
            assert np.array_equal(loc_vis, gl)


def test_localize_hand_example():
    # chunks of 4 rows at global offsets 0 and 8: global 10 -> 4 + 2 = 6 rows before it
    assert oracle.localize(np.array([10, 0, 3, 4, 8, 12, 20]), [0, 8], 4).tolist() == [6, 0, 3, 4, 4, 8, 8]


# ------------------------------------------- visible-columns mode
# The full-size parity tests run the oracle over only the key columns each row
# chunk sees (masked columns add exact zeros). It is pinned here against the
# strict mode and, independently, against torch's own SDPA and autograd.
def _strict_vs_visible(q, k, v, do, vec, causal, scale, rows=None, cols=None, tol=1e-12):
    O, L = oracle.forward(q, k, v, vec, causal, scale, rows=rows)
    Ov, Lv = oracle.forward(q, k, v, vec, causal, scale, rows=rows, visible_only=True, row_chunk=37)
    assert np.array_equal(np.isneginf(L), np.isneginf(Lv))
    fin = ~np.isneginf(L)
    assert np.abs(L[fin] - Lv[fin]).max() <= tol
    assert np.abs(O - Ov).max() <= tol
    g = oracle.backward(q, k, v, do, vec, causal, scale, rows=rows, cols=cols)
    gv = oracle.backward(q, k, v, do, vec, causal, scale, rows=rows, cols=cols, visible_only=True, row_chunk=29)
    for a, b in zip(g, gv):
        assert a.shape == b.shape and np.abs(a - b).max() <= tol * max(1.0, np.abs(a).max())


@pytest.mark.parametrize("causal", [False, True])
def test_visible_only_equals_strict_on_general_masks(causal):
    rng = np.random.default_rng(31)
    B, hq, hkv, n, d = 2, 4, 2, 96, 16
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, B, hq, hkv, n, d, seed=7))
    vec = _stack_vec([_random_vectors(rng, n, True) for _ in range(B)])
    _strict_vs_visible(q, k, v, do, vec, causal, 0.31)
    rows = np.sort(rng.choice(n, 20, replace=False))
    cols = np.sort(rng.choice(n, 12, replace=False))
    _strict_vs_visible(q, k, v, do, vec, causal, 0.31, rows=rows, cols=cols)


def test_visible_only_equals_strict_on_the_workload_families():
    rng = np.random.default_rng(32)
    n, d = 512, 32
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, 1, 2, 1, n, d, seed=8))
    for t in range(4):
        vec = _stack_vec([_structured_vectors(rng, n, t)])
        _strict_vs_visible(q, k, v, do, vec, t != 1, 0.2)


def test_visible_only_equals_strict_on_the_tiny_workload():
    cfg = configs.make("tiny")
    rng = np.random.default_rng(33)
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, 1, 2, 2, cfg["N"], cfg["d"], seed=9))
    vec = (cfg["lts"], cfg["lte"], cfg["uts"], cfg["ute"])
    _strict_vs_visible(q, k, v, do, vec, True, cfg["scale"])


def test_visible_only_per_head_and_multi_interval_forms():
    rng = np.random.default_rng(34)
    B, hq, hkv, n, d = 1, 4, 2, 80, 8
    q, k, v, do = (x.numpy() for x in _rand_problem(rng, B, hq, hkv, n, d, seed=10))
    heads = tuple(np.stack([np.stack([_random_vectors(rng, n, True)[i] for _ in range(hq)])])
                  for i in range(4))
    _strict_vs_visible(q, k, v, do, {"heads": heads}, True, 0.4)
    cuts = np.sort(rng.integers(0, n, size=(B, 4, n)), axis=1)
    multi = {"fms": cuts[:, 0::2].astype(np.int32), "fme": cuts[:, 1::2].astype(np.int32)}
    _strict_vs_visible(q, k, v, do, multi, False, 0.4)


def test_visible_only_against_torch_autograd():
    # independent of the strict mode: torch SDPA + autograd in float64
    rng = np.random.default_rng(35)
    B, hq, hkv, n, d = 1, 2, 1, 64, 8
    q, k, v, do = _rand_problem(rng, B, hq, hkv, n, d, seed=11)
    vec = _stack_vec([_structured_vectors(rng, n, 0)])
    vis = ~oracle.dense_mask(*(x[0] for x in vec), True)
    qq, kk, vv = (x.clone().requires_grad_(True) for x in (q, k, v))
    out = _torch_sdpa(qq, kk, vv, vis[None], 0.3)
    out.backward(do)
    O, _ = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, True, 0.3, visible_only=True)
    dQ, dK, dV = oracle.backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), vec, True, 0.3, visible_only=True)
    assert np.allclose(O, out.detach().numpy(), atol=1e-12)
    assert np.allclose(dQ, qq.grad.numpy(), atol=1e-11)
    assert np.allclose(dK, kk.grad.numpy(), atol=1e-11)
    assert np.allclose(dV, vv.grad.numpy(), atol=1e-11)
