"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot afford a whole 64-head x 131072^2 problem, so:
  * tile classes and queues: the whole problem, bit-exact (test_gpu_classify);
  * O, LSE and dQ: EVERY row of two seeded query heads, from the full-size GPU
    run (the random-eviction workload, whose rows see ~16K keys each at
    N = 131072: 2,048+ sampled rows including its whole last Q block);
  * dK and dV: a group slice. The GPU reruns the same kernels on the same N,
    mask and data with the query heads cut to (at most) four heads of one kv
    group; the oracle computes dK / dV of every key column of the two KV
    blocks with the longest backward queues (the columns whose sums run over
    the most Q blocks), plus a few sampled lightly-seen columns. For the
    random-eviction family, whose longest queues feed ~100K rows, the same
    family runs at N = 16384 with the workload's head layout (64 query heads,
    one kv head).
The oracle runs over the key columns each row chunk sees (`visible_only`:
masked columns add exact zeros; pinned against its strict mode and torch in
tests/test_oracle.py), in threads over row segments and heads.
Inputs are drawn on the GPU with seeded CUDA generators (an input generator,
not the library) and copied to the host for the oracle.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, tensors

from helpers import assert_grad, assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu

FULL = ["doc8k", "share_question32k", "prefix_lm64k", "sliding_window64k", "eviction128k"]
_POOL = 16


def _run_gpu(cfg, q, k, v, do, vec):
    qs = fm.fm_classify_tiles(*vec, causal=cfg["causal"])
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=cfg["scale"], causal=cfg["causal"])
    dq, dk, dv = fm.fm_attn_bwd(q, k, v, o, lse, do, *vec, qs, scale=cfg["scale"], causal=cfg["causal"])
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    return qs, o, lse, dq, dk, dv


def _oracle_rows(qh, kh, vh, doh, vec_np, cfg, rows):
    """O, LSE, dQ of one head on `rows`, in threads over row segments."""
    segs = [s for s in np.array_split(rows, _POOL) if len(s)]

    def one(r):
        O, L = oracle.forward(qh, kh, vh, vec_np, cfg["causal"], cfg["scale"], rows=r, visible_only=True)
        dQ, _, _ = oracle.backward(qh, kh, vh, doh, vec_np, cfg["causal"], cfg["scale"], rows=r,
                                   cols=np.array([], dtype=np.int64), visible_only=True)
        return O, L, dQ

    with ThreadPoolExecutor(len(segs)) as ex:
        parts = list(ex.map(one, segs))
    return tuple(np.concatenate([p[i] for p in parts], axis=2) for i in range(3))


def _oracle_key_grads(q, k, v, do, vec_np, cfg, cols):
    """dK, dV of `cols` summed over all query heads of q, one thread per head."""
    def one(h):
        _, dK, dV = oracle.backward(q, k, v, do, vec_np, cfg["causal"], cfg["scale"], heads=[h],
                                    rows=np.array([], dtype=np.int64), cols=cols, visible_only=True)
        return dK, dV

    with ThreadPoolExecutor(q.shape[1]) as ex:
        parts = list(ex.map(one, range(q.shape[1])))
    return sum(p[0] for p in parts), sum(p[1] for p in parts)


def _longest_queue_columns(queues, n, count=2):
    """Every key column of the `count` KV blocks whose backward queues are longest."""
    k_off = queues.k_off.cpu().numpy().astype(np.int64)
    lens = np.diff(k_off)
    top = np.sort(np.argsort(-lens, kind="stable")[:count])
    cols = np.concatenate([np.arange(kb * 128, min((kb + 1) * 128, n)) for kb in top])
    return cols, lens[top]


def _visible_rows_per_column(vec_b, causal, n):
    """Rows that see each key column: N minus the union of its masked intervals
    (inclusion-exclusion over the two intervals and the causal range)."""
    lts, lte, uts, ute = (x.astype(np.int64) for x in vec_b)
    j = np.arange(n, dtype=np.int64)
    a = [lts, uts, np.zeros(n, np.int64)]
    b = [lte, ute, j if causal else np.zeros(n, np.int64)]
    ln = lambda lo, hi: np.maximum(0, hi - lo)
    u = ln(a[0], b[0]) + ln(a[1], b[1]) + ln(a[2], b[2])
    u -= ln(np.maximum(a[0], a[1]), np.minimum(b[0], b[1]))
    u -= ln(np.maximum(a[0], a[2]), np.minimum(b[0], b[2]))
    u -= ln(np.maximum(a[1], a[2]), np.minimum(b[1], b[2]))
    u += ln(np.maximum(np.maximum(a[0], a[1]), a[2]), np.minimum(np.minimum(b[0], b[1]), b[2]))
    return n - u


def _light_columns(vec_b, causal, n, rng, count=16):
    """A few key columns seen by 1..256 rows (short sums, the other extreme)."""
    seen = _visible_rows_per_column(vec_b, causal, n)
    cand = np.nonzero((seen > 0) & (seen <= 256))[0]
    return np.sort(rng.choice(cand, size=min(count, len(cand)), replace=False)) if len(cand) else cand


def _group_slice_check(cfg, q, k, v, do, vec, vec_np, rng, name):
    """dK, dV of a <= 4-head group slice on the heavily-seen and lightly-seen columns."""
    B, Hq, Hkv, N = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"]
    G = Hq // Hkv
    dev = q.device
    g0 = int(rng.integers(Hkv))
    nh = min(4, G)
    hsel = g0 * G + np.sort(rng.choice(G, size=nh, replace=False))
    thsel = torch.as_tensor(hsel, device=dev)
    qs_ = q[:, thsel].contiguous()
    dos_ = do[:, thsel].contiguous()
    ks_, vs_ = k[:, g0:g0 + 1].contiguous(), v[:, g0:g0 + 1].contiguous()
    sub = dict(cfg, H_q=nh, H_kv=1)
    queues, _, _, _, dk_s, dv_s = _run_gpu(sub, qs_, ks_, vs_, dos_, vec)
    heavy, qlen = _longest_queue_columns(queues, N)
    light = _light_columns(tuple(x[0] for x in vec_np), cfg["causal"], N, rng)
    cols = np.union1d(heavy, light)
    dK_ref, dV_ref = _oracle_key_grads(f64(qs_), f64(ks_), f64(vs_), f64(dos_), vec_np, cfg, cols)
    tcols = torch.as_tensor(cols, device=dev)
    assert_grad(f64(dk_s[:, :, tcols]), dK_ref, f"dK[{name}, KV blocks with queues of {qlen.tolist()} units]")
    assert_grad(f64(dv_s[:, :, tcols]), dV_ref, f"dV[{name}, KV blocks with queues of {qlen.tolist()} units]")
    # the heavy columns alone, so the light ones cannot dilute a heavy mismatch
    hm = np.isin(cols, heavy)
    assert_grad(f64(dk_s[:, :, tcols])[:, :, hm], dK_ref[:, :, hm], f"dK[{name}, heavy columns]")
    assert_grad(f64(dv_s[:, :, tcols])[:, :, hm], dV_ref[:, :, hm], f"dV[{name}, heavy columns]")


@pytest.mark.parametrize("name", FULL)
def test_full_size_rows_and_group_slice(name):
    cfg = configs.make(name)
    Hq, Hkv, N = cfg["H_q"], cfg["H_kv"], cfg["N"]
    G = Hq // Hkv
    rng = np.random.default_rng(123)
    dev = "cuda"
    vec_np = tuple(cfg[n] for n in ("lts", "lte", "uts", "ute"))
    vec = [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device=dev)

    # ---- full problem: O, LSE, dQ on all rows (eviction: sampled rows) of two heads
    _, o, lse, dq, dk, dv = _run_gpu(cfg, q, k, v, do, vec)
    heads = sorted(rng.choice(Hq, size=2, replace=False).tolist())
    if name == "eviction128k":
        rows = np.union1d(np.sort(rng.choice(N, size=2048, replace=False)), np.arange(N - 128, N))
        rows = np.union1d(rows, [0])
    else:
        rows = np.arange(N)
    trows = torch.as_tensor(rows, device=dev)
    for h in heads:
        g = h // G
        qh, doh = f64(q[:, h:h + 1]), f64(do[:, h:h + 1])
        kh, vh = f64(k[:, g:g + 1]), f64(v[:, g:g + 1])
        O_ref, L_ref, dQ_ref = _oracle_rows(qh, kh, vh, doh, vec_np, cfg, rows)
        assert_out(f64(o[:, h:h + 1, trows]), O_ref)
        assert_lse(f64(lse[:, h:h + 1, trows]), L_ref)
        assert_grad(f64(dq[:, h:h + 1, trows]), dQ_ref, f"dQ[{name} h{h}]")
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()

    # ---- group slice: dK / dV on the longest-queue KV blocks
    if name == "eviction128k":
        # same family and head layout at N = 16384 (the longest queues at full N
        # feed ~100K rows, beyond the oracle's budget here)
        cfg = configs.make(name, N=16384)
        vec_np = tuple(cfg[n] for n in ("lts", "lte", "uts", "ute"))
        vec = [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in vec_np]
        q, k, v, do = tensors.make_qkvdo(cfg, device=dev)
    _group_slice_check(cfg, q, k, v, do, vec, vec_np, rng, name)
