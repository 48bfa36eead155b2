"""Parity at the full workload sizes, in the launch configuration the benchmark times.

The oracle cannot afford a whole 64-head x 131072^2 problem, so:
  * tile classes and queues: the whole problem, bit-exact (test_gpu_classify);
  * O, LSE and dQ: every output of sampled query rows of two seeded heads, from
    the full-size GPU run;
  * dK and dV: a group slice. The GPU reruns the same kernels on the same N,
    mask and data with the query heads cut to (at most) four heads of one kv
    group; the oracle computes dK / dV of sampled key columns of that slice,
    choosing columns whose feeding rows it can afford.
Inputs are drawn on the GPU with seeded CUDA generators (an input generator,
not the library) and copied to the host for the oracle.
"""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs, tensors

from helpers import assert_grad, assert_lse, assert_out, f64

pytestmark = pytest.mark.gpu

FULL = ["doc8k", "share_question32k", "prefix_lm64k", "sliding_window64k", "eviction128k"]


def _run_gpu(cfg, q, k, v, do, vec):
    qs = fm.fm_classify_tiles(*vec, causal=cfg["causal"])
    o, lse = fm.fm_attn_fwd(q, k, v, *vec, qs, scale=cfg["scale"], causal=cfg["causal"])
    dq, dk, dv = fm.fm_attn_bwd(q, k, v, o, lse, do, *vec, qs, scale=cfg["scale"], causal=cfg["causal"])
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    return o, lse, dq, dk, dv


def _visible_rows_per_column(vec_b, causal, n):
    """Rows that see each key column: N minus the union of its masked intervals."""
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


def _cheap_columns(vec_b, causal, n, rng, budget_rows=3000, count=48):
    """Key columns seen by few rows (the oracle needs each of those rows in full)."""
    seen = _visible_rows_per_column(vec_b, causal, n)
    cand = np.nonzero((seen > 0) & (seen <= 256))[0]
    pick = np.sort(rng.choice(cand, size=min(count, len(cand)), replace=False))
    tot, out = 0, []
    for c in pick:
        if tot + seen[c] > budget_rows:
            break
        tot += seen[c]
        out.append(c)
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("name", FULL)
def test_full_size_rows_and_group_slice(name):
    cfg = configs.make(name)
    B, Hq, Hkv, N, d = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], cfg["d"]
    G = Hq // Hkv
    rng = np.random.default_rng(123)
    dev = "cuda"
    vec_np = tuple(cfg[n] for n in ("lts", "lte", "uts", "ute"))
    vec = [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in vec_np]
    q, k, v, do = tensors.make_qkvdo(cfg, device=dev)

    # ---- full problem: O, LSE, dQ on sampled rows of two heads
    o, lse, dq, dk, dv = _run_gpu(cfg, q, k, v, do, vec)
    heads = sorted(rng.choice(Hq, size=2, replace=False).tolist())
    rows = np.sort(rng.choice(N, size=96, replace=False))
    rows = np.unique(np.concatenate([rows, [0, N - 1]]))
    trows = torch.as_tensor(rows, device=dev)
    for h in heads:
        g = h // G
        qh, doh = f64(q[:, h:h + 1]), f64(do[:, h:h + 1])
        kh, vh = f64(k[:, g:g + 1]), f64(v[:, g:g + 1])
        O_ref, L_ref = oracle.forward(qh, kh, vh, vec_np, cfg["causal"], cfg["scale"], rows=rows)
        dQ_ref, _, _ = oracle.backward(qh, kh, vh, doh, vec_np, cfg["causal"], cfg["scale"], rows=rows,
                                       cols=np.array([], dtype=np.int64))
        assert_out(f64(o[:, h:h + 1, trows]), O_ref)
        assert_lse(f64(lse[:, h:h + 1, trows]), L_ref)
        assert_grad(f64(dq[:, h:h + 1, trows]), dQ_ref, f"dQ[{name} h{h}]")
    del o, lse, dq, dk, dv
    torch.cuda.empty_cache()

    # ---- group slice: up to four query heads of one kv group, same N / mask / data
    g0 = int(rng.integers(Hkv))
    nh = min(4, G)
    hsel = g0 * G + np.sort(rng.choice(G, size=nh, replace=False))
    thsel = torch.as_tensor(hsel, device=dev)
    qs_ = q[:, thsel].contiguous()
    dos_ = do[:, thsel].contiguous()
    ks_, vs_ = k[:, g0:g0 + 1].contiguous(), v[:, g0:g0 + 1].contiguous()
    sub = dict(cfg, H_q=nh, H_kv=1)
    _, _, _, dk_s, dv_s = _run_gpu(sub, qs_, ks_, vs_, dos_, vec)
    cols = _cheap_columns(tuple(x[0] for x in vec_np), cfg["causal"], N, rng)
    assert len(cols) >= 8
    _, dK_ref, dV_ref = oracle.backward(f64(qs_), f64(ks_), f64(vs_), f64(dos_), vec_np, cfg["causal"],
                                        cfg["scale"], rows=np.array([], dtype=np.int64), cols=cols)
    tcols = torch.as_tensor(cols, device=dev)
    assert_grad(f64(dk_s[:, :, tcols]), dK_ref, f"dK[{name}]")
    assert_grad(f64(dv_s[:, :, tcols]), dV_ref, f"dV[{name}]")
