"""Run by tests/test_gpu_debug_build.py in a fresh process with FM_LIBRARY=debug:
every attention kernel of the range-checked debug library on small cases,
checked against the oracle; exits non-zero on a parity failure or any device
error bit (a failed range check is FM_DEVERR_DEBUG)."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import mask_aware_sparse_gb300 as fm  # noqa: E402
import oracle  # noqa: E402
from helpers import assert_grad, assert_lse, assert_out, f64, random_vectors  # noqa: E402
from workloads import configs, tensors  # noqa: E402


def status_ok(what):
    st, bits = fm.fm_device_status()
    if st != fm.FM_OK:
        raise SystemExit(f"{what}: device status {st} bits {bits}")


def fwd_bwd(vec, B, hq, hkv, n, d, causal):
    scale = d ** -0.5
    q, k, v, do = tensors.make_qkvdo(dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d))
    dv_ = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv_, causal=causal)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fm.fm_attn_fwd(qd, kd, vd, *dv_, qs, scale=scale, causal=causal)
    dq, dk, dvv = fm.fm_attn_bwd(qd, kd, vd, o, lse, dod, *dv_, qs, scale=scale, causal=causal)
    status_ok(f"fwd/bwd d={d} n={n}")
    O, L = oracle.forward(f64(q), f64(k), f64(v), vec, causal, scale)
    assert_out(f64(o), O)
    assert_lse(f64(lse), L)
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), vec, causal, scale)
    for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dvv), ref):
        assert_grad(f64(a), r, name)


def main():
    assert fm.LIB_PATH.endswith("libfm_debug.so"), fm.LIB_PATH
    cfg = configs.make("tiny")
    fwd_bwd(tuple(cfg[x] for x in ("lts", "lte", "uts", "ute")), 1, 2, 2, 256, 64, True)
    rng = np.random.default_rng(99)
    for d in (64, 128, 256):
        for causal in (False, True):
            fwd_bwd(random_vectors(rng, 2, 389, "general"), 2, 4, 2, 389, d, causal)
    # the FP8 forward
    q, k, v, _ = tensors.make_qkvdo(dict(B=1, H_q=4, H_kv=2, N=384, d=128))
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in random_vectors(rng, 1, 384, "general")]
    qs = fm.fm_classify_tiles(*vec, causal=True)
    q8, k8, v8 = ((x.float() / (x.float().abs().max() / 448)).to(torch.float8_e4m3fn).cuda() for x in (q, k, v))
    fm.fm_attn_fwd_fp8(q8, k8, v8, *vec, qs, q_scale=1.0, k_scale=1.0, v_scale=1.0, scale=0.01, causal=True)
    status_ok("fp8 forward")
    # per-head and multi-interval masks (one launch over every head / interval)
    for d in (64, 128, 256):
        B, hq, hkv, n = 1, 4, 2, 389
        q, k, v, do = tensors.make_qkvdo(dict(B=B, H_q=hq, H_kv=hkv, N=n, d=d))
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        per = [torch.from_numpy(np.ascontiguousarray(x.reshape(B, hq, n))).cuda()
               for x in random_vectors(rng, B * hq, n, "general")]
        fm.fm_attn_per_head(qd, kd, vd, *per, causal=True, scale=d ** -0.5, do=dod)
        status_ok(f"per-head d={d}")
        cuts = np.sort(rng.integers(0, n + 1, size=(6, B, n)), axis=0)
        fms = torch.from_numpy(cuts[0::2].astype(np.int32)).cuda()
        fme = torch.from_numpy((cuts[1::2] - 1).astype(np.int32)).cuda()
        o, lse, dq, dk, dvv = fm.fm_attn_multi_interval(qd, kd, vd, fms, fme, scale=d ** -0.5, do=dod)
        status_ok(f"multi-interval d={d}")
        spec = {"fms": cuts[0::2].transpose(1, 0, 2), "fme": (cuts[1::2] - 1).transpose(1, 0, 2)}
        O, L = oracle.forward(f64(q), f64(k), f64(v), spec, False, d ** -0.5)
        assert_out(f64(o), O)
        ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), spec, False, d ** -0.5)
        for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dvv), ref):
            assert_grad(f64(a), r, name)
    print("debug build clean")


if __name__ == "__main__":
    main()
