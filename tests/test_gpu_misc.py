"""GPU: localization parity (bit-exact) and the bounded-wait error path."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(4))
def test_localize_bit_exact(seed):
    rng = np.random.default_rng(seed)
    P, kappa, C = 4, 3 + seed, 64 + 13 * seed
    n = P * kappa * C
    x = rng.integers(0, n + 1, size=4 * n + 3).astype(np.int32)  # 4 vectors + a ragged tail
    owner = rng.permutation(np.repeat(np.arange(P), kappa))
    for r in range(P):
        offs = (np.sort(np.nonzero(owner == r)[0]) * C).astype(np.int32)
        got = fm.fm_localize(torch.from_numpy(x).cuda(), torch.from_numpy(offs).cuda(), C).cpu().numpy()
        assert np.array_equal(got, oracle.localize(x, offs, C))
        # unaligned start exercises the scalar path
        got2 = fm.fm_localize(torch.from_numpy(x).cuda()[1:], torch.from_numpy(offs).cuda(), C).cpu().numpy()
        assert np.array_equal(got2, oracle.localize(x[1:], offs, C))


def test_bounded_wait_times_out_and_context_survives():
    fm.fm_selftest_wait_timeout(20000)  # 20 ms, no arrival ever comes
    st, bits = fm.fm_device_status()
    assert st == fm.FM_ERR_TIMEOUT and bits & fm.FM_DEVERR_TIMEOUT
    # the context is still usable and the word was cleared
    x = torch.arange(10, dtype=torch.int32, device="cuda")
    y = fm.fm_localize(x, torch.tensor([0], dtype=torch.int32, device="cuda"), 4)
    assert y.cpu().tolist() == [0, 1, 2, 3, 4, 4, 4, 4, 4, 4]
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK and bits == 0


def test_host_buffer_entry_point_matches_device_calls():
    # fm_attn_fwd_bwd_host runs the same kernels on copies of host buffers:
    # O, LSE, dK, dV bit for bit; dQ (fp32 reductions in any order) within the
    # parity tolerance
    import ctypes

    import mask_aware_sparse_gb300 as fm
    from workloads import masks, tensors

    from helpers import GRAD_REL_L2, rel_l2

    rng = np.random.default_rng(4)
    n = 1000
    v_ = masks.causal_documents(masks.draw_fill(rng, n, 100, 400), n)
    cfg = dict(B=1, H_q=4, H_kv=2, N=n, d=128)
    q, k, v, do = tensors.make_qkvdo(cfg)
    vec = [torch.from_numpy(np.ascontiguousarray(x[None])) for x in v_]
    scale = 128 ** -0.5
    pin = lambda t: t.pin_memory()
    out = fm.fm_attn_fwd_bwd_host(pin(q), pin(k), pin(v), pin(do), *[pin(x) for x in vec], scale=scale, causal=True)
    torch.cuda.synchronize()
    dvec = [x.cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dvec, causal=True)
    o, lse = fm.fm_attn_fwd(q.cuda(), k.cuda(), v.cuda(), *dvec, qs, scale=scale, causal=True)
    dq, dk, dv = fm.fm_attn_bwd(q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda(), *dvec, qs, scale=scale, causal=True)
    assert fm.fm_device_status()[0] == fm.FM_OK
    for a, b in ((out[0], o), (out[1], lse), (out[3], dk), (out[4], dv)):
        assert torch.equal(a, b.cpu())
    assert rel_l2(out[2].double().numpy(), dq.double().cpu().numpy()) <= GRAD_REL_L2 / 10
    # host tensors only: a device tensor is refused before any call
    with pytest.raises(ValueError):
        fm.fm_attn_fwd_bwd_host(q.cuda(), k, v, do, *vec, scale=scale, causal=True)
