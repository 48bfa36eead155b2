"""fm_attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc when they run the forward, for example a
plugin inside a host framework that owns all device memory and gives plugins
no allocator, or a service that reserves its memory once at start-up. For them
the library keeps the forward's only scratch (its launch-order table) in a
fixed array of its own. These tests call that entry point through the C ABI,
twice in a row (the array keeps the previous call's contents), and compare with
the ordinary fm_attn_fwd, which takes a caller-provided workspace. Inputs and
outputs are still allocated by the test: only the scratch is the library's.
"""
import ctypes

import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
from workloads import masks, tensors


pytestmark = pytest.mark.gpu


def _noalloc(prob, q, k, v, vec, queues, o, lse):
    P = fm._ptr
    return fm.lib().fm_attn_fwd_noalloc(ctypes.byref(prob), P(q), P(k), P(v), *(P(x) for x in vec),
                                        P(queues.q_off), P(queues.q_queue), P(o), P(lse), fm._stream())


def _case(n, hq, hkv, causal, vec_np, seed):
    cfg = dict(B=vec_np[0].shape[0], H_q=hq, H_kv=hkv, N=n, d=128)
    q, k, v, _ = (t.cuda() for t in tensors.make_qkvdo(cfg))
    vec = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec_np]
    queues = fm.fm_classify_tiles(*vec, causal=causal)
    scale = 128 ** -0.5
    o_ref, lse_ref = fm.fm_attn_fwd(q, k, v, *vec, queues, scale=scale, causal=causal)
    prob = fm._problem(cfg["B"], hq, hkv, n, 128, scale, causal)
    return prob, q, k, v, vec, queues, o_ref, lse_ref


def _compare(o, lse, o_ref, lse_ref):
    # the same kernel on the same inputs: every unit is computed the same way
    # whichever CTA takes it, so the results agree bit for bit
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_noalloc_forward_matches_forward_twice():
    rng = np.random.default_rng(5)
    n = 1024
    vec_np = tuple(x[None] for x in masks.causal_documents(masks.draw_fill(rng, n, 100, 400), n))
    prob, q, k, v, vec, queues, o_ref, lse_ref = _case(n, 4, 2, True, vec_np, 0)
    for _ in range(2):  # the second call reuses whatever the first left in the array
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(prob, q, k, v, vec, queues, o, lse) == fm.FM_OK
        torch.cuda.synchronize()
        _compare(o, lse, o_ref, lse_ref)
    assert fm.fm_device_status()[0] == fm.FM_OK


def test_noalloc_second_problem_after_a_larger_one():
    # a smaller problem after a larger one must not see stale order entries
    rng = np.random.default_rng(6)
    for n in (2048, 384):
        vec_np = (masks.random_eviction(n, 1 / 64, rng),)[0]
        vec_np = tuple(x[None] for x in vec_np)
        prob, q, k, v, vec, queues, o_ref, lse_ref = _case(n, 2, 1, True, vec_np, 1)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(lse_ref)
        assert _noalloc(prob, q, k, v, vec, queues, o, lse) == fm.FM_OK
        torch.cuda.synchronize()
        _compare(o, lse, o_ref, lse_ref)


def test_noalloc_long_pass_natural_order():
    # eight or more waves of work units: the forward takes its units in natural
    # order, so only the work counter of the fixed array is used (no order table)
    rng = np.random.default_rng(7)
    n = 32768
    vec_np = tuple(x[None] for x in masks.causal_documents(masks.draw_fill(rng, n, 256, 2048), n))
    prob, q, k, v, vec, queues, o_ref, lse_ref = _case(n, 8, 8, True, vec_np, 2)
    units = 8 * (n // 128)
    assert units >= 8 * torch.cuda.get_device_properties(0).multi_processor_count
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        assert _noalloc(prob, q, k, v, vec, queues, o, lse) == fm.FM_OK
        torch.cuda.synchronize()
        _compare(o, lse, o_ref, lse_ref)
    assert fm.fm_device_status()[0] == fm.FM_OK


def test_noalloc_rejects_too_many_q_blocks():
    # B * ceil(N / 128) above the fixed capacity: refused before anything runs
    n = 128 * 1024                    # 1024 Q blocks per batch entry
    max_qblocks = 65536               # FM_NOALLOC_MAX_QBLOCKS in include/fm.h
    batch = max_qblocks // 1024 + 1
    prob = fm._problem(batch, 2, 1, n, 128, 0.1, 1)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    P = fm._ptr
    st = fm.lib().fm_attn_fwd_noalloc(ctypes.byref(prob), *([P(dummy)] * 11), fm._stream())
    assert st == fm.FM_ERR_WORKSPACE
