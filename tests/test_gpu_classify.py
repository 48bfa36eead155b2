"""GPU tile classification and queues: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import mask_aware_sparse_gb300 as fm
import oracle
from workloads import configs

from helpers import random_vectors, vec_dev, vec_np

pytestmark = pytest.mark.gpu


def _check(vec, causal, bm, bn):
    B, N = vec[0].shape
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    qs = fm.fm_classify_tiles(*dv, causal=causal, block_m=bm, block_n=bn)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_OK, bits
    cls_ref = [oracle.classify_tiles(*(x[b] for x in vec), causal, bm, bn) for b in range(B)]
    q_off, q_q, k_off, k_q = oracle.build_queues(cls_ref)
    assert np.array_equal(qs.tile_class.cpu().numpy(), np.stack(cls_ref))
    assert np.array_equal(qs.q_off.cpu().numpy(), q_off)
    assert np.array_equal(qs.k_off.cpu().numpy(), k_off)
    assert np.array_equal(qs.q_queue.cpu().numpy()[: len(q_q)], q_q)
    assert np.array_equal(qs.k_queue.cpu().numpy()[: len(k_q)], k_q)


@pytest.mark.parametrize("name", configs.NAMES)
def test_classify_full_configs(name):
    cfg = configs.make(name)
    bm, bn = cfg["tile"]
    _check(vec_np(cfg), cfg["causal"], bm, bn)
    if (bm, bn) != (128, 128):
        _check(vec_np(cfg), cfg["causal"], 128, 128)


@pytest.mark.parametrize("tile", [(32, 32), (64, 128), (128, 64), (256, 128), (128, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_classify_random_general(tile, causal):
    rng = np.random.default_rng(hash((tile, causal)) % 1000)
    for n in (1, 77, 256, 1000):
        vec = random_vectors(rng, 2, n, "general")
        _check(vec, causal, *tile)


def test_classify_out_of_range_is_flagged():
    n = 256
    rng = np.random.default_rng(0)
    vec = list(random_vectors(rng, 1, n, "lower"))
    vec[0] = vec[0].copy()
    vec[0][0, 5] = n + 7
    dv = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in vec]
    fm.fm_classify_tiles(*dv, causal=True)
    st, bits = fm.fm_device_status()
    assert st == fm.FM_ERR_DEVICE and bits & fm.FM_DEVERR_RANGE
    st, bits = fm.fm_device_status()  # cleared
    assert st == fm.FM_OK and bits == 0
