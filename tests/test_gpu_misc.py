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
