"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the parity contract (all floating point vs the fp64 oracle).
O_REL_L2, O_MAX_ABS = 5e-3, 2e-2
GRAD_REL_L2 = 1e-2
LSE_MAX_ABS = 1e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    if den == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / den)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def vec_np(cfg):
    return tuple(cfg[n] for n in ("lts", "lte", "uts", "ute"))


def vec_dev(cfg, dev="cuda"):
    return [torch.from_numpy(np.ascontiguousarray(cfg[n])).to(dev) for n in ("lts", "lte", "uts", "ute")]


def assert_lse(lse_gpu: np.ndarray, lse_ref: np.ndarray):
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), inf_ref), "fully-masked rows differ"
    if (~inf_ref).any():
        err = np.abs(lse_gpu[~inf_ref] - lse_ref[~inf_ref]).max()
        assert err <= LSE_MAX_ABS, f"LSE max-abs {err}"


def assert_out(o_gpu: np.ndarray, o_ref: np.ndarray):
    r = rel_l2(o_gpu, o_ref)
    m = float(np.abs(o_gpu - o_ref).max()) if o_ref.size else 0.0
    assert r <= O_REL_L2 and m <= O_MAX_ABS, f"O rel-L2 {r:.3e} max-abs {m:.3e}"


def assert_grad(g_gpu: np.ndarray, g_ref: np.ndarray, name: str):
    r = rel_l2(g_gpu, g_ref)
    assert r <= GRAD_REL_L2, f"{name} rel-L2 {r:.3e}"


def random_vectors(rng, B, n, kind="general"):
    """(B, N) int32 boundary vectors of a random kind (test inputs)."""
    out = []
    for _ in range(B):
        if kind == "general":
            a = rng.integers(0, n + 1, size=(2, n))
            c = rng.integers(0, n + 1, size=(2, n))
            v = (a.min(0), a.max(0), c.min(0), c.max(0))
        elif kind == "lower":
            v = (rng.integers(0, n + 1, size=n), np.full(n, n), np.zeros(n, np.int64), np.zeros(n, np.int64))
        else:
            raise KeyError(kind)
        out.append(tuple(x.astype(np.int32) for x in v))
    return tuple(np.stack(x) for x in zip(*out))
