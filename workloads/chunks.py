"""Seeded chunk-load instances for the chunk balancer (inputs only).

The instance families of the "IPO phase ablation" table (FlashMask-3 project
page, §4): (n chunks, P ranks, kappa chunks per rank, w_max). The table does
not say how its random loads are drawn; the reading used here:
  - "uniform": i.i.d. integers in [1, w_max];
  - "causal": a load that grows with the chunk's position, as under a causal
    mask, with a random fraction of a step: w_i = max(1, round(w_max * (i + u_i) / n)),
    u_i uniform in [0, 1).
"""
from __future__ import annotations

import numpy as np

# name: (kind, n, P, kappa, w_max, instances)
TABLE = {
    "uniform": ("uniform", 64, 16, 4, 1000, 200),
    "uniform_wide": ("uniform", 64, 16, 4, 10000, 200),
    "causal": ("causal", 64, 8, 8, 200, 200),
    "uniform_128": ("uniform", 128, 16, 8, 200, 100),
}


def random_loads(rng: np.random.Generator, kind: str, n: int, w_max: int) -> np.ndarray:
    """int64 loads of one random instance."""
    if kind == "uniform":
        return rng.integers(1, w_max + 1, size=n).astype(np.int64)
    if kind == "causal":
        u = rng.random(n)
        return np.maximum(1, np.rint(w_max * (np.arange(n) + u) / n)).astype(np.int64)
    raise KeyError(kind)
