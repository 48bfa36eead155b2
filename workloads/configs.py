"""The benchmark workloads, as seeded synthetic inputs.

Each workload is a dict with the problem shape and the (B, N) int32 boundary
vectors. Structure seed 0 (numpy default_rng) draws the mask; tensors are
drawn by `workloads.tensors` from torch CPU generators seeded 1..4 for
Q, K, V and dO. None of the pages' datasets is available; these seeded masks
stand in for the mask families the pages evaluate (document packing,
share-question / DPO, prefix-LM, sliding window with sinks, random eviction).
"""
from __future__ import annotations

import numpy as np

from . import masks

NAMES = ("tiny", "doc8k", "share_question32k", "prefix_lm64k", "sliding_window64k", "eviction128k")


def _stack(vecs, batch):
    return tuple(np.stack([v] * batch).astype(np.int32) for v in vecs)


def make(name: str, seed: int = 0, **over) -> dict:
    """Build workload `name` (one of NAMES). Keyword overrides replace shape keys."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        n = over.get("N", 256)
        lens = masks.draw_tiny_split(rng, n)
        vecs = masks.causal_documents(lens, n)
        cfg = dict(B=1, H_q=2, H_kv=2, N=n, d=64, causal=True, tile=(64, 64), docs=lens)
    elif name == "doc8k":
        n = over.get("N", 8192)
        lens = masks.draw_fill(rng, n, 256, 2048)
        vecs = masks.causal_documents(lens, n)
        cfg = dict(B=1, H_q=32, H_kv=8, N=n, d=128, causal=True, docs=lens)
    elif name == "share_question32k":
        n = over.get("N", 32768)
        samples = masks.draw_share_question(rng)
        vecs = masks.share_question(samples, n)
        cfg = dict(B=1, H_q=32, H_kv=8, N=n, d=128, causal=True, samples=samples)
    elif name == "prefix_lm64k":
        n = over.get("N", 65536)
        lens = masks.draw_fill(rng, n, 2048, 16384)
        vecs = masks.prefix_lm_documents(lens, n)
        cfg = dict(B=1, H_q=64, H_kv=8, N=n, d=128, causal=False, docs=lens)
    elif name == "sliding_window64k":
        n = over.get("N", 65536)
        vecs = masks.sliding_window(n, 4096, 4)
        cfg = dict(B=1, H_q=64, H_kv=8, N=n, d=128, causal=True, window=4096, sinks=4)
    elif name == "eviction128k":
        n = over.get("N", 131072)
        vecs = masks.random_eviction(n, 1.0 / 16384, rng)
        cfg = dict(B=1, H_q=64, H_kv=1, N=n, d=128, causal=True)
    else:
        raise KeyError(name)
    cfg.setdefault("tile", (128, 128))
    cfg.update({k: v for k, v in over.items() if k in ("B", "H_q", "H_kv", "d")})
    cfg["name"] = name
    cfg["scale"] = 1.0 / float(np.sqrt(cfg["d"]))
    cfg["lts"], cfg["lte"], cfg["uts"], cfg["ute"] = _stack(vecs, cfg["B"])
    return cfg
