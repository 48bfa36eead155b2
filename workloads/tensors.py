"""Seeded bf16 tensors for a workload: Q, K, V, dO ~ N(0, 1).

Drawn in fp32 from torch CPU generators seeded 1, 2, 3, 4 (Q, K, V, dO in
that order) and rounded to bf16 (round-to-nearest-even). Layout is
contiguous (B, H, N, d). The oracle widens exactly these bf16 values.
"""
from __future__ import annotations

import torch


def randn_bf16(shape, seed: int, device="cpu"):
    """N(0,1) bf16 tensor. CPU draws are the reference; `device` only moves it.

    For very large benchmark inputs `device="cuda"` draws directly on the GPU
    with a seeded CUDA generator (a different stream of numbers, same law).
    """
    if str(device).startswith("cuda"):
        g = torch.Generator(device=device).manual_seed(seed)
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_qkvdo(cfg: dict, device="cpu", heads_q=None):
    """Return (q, k, v, do) bf16 tensors for workload `cfg`.

    heads_q: optional number of query heads to draw instead of cfg["H_q"]
    (used for head-subset parity runs; the first heads of the full draw are
    NOT reproduced — subsets are drawn as their own seeded tensors).
    """
    B, Hq, Hkv, N, d = cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N"], cfg["d"]
    if heads_q is not None:
        Hq = heads_q
    q = randn_bf16((B, Hq, N, d), 1, device)
    k = randn_bf16((B, Hkv, N, d), 2, device)
    v = randn_bf16((B, Hkv, N, d), 3, device)
    do = randn_bf16((B, Hq, N, d), 4, device)
    return q, k, v, do
