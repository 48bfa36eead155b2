"""Seeded mask encoders: build the four column-wise boundary vectors.

This module only builds inputs. It holds none of the attention arithmetic:
it turns a description of a packed sequence (documents, prompts and
responses, a window, an eviction row per key) into the FlashMask
column-wise representation that both the CUDA path and the oracle consume.

Representation (FlashMask-3 project page, "Overview": the four column-wise
boundary vectors LTS, LTE, UTS, UTE, indexed by key column and holding
query-row boundaries). For key column j the masked query rows are the two
half-open intervals [LTS_j, LTE_j) and [UTS_j, UTE_j); with the causal flag
set, rows i < j are masked as well. An interval with start >= end is empty.

All vectors are int32 numpy arrays of shape (N,), values in [0, N].
"""
from __future__ import annotations

import numpy as np

I32 = np.int32


def _empty(n: int):
    lts = np.full(n, n, dtype=I32)
    lte = np.full(n, n, dtype=I32)
    uts = np.zeros(n, dtype=I32)
    ute = np.zeros(n, dtype=I32)
    return lts, lte, uts, ute


def causal_documents(lengths, n: int):
    """Causal document packing: a row sees key j only inside j's document.

    Key columns of a document [s, e) get LTS = e and LTE = N, so every later
    row (a later document) is masked; the causal flag masks earlier rows.
    Returns (lts, lte, uts, ute); use with causal=True.
    """
    lts, lte, uts, ute = _empty(n)
    s = 0
    for length in lengths:
        e = min(s + int(length), n)
        lts[s:e] = e
        s = e
        if s >= n:
            break
    if s < n:  # uncovered tail is its own document
        lts[s:n] = n
    return lts, lte, uts, ute


def share_question(samples, n: int):
    """Share-question / DPO packing, causal.

    `samples` is a list of (prompt, response_a, response_b) lengths laid out
    back to back. Both responses see their prompt but not each other, and no
    row sees an earlier sample. Encoding (one interval per column suffices):
      prompt keys     LTS = end of the sample
      response-a keys LTS = start of response b (masks b and everything after)
      response-b keys LTS = end of the sample
    Keys beyond the last sample are padding: LTS = end of the last sample,
    which masks those rows and columns completely (fully-masked rows).
    """
    lts, lte, uts, ute = _empty(n)
    s = 0
    for p, a, b in samples:
        e = s + p + a + b
        if e > n:
            raise ValueError("samples overflow the sequence")
        lts[s : s + p] = e
        lts[s + p : s + p + a] = s + p + a
        lts[s + p + a : e] = e
        s = e
    lts[s:n] = s
    return lts, lte, uts, ute


def prefix_lm_documents(lengths, n: int, prefix_frac: float = 0.25):
    """Prefix-LM document packing, NON-causal mode.

    Document [s, e) of length L has a bidirectional prefix of floor(L*frac)
    tokens. Every key column of the document has LTS = e, LTE = N (later
    documents are masked). Prefix keys have UTS = 0, UTE = s (earlier
    documents masked); a non-prefix key j has UTS = 0, UTE = j (rows before j
    masked: causal inside the document).
    """
    lts, lte, uts, ute = _empty(n)
    s = 0
    for length in lengths:
        e = min(s + int(length), n)
        L = e - s
        p = int(np.floor(L * prefix_frac))
        lts[s:e] = e
        ute[s : s + p] = s
        ute[s + p : e] = np.arange(s + p, e, dtype=I32)
        s = e
        if s >= n:
            break
    if s < n:
        raise ValueError("document lengths do not fill the sequence")
    return lts, lte, uts, ute


def sliding_window(n: int, window: int, sinks: int):
    """Causal sliding window with attention sinks.

    Key j >= sinks is evicted from row j + window on (LTS = min(j+window, N),
    LTE = N); sink keys j < sinks are never evicted (empty interval).
    Row i then sees key j iff j <= i < j + window, or j < sinks (and j <= i).
    """
    lts, lte, uts, ute = _empty(n)
    j = np.arange(n, dtype=np.int64)
    lts[:] = np.minimum(j + window, n).astype(I32)
    lts[: min(sinks, n)] = n
    return lts, lte, uts, ute


def random_eviction(n: int, p: float, rng: np.random.Generator):
    """Causal random eviction: key j is evicted at row j + G_j, G_j ~ Geometric(p).

    numpy's geometric distribution has support {1, 2, ...}, so the diagonal
    is always visible. LTS = min(j + G_j, N), LTE = N.
    """
    lts, lte, uts, ute = _empty(n)
    g = rng.geometric(p, size=n).astype(np.int64)
    lts[:] = np.minimum(np.arange(n, dtype=np.int64) + g, n).astype(I32)
    return lts, lte, uts, ute


# ---------------------------------------------------------------- draws
def draw_tiny_split(rng: np.random.Generator, n: int = 256, min_len: int = 32):
    """Three documents: two distinct cut points uniform in 1..n-1, all >= min_len."""
    while True:
        c = np.sort(rng.choice(np.arange(1, n), size=2, replace=False))
        lens = [int(c[0]), int(c[1] - c[0]), int(n - c[1])]
        if min(lens) >= min_len:
            return lens


def draw_fill(rng: np.random.Generator, n: int, lo: int, hi: int):
    """Lengths uniform in [lo, hi] until they cover n; the last is truncated."""
    lens, tot = [], 0
    while tot < n:
        L = int(rng.integers(lo, hi, endpoint=True))
        L = min(L, n - tot)
        lens.append(L)
        tot += L
    return lens


def draw_share_question(rng: np.random.Generator, n_samples: int = 8, prompt=(512, 2048), resp=(256, 1024)):
    out = []
    for _ in range(n_samples):
        p = int(rng.integers(prompt[0], prompt[1], endpoint=True))
        a = int(rng.integers(resp[0], resp[1], endpoint=True))
        b = int(rng.integers(resp[0], resp[1], endpoint=True))
        out.append((p, a, b))
    return out
