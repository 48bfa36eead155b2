"""The context-parallel protocol of FlashMask-3 project page, §3.2-3.4, run by
two CPU processes over gloo, with the oracle as each rank's attention: the
balancer deals the query chunks, each rank holds the Q, K, V, dO rows of its
own chunks and receives only the K / V chunks its rows can see (mask-aware
pruning of the exchange), localizes the global mask vectors to its rows (no
mask bytes move), computes its rows against the keys, and sends its key
gradients back to each chunk's owner, again only for chunks it needed. Every
rank's O, LSE, dQ and its dK, dV shard must equal the whole problem's."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from oracle import balance as ob

from test_cp_oracle import cases

N, C, KAPPA, D, HQ, HKV = 256, 32, 4, 16, 2, 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem(name):
    vec = tuple(np.asarray(x, np.int32) for x in cases(N)[name])
    rng = np.random.default_rng(3)
    q, do = (rng.standard_normal((1, HQ, N, D)) for _ in range(2))
    k, v = (rng.standard_normal((1, HKV, N, D)) for _ in range(2))
    return vec, q, k, v, do


def _rows(chunks):
    return np.concatenate([np.arange(c * C, (c + 1) * C) for c in chunks])


def _worker(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vec, q, k, v, do = _problem(name)
    scale = D ** -0.5
    # every rank derives the same deal and exchange plan from the global mask
    cls = oracle.classify_tiles(*vec, False, C, C)[None]
    owner, _ = ob.ipo(ob.chunk_loads(cls, 1, 13, 10), world, KAPPA)
    owner = np.asarray(owner)
    need = ob.needed_chunks(cls, owner.tolist(), world, 1)
    n = owner.size
    mine = np.sort(np.nonzero(owner == rank)[0])
    rows = _rows(mine)
    # K / V exchange, pruned: a chunk goes from its owner to every other rank
    # that needs it, and nowhere else; chunks nobody sends stay zero (the mask
    # hides them from every row of the receiving rank)
    k_full, v_full = np.zeros_like(k), np.zeros_like(v)
    k_full[:, :, rows], v_full[:, :, rows] = k[:, :, rows], v[:, :, rows]
    reqs, recv = [], []
    for c in range(n):
        cr = np.arange(c * C, (c + 1) * C)
        src = int(owner[c])
        if src == rank:
            for dst in range(world):
                if dst != rank and need[dst, c]:
                    kv = torch.from_numpy(np.ascontiguousarray(np.concatenate([k[:, :, cr], v[:, :, cr]], 1)))
                    reqs.append(dist.isend(kv, dst))
        elif need[rank, c]:
            buf = torch.empty((1, 2 * HKV, C, D), dtype=torch.float64)
            reqs.append(dist.irecv(buf, src))
            recv.append((cr, buf))
    for r in reqs:
        r.wait()
    for cr, buf in recv:
        k_full[:, :, cr], v_full[:, :, cr] = buf[:, :HKV].numpy(), buf[:, HKV:].numpy()
    # zero-communication localization of the (replicated) global vectors
    loc = tuple(oracle.localize(x, mine * C, C)[None] for x in vec)
    O_r, L_r = oracle.forward(q[:, :, rows], k_full, v_full, loc, False, scale)
    dQ_r, dK_p, dV_p = oracle.backward(q[:, :, rows], k_full, v_full, do[:, :, rows], loc, False, scale)
    # key gradients back to each chunk's owner, only from the ranks that
    # needed the chunk (the others' contributions are zero)
    dK_own, dV_own = dK_p.copy(), dV_p.copy()
    reqs, recv = [], []
    for c in range(n):
        cr = np.arange(c * C, (c + 1) * C)
        dst = int(owner[c])
        if dst != rank and need[rank, c]:
            g = torch.from_numpy(np.ascontiguousarray(np.concatenate([dK_p[:, :, cr], dV_p[:, :, cr]], 1)))
            reqs.append(dist.isend(g, dst))
        elif dst == rank:
            for src in range(world):
                if src != rank and need[src, c]:
                    buf = torch.empty((1, 2 * HKV, C, D), dtype=torch.float64)
                    reqs.append(dist.irecv(buf, src))
                    recv.append((cr, buf))
    for r in reqs:
        r.wait()
    for cr, buf in recv:
        dK_own[:, :, cr] += buf[:, :HKV].numpy()
        dV_own[:, :, cr] += buf[:, HKV:].numpy()
    sent = int(sum(need[r, c] for c in range(n) for r in range(world) if owner[c] != r))
    out[rank] = (rows, O_r, L_r, dQ_r, dK_own[:, :, rows], dV_own[:, :, rows], sent, world * n - n)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["doc_causal_folded", "prefix_lm", "general"])
def test_cp_protocol_two_ranks_gloo(name):
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), name, out), nprocs=world, join=True)
    vec, q, k, v, do = _problem(name)
    vb = tuple(x[None] for x in vec)
    scale = D ** -0.5
    O, L = oracle.forward(q, k, v, vb, False, scale)
    dQ, dK, dV = oracle.backward(q, k, v, do, vb, False, scale)
    seen = []
    for r in range(world):
        rows, O_r, L_r, dQ_r, dK_r, dV_r, sent, remote = out[r]
        if name == "doc_causal_folded":
            assert sent < remote  # pruning drops chunks the mask hides
        seen.append(rows)
        assert np.allclose(O_r, O[:, :, rows], atol=1e-12)
        assert np.array_equal(np.isneginf(L_r), np.isneginf(L[:, :, rows]))
        assert np.allclose(dQ_r, dQ[:, :, rows], atol=1e-12)
        assert np.allclose(dK_r, dK[:, :, rows], atol=1e-10)
        assert np.allclose(dV_r, dV[:, :, rows], atol=1e-10)
    assert np.array_equal(np.sort(np.concatenate(seen)), np.arange(N))
