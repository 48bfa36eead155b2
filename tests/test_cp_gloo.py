"""The context-parallel protocol of FlashMask-3 project page, §3.2-3.4, run by
two CPU processes over gloo, with the oracle as each rank's attention: the
balancer deals the query chunks, each rank holds the Q, K, V, dO rows of its
own chunks, all-gathers K and V, localizes the global mask vectors to its rows
(no mask bytes move), computes its rows against every key, and reduces the
key gradients so that each rank ends with dK, dV of its own chunks. Every
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
    # every rank derives the same deal from the global mask (deterministic)
    cls = oracle.classify_tiles(*vec, False, C, C)[None]
    w = ob.chunk_loads(cls, 1, 13, 10)
    owner, _ = ob.ipo(w, world, KAPPA)
    owner = np.asarray(owner)
    mine = np.sort(np.nonzero(owner == rank)[0])
    rows = _rows(mine)
    # this rank's shards: Q / dO rows and K / V rows of its own chunks
    k_sh = torch.from_numpy(np.ascontiguousarray(k[:, :, rows]))
    v_sh = torch.from_numpy(np.ascontiguousarray(v[:, :, rows]))
    # all-gather K and V, then place every rank's rows at their global positions
    ks = [torch.empty_like(k_sh) for _ in range(world)]
    vs = [torch.empty_like(v_sh) for _ in range(world)]
    dist.all_gather(ks, k_sh)
    dist.all_gather(vs, v_sh)
    k_full, v_full = np.empty_like(k), np.empty_like(v)
    for r in range(world):
        rr = _rows(np.sort(np.nonzero(owner == r)[0]))
        k_full[:, :, rr] = ks[r].numpy()
        v_full[:, :, rr] = vs[r].numpy()
    # zero-communication localization of the (replicated) global vectors
    loc = tuple(oracle.localize(x, mine * C, C)[None] for x in vec)
    O_r, L_r = oracle.forward(q[:, :, rows], k_full, v_full, loc, False, scale)
    dQ_r, dK_p, dV_p = oracle.backward(q[:, :, rows], k_full, v_full, do[:, :, rows], loc, False, scale)
    # reduce the key gradients of all ranks; keep this rank's own key rows
    dK_t, dV_t = torch.from_numpy(dK_p), torch.from_numpy(dV_p)
    dist.all_reduce(dK_t)
    dist.all_reduce(dV_t)
    out[rank] = (rows, O_r, L_r, dQ_r, dK_t.numpy()[:, :, rows], dV_t.numpy()[:, :, rows])
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
        rows, O_r, L_r, dQ_r, dK_r, dV_r = out[r]
        seen.append(rows)
        assert np.allclose(O_r, O[:, :, rows], atol=1e-12)
        assert np.array_equal(np.isneginf(L_r), np.isneginf(L[:, :, rows]))
        assert np.allclose(dQ_r, dQ[:, :, rows], atol=1e-12)
        assert np.allclose(dK_r, dK[:, :, rows], atol=1e-10)
        assert np.allclose(dV_r, dV[:, :, rows], atol=1e-10)
    assert np.array_equal(np.sort(np.concatenate(seen)), np.arange(N))
