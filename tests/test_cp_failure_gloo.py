"""A rank lost in the middle of the context-parallel protocol (FlashMask-3
project page, §3.2-3.4), emulated on host ranks: three CPU processes over gloo,
the oracle as each rank's attention, the library's host balancer
(fm_balance_chunks) and exchange plan (fm_needed_chunks) for the deal.

Protocol, per epoch:
  1. deal: every member derives the same chunk owners from the global mask
     (fm_chunk_loads -> fm_balance_chunks over the members, kappa = chunks /
     members) and the same pruned K / V exchange plan (fm_needed_chunks);
  2. K / V exchange: a chunk goes from its owner to the members that need it;
  3. each member localizes the replicated vectors and computes its rows;
  4. heartbeat: before the key-gradient exchange every member announces itself
     in the store; rank 0 (which hosts the store, so its own loss ends the job)
     waits a bounded time for the others and publishes who did not arrive;
  5. if nobody is missing, key gradients go back to each chunk's owner and the
     epoch is final; otherwise the members that arrived drop this epoch's
     results and run the next epoch over themselves (a fresh deal and a full
     recompute: the lost rank's K / V, Q and dO chunks are re-read from the
     inputs, which every rank can regenerate).
Rank 2 leaves after the K / V exchange of epoch 0 (it exits between steps,
with no exchange in flight). The survivors must detect it within the bounded
wait, re-deal the 12 chunks over two ranks (6 each) and still produce the whole
problem's O, LSE, dQ and dK / dV for every row. No GPU is involved.
"""
import json
import os
import socket
from datetime import timedelta

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import mask_aware_sparse_gb300 as fm
import oracle
from mask_aware_sparse_gb300 import build as fmbuild
from oracle import balance as ob

from test_cp_oracle import cases

N, C, D, HQ, HKV = 384, 32, 16, 2, 1
WORLD = 3                          # 12 chunks: 3 ranks x 4, then 2 survivors x 6
HEARTBEAT = timedelta(seconds=3)   # bounded wait that detects a lost rank
STORE_TIMEOUT = timedelta(seconds=60)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fmbuild.build()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _problem(name):
    vec = tuple(np.asarray(x, np.int32) for x in cases(N)[name])
    rng = np.random.default_rng(5)
    q, do = (rng.standard_normal((1, HQ, N, D)) for _ in range(2))
    k, v = (rng.standard_normal((1, HKV, N, D)) for _ in range(2))
    return vec, q, k, v, do


def _deal(cls, members):
    """Chunk owners (actual ranks) and the pruned exchange plan over `members`."""
    P, n = len(members), cls.shape[1]
    w = fm.fm_chunk_loads(cls, 1, 13, 10)
    owner_v, _ = fm.fm_balance_chunks(w, P, n // P)
    need_v = fm.fm_needed_chunks(cls, owner_v, P, 1)
    owner = np.asarray(members)[owner_v]
    return owner, {members[i]: need_v[i] for i in range(P)}


def _rows(owner, rank):
    return np.concatenate([np.arange(c * C, (c + 1) * C) for c in np.sort(np.nonzero(owner == rank)[0])])


def _exchange_kv(rank, members, owner, need, k, v, tag):
    rows = _rows(owner, rank)
    k_full, v_full = np.zeros_like(k), np.zeros_like(v)
    k_full[:, :, rows], v_full[:, :, rows] = k[:, :, rows], v[:, :, rows]
    reqs, recv = [], []
    for c in range(owner.size):
        cr = np.arange(c * C, (c + 1) * C)
        src = int(owner[c])
        if src == rank:
            for dst in members:
                if dst != rank and need[dst][c]:
                    kv = torch.from_numpy(np.ascontiguousarray(np.concatenate([k[:, :, cr], v[:, :, cr]], 1)))
                    reqs.append(dist.isend(kv, dst, tag=tag + c))
        elif need[rank][c]:
            buf = torch.empty((1, 2 * HKV, C, D), dtype=torch.float64)
            reqs.append(dist.irecv(buf, src, tag=tag + c))
            recv.append((cr, buf))
    for r in reqs:
        r.wait()
    for cr, buf in recv:
        k_full[:, :, cr], v_full[:, :, cr] = buf[:, :HKV].numpy(), buf[:, HKV:].numpy()
    return k_full, v_full


def _return_key_grads(rank, members, owner, need, dK_p, dV_p, tag):
    dK_own, dV_own = dK_p.copy(), dV_p.copy()
    reqs, recv = [], []
    for c in range(owner.size):
        cr = np.arange(c * C, (c + 1) * C)
        dst = int(owner[c])
        if dst != rank and need[rank][c]:
            g = torch.from_numpy(np.ascontiguousarray(np.concatenate([dK_p[:, :, cr], dV_p[:, :, cr]], 1)))
            reqs.append(dist.isend(g, dst, tag=tag + c))
        elif dst == rank:
            for src in members:
                if src != rank and need[src][c]:
                    buf = torch.empty((1, 2 * HKV, C, D), dtype=torch.float64)
                    reqs.append(dist.irecv(buf, src, tag=tag + c))
                    recv.append((cr, buf))
    for r in reqs:
        r.wait()
    for cr, buf in recv:
        dK_own[:, :, cr] += buf[:, :HKV].numpy()
        dV_own[:, :, cr] += buf[:, HKV:].numpy()
    return dK_own, dV_own


def _heartbeat(store, epoch, rank, members):
    """Members of `epoch` that reached its key-gradient exchange. Rank 0 waits
    (bounded) for the others and publishes the missing ones; everyone follows
    rank 0's view, so all survivors agree."""
    store.set(f"ready/{epoch}/{rank}", "1")
    if rank == 0:
        others = [f"ready/{epoch}/{r}" for r in members if r != 0]
        try:
            if others:
                store.wait(others, HEARTBEAT)
            missing = []
        except Exception:  # the bounded wait expired: somebody did not arrive
            missing = [r for r in members if r != 0 and not store.check([f"ready/{epoch}/{r}"])]
        store.set(f"missing/{epoch}", json.dumps(missing))
    missing = json.loads(store.get(f"missing/{epoch}").decode())
    return [r for r in members if r not in missing], missing


def _worker(rank, world, port, name, leaver, out):
    store = dist.TCPStore("127.0.0.1", port, world, rank == 0, timeout=STORE_TIMEOUT)
    dist.init_process_group("gloo", store=store, rank=rank, world_size=world, timeout=STORE_TIMEOUT)
    vec, q, k, v, do = _problem(name)
    scale = D ** -0.5
    cls = oracle.classify_tiles(*vec, False, C, C)[None]
    members, epoch, lost = list(range(world)), 0, []
    while True:
        owner, need = _deal(cls, members)
        k_full, v_full = _exchange_kv(rank, members, owner, need, k, v, tag=1000 * (2 * epoch))
        if rank == leaver and epoch == 0:
            return  # leaves between steps: nothing of its own is in flight
        rows = _rows(owner, rank)
        loc = tuple(oracle.localize(x, np.unique(rows // C) * C, C)[None] for x in vec)
        O_r, L_r = oracle.forward(q[:, :, rows], k_full, v_full, loc, False, scale)
        dQ_r, dK_p, dV_p = oracle.backward(q[:, :, rows], k_full, v_full, do[:, :, rows], loc, False, scale)
        alive, missing = _heartbeat(store, epoch, rank, members)
        if rank not in alive:
            return
        if missing:
            lost += missing
            members, epoch = alive, epoch + 1  # drop this epoch's results, re-deal, recompute
            continue
        dK_own, dV_own = _return_key_grads(rank, members, owner, need, dK_p, dV_p, tag=1000 * (2 * epoch + 1))
        out[rank] = dict(epoch=epoch, members=members, lost=lost, owner=owner, rows=rows, O=O_r, L=L_r, dQ=dQ_r,
                         dK=dK_own[:, :, rows], dV=dV_own[:, :, rows])
        break
    store.set(f"done/{rank}", "1")
    store.wait([f"done/{r}" for r in members], STORE_TIMEOUT)
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["doc_causal_folded", "general"])
@pytest.mark.parametrize("leaver", [None, 2])
def test_cp_rank_failure_detected_redealt_recomputed(name, leaver):
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(WORLD, _free_port(), name, leaver, out), nprocs=WORLD, join=True)
    vec, q, k, v, do = _problem(name)
    vb = tuple(x[None] for x in vec)
    scale = D ** -0.5
    O, L = oracle.forward(q, k, v, vb, False, scale)
    dQ, dK, dV = oracle.backward(q, k, v, do, vb, False, scale)
    survivors = [r for r in range(WORLD) if r != leaver]
    assert sorted(out.keys()) == survivors
    cls = oracle.classify_tiles(*vec, False, C, C)[None]
    n = cls.shape[1]
    seen = []
    for r in survivors:
        res = out[r]
        assert res["members"] == survivors
        assert res["epoch"] == (0 if leaver is None else 1)
        assert res["lost"] == ([] if leaver is None else [leaver])
        # the final deal is the balancer's over the survivors, kappa = n / survivors
        owner_v, _ = ob.ipo(ob.chunk_loads(cls, 1, 13, 10), len(survivors), n // len(survivors))
        assert np.array_equal(res["owner"], np.asarray(survivors)[np.asarray(owner_v)])
        rows = res["rows"]
        seen.append(rows)
        assert np.allclose(res["O"], O[:, :, rows], atol=1e-12)
        assert np.array_equal(np.isneginf(res["L"]), np.isneginf(L[:, :, rows]))
        fin = ~np.isneginf(L[:, :, rows])
        assert np.allclose(res["L"][fin], L[:, :, rows][fin], atol=1e-12)
        assert np.allclose(res["dQ"], dQ[:, :, rows], atol=1e-12)
        assert np.allclose(res["dK"], dK[:, :, rows], atol=1e-10)
        assert np.allclose(res["dV"], dV[:, :, rows], atol=1e-10)
    assert np.array_equal(np.sort(np.concatenate(seen)), np.arange(N))
