"""Host-side logic of bench.py: the metric's pair count and the multi-rank
aggregation (weak scaling: total work over the slowest rank's time)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from workloads import configs, masks


def _vec(cfg):
    return tuple(cfg[n][0] for n in ("lts", "lte", "uts", "ute"))


@pytest.mark.parametrize("name", ["tiny", "doc8k"])
def test_visible_pairs_matches_oracle_on_workloads(name):
    cfg = configs.make(name)
    assert bench.visible_pairs(*_vec(cfg), cfg["causal"]) == oracle.unmasked_pairs(_vec(cfg), cfg["causal"])


def test_visible_pairs_general_vectors():
    rng = np.random.default_rng(0)
    for causal in (False, True):
        for _ in range(20):
            n = int(rng.integers(1, 90))
            a = rng.integers(0, n + 1, size=(2, n))
            c = rng.integers(0, n + 1, size=(2, n))
            vec = (a[0], a[1], c[0], c[1])  # includes reversed (empty) intervals
            vec = tuple(x.astype(np.int32) for x in vec)
            assert bench.visible_pairs(*vec, causal) == oracle.unmasked_pairs(vec, causal)


def test_closed_blocks_are_closed():
    cfg = configs.make("tiny")
    vis = ~oracle.dense_mask(*_vec(cfg), True)
    for r0, r1 in bench.closed_blocks(cfg):
        inside = np.zeros(cfg["N"], bool)
        inside[r0:r1] = True
        assert not vis[inside][:, ~inside].any() and not vis[~inside][:, inside].any()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r pretends its timed region took 1 + r seconds for the same work
    tot, tmax = bench.aggregate(10.0, 1.0 + rank, world, torch.device("cpu"))
    out[rank] = (tot, tmax)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == (20.0, 2.0)  # sum of work, max of times


def test_closed_block_subproblem_equals_full_problem():
    """The oracle on a closed block's own tensors reproduces the full problem's rows."""
    rng = np.random.default_rng(1)
    samples = [(5, 3, 4), (6, 2, 2)]
    n = 26
    cfg = dict(B=1, H_q=2, H_kv=1, N=n, d=8, causal=True, scale=0.3, samples=samples)
    vec = tuple(x[None] for x in masks.share_question(samples, n))
    cfg.update(zip(("lts", "lte", "uts", "ute"), vec))
    g = torch.Generator().manual_seed(0)
    q, k, v, do = (torch.randn(1, h, n, 8, generator=g, dtype=torch.float64) for h in (2, 1, 1, 2))
    O, L = oracle.forward(q.numpy(), k.numpy(), v.numpy(), vec, True, 0.3)
    dQ, dK, dV = oracle.backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), vec, True, 0.3)
    for (r0, r1) in bench.closed_blocks(cfg):
        sub = bench.sub_vectors(cfg, (r0, r1))
        sl = slice(r0, r1)
        Os, Ls = oracle.forward(q[:, :, sl].numpy(), k[:, :, sl].numpy(), v[:, :, sl].numpy(), sub, True, 0.3)
        dQs, dKs, dVs = oracle.backward(q[:, :, sl].numpy(), k[:, :, sl].numpy(), v[:, :, sl].numpy(),
                                        do[:, :, sl].numpy(), sub, True, 0.3)
        assert np.allclose(Os, O[:, :, sl], atol=1e-13) and np.allclose(dQs, dQ[:, :, sl], atol=1e-13)
        assert np.allclose(dKs, dK[:, :, sl], atol=1e-13) and np.allclose(dVs, dV[:, :, sl], atol=1e-13)


def test_bench_balance_line_without_gpu():
    """`bench.py --balance` prints one JSON line; it always measures the
    ablation table's families, and the workloads' chunk loads where a GPU
    runs the classifier."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--balance", "--no-cpu-baseline"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["unit"] == "ratio" and line["higher_is_better"] is False
    assert set(line["table"]) == {"uniform", "uniform_wide", "causal", "uniform_128"}
    t = line["table"]["causal"]
    assert t["lb_certified"] == t["instances"] == 200
    for c in line["cases"]:
        poa = c["peak_over_avg"]
        assert poa["ipo"] <= poa["lpt"] + 1e-12 and poa["ipo"] >= poa["lower_bound_kappa"] - 1e-12
