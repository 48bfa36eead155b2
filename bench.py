#!/usr/bin/env python
"""Benchmark: fwd+bwd effective TFLOP/s of FlashMask column-wise masked attention on GB300.

One step = the whole hot path over one batch of synthetic input: tile
classification + queues, mask localization (a 2-rank chunking, the utility
row), forward, backward (row terms, main kernel, dQ convert). The metric counts
only unmasked (i, j) pairs: 4*d FLOPs each for the forward and 10*d for the
backward, per query head.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
       python bench.py --balance
Prints ONE JSON line on rank 0. Under torchrun every rank runs its own replica
of the workload (weak scaling, no collective on the data path); the time is
the max over ranks and the value the sum of all ranks' work over that time.
--impl reference times the fp64 CPU oracle on the host cores instead.
--balance measures the chunk balancer for context parallelism (host code):
peak / average rank load on the workloads' own chunk loads and the ablation
table's instance families, and its time per call.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import configs, tensors  # noqa: E402

DEFAULT_WORKLOAD = "share_question32k"
METRIC = "effective TFLOP/s (unmasked FLOPs) fwd+bwd, % of GB300 BF16 peak; tile-skip %"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB of L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ metric
def visible_pairs(lts, lte, uts, ute, causal: bool) -> int:
    """Unmasked (i, j) pairs of one (N,) mask: N*N minus, per key column, the
    length of the union of its masked row intervals (inclusion-exclusion)."""
    n = lts.shape[0]
    j = np.arange(n, dtype=np.int64)
    a = [lts.astype(np.int64), uts.astype(np.int64), np.zeros(n, np.int64)]
    b = [lte.astype(np.int64), ute.astype(np.int64), j if causal else np.zeros(n, np.int64)]
    length = lambda lo, hi: np.maximum(0, hi - lo)
    tot = sum(length(a[k], b[k]) for k in range(3))
    for x in range(3):
        for y in range(x + 1, 3):
            tot = tot - length(np.maximum(a[x], a[y]), np.minimum(b[x], b[y]))
    tot = tot + length(np.maximum(np.maximum(a[0], a[1]), a[2]), np.minimum(np.minimum(b[0], b[1]), b[2]))
    return int(n * n - tot.sum())


def workload_flops(cfg) -> dict:
    pairs = sum(visible_pairs(cfg["lts"][b], cfg["lte"][b], cfg["uts"][b], cfg["ute"][b], cfg["causal"])
                for b in range(cfg["B"]))
    per_head = pairs
    d, hq = cfg["d"], cfg["H_q"]
    return dict(pairs=pairs, fwd=per_head * 4 * d * hq, bwd=per_head * 10 * d * hq)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background (timestamps kept)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", f"-lms={period_ms}",
                 f"--id={index}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        inside = [r for (t, r) in self.rows if t0 <= t <= t1 and len(r) >= 9]
        scope = "timed region"
        if not inside:
            inside = [r for (_, r) in self.rows if len(r) >= 9]
            scope = "whole run (no sample fell inside the timed region)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "scope": "nvidia-smi unavailable"}
        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in inside for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": num(inside[0][3]),
                "reasons": reasons, "samples": len(inside), "scope": scope,
                "power_w_max": max((num(r[4]) or 0.0) for r in inside)}


# ------------------------------------------------------------- distributed
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, use_cuda):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if use_cuda else "gloo")


def reduce_max(x: float, world: int, device) -> float:
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_flops: float, per_rank_seconds: float, world: int, device) -> tuple:
    """(total work over all ranks, max time over ranks) — the weak-scaling value is their ratio."""
    t = reduce_max(per_rank_seconds, world, device)
    return per_rank_flops * world, t


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


# ---------------------------------------------------------- oracle baseline
def closed_blocks(cfg):
    """Row ranges that only see, and are only seen by, themselves (documents /
    packed samples): each is an independent sub-problem of the workload."""
    if "samples" in cfg:
        out, s = [], 0
        for p, a, b in cfg["samples"]:
            out.append((s, s + p + a + b))
            s += p + a + b
        return out
    if "docs" in cfg and cfg["causal"]:
        out, s = [], 0
        for L in cfg["docs"]:
            out.append((s, s + L))
            s += L
        return out
    return None


def sub_vectors(cfg, block):
    """Boundary vectors of a closed block as its own problem (rows renumbered from 0)."""
    r0, r1 = block
    L = r1 - r0
    return tuple(np.clip(cfg[n][0][r0:r1].astype(np.int64) - r0, 0, L).astype(np.int32)[None]
                 for n in ("lts", "lte", "uts", "ute"))


def oracle_unit(cfg, q, k, v, do, h, block):
    """fwd + bwd of one query head on one closed block with the CPU oracle.

    A closed block is an independent sub-problem (its rows see only its keys
    and its keys are seen only by its rows), so the oracle runs on the block's
    own rows, keys and renumbered boundary vectors; the result equals the full
    problem's restricted to the block. Returns (effective FLOPs, seconds)."""
    import oracle  # test infrastructure: only the CPU-baseline leg uses it

    r0, r1 = block
    g = h // (cfg["H_q"] // cfg["H_kv"])
    vec = sub_vectors(cfg, block)
    f64 = lambda t: np.ascontiguousarray(t.double().numpy())
    qq, dd = f64(q[:1, h:h + 1, r0:r1]), f64(do[:1, h:h + 1, r0:r1])
    kk, vv = f64(k[:1, g:g + 1, r0:r1]), f64(v[:1, g:g + 1, r0:r1])
    t0 = time.perf_counter()
    oracle.forward(qq, kk, vv, vec, cfg["causal"], cfg["scale"])
    oracle.backward(qq, kk, vv, dd, vec, cfg["causal"], cfg["scale"])
    dt = time.perf_counter() - t0
    pairs = visible_pairs(*(x[0] for x in vec), cfg["causal"])
    return pairs * 14 * cfg["d"], dt


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_inputs(cfg):
    small = dict(cfg)
    return tensors.make_qkvdo(small)  # CPU draws (seeds 1..4)


def cpu_baseline(cfg, budget_s: float = 12.0):
    blocks = closed_blocks(cfg)
    if not blocks:
        return None
    q, k, v, do = cpu_inputs(cfg)
    flops = secs = 0.0
    units = 0
    order = sorted(range(len(blocks)), key=lambda i: blocks[i][1] - blocks[i][0])
    for h in range(cfg["H_q"]):
        for bi in order:
            f, t = oracle_unit(cfg, q, k, v, do, h, blocks[bi])
            flops += f
            secs += t
            units += 1
            if secs >= budget_s:
                break
        if secs >= budget_s:
            break
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
            "sample": f"{units} (query head, packed sample) fwd+bwd units of {cfg['name']}, "
                      f"{secs:.1f} s of fp64 numpy on the host (BLAS threads = cores)"}


def run_reference(args, cfg):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    blocks = closed_blocks(cfg)
    if not blocks:
        print(json.dumps({"impl": "reference", "unavailable": f"no closed sub-problem sample for {cfg['name']}"}))
        return 0
    q, k, v, do = cpu_inputs(cfg)
    units = [(h, bi) for h in range(cfg["H_q"]) for bi in range(len(blocks))]
    smallest = min(range(len(blocks)), key=lambda i: blocks[i][1] - blocks[i][0])
    for w in range(args.warmup):
        oracle_unit(cfg, q, k, v, do, w % cfg["H_q"], blocks[smallest])
    flops = secs = 0.0
    for s in range(args.steps):
        h, bi = units[s % len(units)]
        f, t = oracle_unit(cfg, q, k, v, do, h, blocks[bi])
        flops += f
        secs += t
    val = flops / secs / 1e12
    peaks, src = read_peaks()
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, "per step: one (query head, packed sample) fwd+bwd unit, cycling"),
        "pct_of_bf16_peak": 100.0 * val / peaks["bf16_tflops"],
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores_used(), "kind": "oracle",
                         "sample": f"{args.steps} units of one query head x one packed sample (fp64 numpy)"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_dict(cfg, note=""):
    d = {"workload": cfg["name"], "B": cfg["B"], "H_q": cfg["H_q"], "H_kv": cfg["H_kv"], "N": cfg["N"],
         "d": cfg["d"], "causal": bool(cfg["causal"]), "tile": [128, 128], "mask_seed": 0,
         "tensor_seeds": "Q,K,V,dO: torch CUDA generators 1..4, N(0,1) -> bf16",
         "l2": "flushed between timed steps (256 MiB write)"}
    if note:
        d["note"] = note
    return d


# -------------------------------------------------------------- our arm
class Path:
    """Preallocated buffers and the step = classify, localize, forward, backward."""

    def __init__(self, cfg, dev):
        import mask_aware_sparse_gb300 as fm

        self.fm = fm
        self.cfg = cfg
        self.dev = dev
        self.q, self.k, self.v, self.do = tensors.make_qkvdo(cfg, device=dev)
        self.vec = [torch.from_numpy(np.ascontiguousarray(cfg[n])).to(dev) for n in ("lts", "lte", "uts", "ute")]
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.v)
        n = cfg["N"]
        C = (n + 7) // 8  # 8 chunks, a 2-rank round-robin chunking; rank 0 owns chunks 0, 2, 4, 6
        self.loc_off = torch.tensor([0, 2 * C, 4 * C, 6 * C], dtype=torch.int32, device=dev)
        self.loc_C = C
        self.loc_in = torch.cat([x.reshape(-1) for x in self.vec])
        self.loc_out = torch.empty_like(self.loc_in)
        self.queues = None

    def step(self):
        fm, c = self.fm, self.cfg
        self.queues = fm.fm_classify_tiles(*self.vec, causal=c["causal"])
        fm.fm_localize(self.loc_in, self.loc_off, self.loc_C, out=self.loc_out)
        fm.fm_attn_fwd(self.q, self.k, self.v, *self.vec, self.queues, scale=c["scale"], causal=c["causal"],
                       o=self.o, lse=self.lse)
        fm.fm_attn_bwd(self.q, self.k, self.v, self.o, self.lse, self.do, *self.vec, self.queues, scale=c["scale"],
                       causal=c["causal"], dq=self.dq, dk=self.dk, dv=self.dv)


def capture_step(path: Path):
    """CUDA graph of one step (classify, localize, forward, backward) and the
    number of library kernels it launches; (None, 0) if capture fails."""
    fm = path.fm
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            path.step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        n0 = fm.fm_launch_count()
        with torch.cuda.graph(g):
            path.step()
        n = fm.fm_launch_count() - n0
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        st, _ = fm.fm_device_status()
        if st != fm.FM_OK:
            return None, 0
        return g, n
    except Exception:
        torch.cuda.synchronize()
        return None, 0


def e2e_measure(path: Path, steps: int):
    """Same metric through the C ABI's host-buffer entry point
    (fm_attn_fwd_bwd_host): every step hands the library pinned HOST buffers;
    the library copies the step's inputs to its device workspace, classifies,
    runs forward and backward and copies every output back. Steps rotate over
    three streams, each with its own device workspace and host output set, so
    one step's copies overlap its neighbours' compute."""
    fm, c = path.fm, path.cfg
    h_in = [t.cpu().pin_memory() for t in (path.q, path.k, path.v, path.do)]
    h_vec = [t.cpu().pin_memory() for t in path.vec]
    outs = (path.o, path.lse, path.dq, path.dk, path.dv)
    R = 3
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _ in range(R)]
    h2d = sum(t.numel() * t.element_size() for t in h_in + h_vec)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    prob = fm._problem(c["B"], c["H_q"], c["H_kv"], c["N"], c["d"], c["scale"], c["causal"], c["N"])
    wsb = fm.lib().fm_attn_host_workspace_bytes(fm.ctypes.byref(prob))
    ws = [torch.empty(wsb, dtype=torch.uint8, device=path.dev) for _ in range(R)]
    streams = [torch.cuda.Stream() for _ in range(R)]
    q, k, v, do = h_in

    def one(i):
        j = i % R
        o, lse, dq, dk, dv = h_out[j]
        fm.fm_attn_fwd_bwd_host(q, k, v, do, *h_vec, scale=c["scale"], causal=c["causal"], o=o, lse=lse, dq=dq,
                                dk=dk, dv=dv, ws=ws[j], stream=streams[j])

    for i in range(R):
        one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(streams[0])
    for st in streams[1:]:
        st.wait_event(a)
    for i in range(steps):
        one(i)
    for st in streams[1:]:
        streams[0].wait_stream(st)
    b.record(streams[0])
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / steps, h2d, d2h


def run_ours(args, cfg):
    world, rank, local = dist_info()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, True)
    from mask_aware_sparse_gb300 import build as fmbuild

    if rank == 0:
        fmbuild.build()
    barrier(world)
    path = Path(cfg, dev)
    fm = path.fm
    work = workload_flops(cfg)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(max(3, args.warmup)):
        path.step()
    torch.cuda.synchronize()
    st, bits = fm.fm_device_status()
    if st != fm.FM_OK:
        print(json.dumps({"error": f"device status {st} bits {bits} after warm-up"}))
        return 1
    # The timed step is replayed as one CUDA graph (captured from the same
    # calls), so host launch latency between the small kernels stays out of
    # the device timeline; eager issue is the fallback.
    graph, per_step_launches = capture_step(path)
    run_step = graph.replay if graph is not None else path.step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier(world)
    torch.cuda.synchronize()
    launches0 = fm.fm_launch_count()
    t_wall0 = time.time()
    for k in range(args.steps):
        flush.zero_()  # evict L2 between timed steps (outside the events)
        ev[k][0].record()
        run_step()
        ev[k][1].record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    launches = (fm.fm_launch_count() - launches0) if graph is None else per_step_launches * args.steps
    st, bits = fm.fm_device_status()
    if sampler:
        sampler.stop()
    # per-kernel split (live CUDA events around the two main kernels), eager steps
    fm.fm_profile_read()  # clear
    fm.fm_profile_enable(True)
    for _ in range(min(args.steps, 10)):
        flush.zero_()
        path.step()
    torch.cuda.synchronize()
    fm.fm_profile_enable(False)
    prof = fm.fm_profile_read()
    # the classification alone (its four kernels), timed by events on the stream it runs on
    cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(10)]
    for a, b in cev:
        flush.zero_()
        a.record()
        fm.fm_classify_tiles(*path.vec, causal=cfg["causal"])
        b.record()
    torch.cuda.synchronize()
    classify_ms = sum(a.elapsed_time(b) for a, b in cev) / len(cev)
    step_s = sum(a.elapsed_time(b) for a, b in ev) / 1e3
    flops_rank = (work["fwd"] + work["bwd"]) * args.steps
    tot_flops, tmax = aggregate(flops_rank, step_s, world, dev)
    value = tot_flops / tmax / 1e12

    e2e_s, h2d, d2h = e2e_measure(path, max(3, min(20, args.steps // 5)))
    e2e_s = reduce_max(e2e_s, world, dev)
    e2e_value = (work["fwd"] + work["bwd"]) * world / e2e_s / 1e12

    if rank != 0:
        return 0
    peaks, src = read_peaks()
    cls = path.queues.tile_class.cpu().numpy()
    counts = np.bincount(cls.ravel(), minlength=3)
    computed = int(counts[1] + counts[2])
    fwd_ms = prof["fwd_ms"] / max(1, prof["fwd_launches"])
    bwd_ms = prof["bwd_ms"] / max(1, prof["bwd_launches"])
    dom = "bwd" if bwd_ms >= fwd_ms else "fwd"
    dom_ms = bwd_ms if dom == "bwd" else fwd_ms
    dom_flops = work[dom]
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    traffic = ncu_traffic(dom, args.workload, cfg["d"])
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    # the same work against the tensor cores' per-clock peak at the SM clock
    # sampled during the timed region (4096 bf16 MACs per clock per SM,
    # measured by a microbenchmark); the measured cuBLAS peak above was taken
    # at a lower, power-capped clock
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (clocks or {}).get("sm_mhz") or peaks.get("sm_max_mhz")
    clk_peak = 2 * 4096 * sms * mhz * 1e6 / 1e12 if mhz else None
    per_clock = {"sm_mhz": mhz, "sms": sms, "peak": clk_peak,
                 "frac_bwd": (work["bwd"] / (bwd_ms / 1e3) / 1e12) / clk_peak if clk_peak else None,
                 "frac_fwd": (work["fwd"] / (fwd_ms / 1e3) / 1e12) / clk_peak if clk_peak else None}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": tmax / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(cfg),
        "pct_of_bf16_peak": 100.0 * value / world / peak,
        "peak_source": f"{src}: bf16_tflops {peak} (burst); sustained {peaks.get('bf16_tflops_sustained')}",
        "tile_skip_pct": 100.0 * counts[0] / cls.size,
        "tiles": {"skip": int(counts[0]), "partial": int(counts[1]), "unmasked": int(counts[2])},
        "computed_tile_tflops": computed * 128 * 128 * 14 * cfg["d"] * cfg["H_q"] * cfg["B"] * args.steps / step_s / 1e12,
        "kernel_ms": {"fwd_main": fwd_ms, "bwd_main": bwd_ms,
                      "rest_of_step": tmax / args.steps * 1e3 - fwd_ms - bwd_ms, "classify": classify_ms},
        "kernel_frac_of_measured_peak": {"fwd_main": work["fwd"] / (fwd_ms / 1e3) / 1e12 / peak,
                                         "bwd_main": work["bwd"] / (bwd_ms / 1e3) / 1e12 / peak},
        "per_clock_peak": per_clock,
        # tensor pipe active, % of elapsed cycles, from the ncu capture of the
        # same kernel source on this workload (None once the source changed)
        "ncu_tensor_pipe_pct": {"fwd_main": ncu_traffic("fwd", args.workload, cfg["d"], "tensor_pipe_pct"),
                                "bwd_main": ncu_traffic("bwd", args.workload, cfg["d"], "tensor_pipe_pct")},
        "roofline": {"kernel": "fm_attn_bwd main" if dom == "bwd" else "fm_attn_fwd main", "bound": "tensor",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": traffic,
                     "algorithmic": f"{'10' if dom == 'bwd' else '4'}*d FLOPs x {work['pairs']} unmasked pairs x "
                                    f"{cfg['H_q']} heads per launch"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "device_status": int(st),
    }
    line["config"]["step_issue"] = "one CUDA graph per step" if graph is not None else "eager"
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line))
    return 0


# ncu DRAM traffic (read + write bytes per launch) of the main kernels on the
# workload it was captured on, valid only while the kernel source is the one
# the counters were taken from.
NCU_TRAFFIC = {
    ("bwd", 128): {"file": "fm_bwd.cu", "workload": "share_question32k",
                   "sha256": "b9838b53ff643061f94fb721f02c52b2658fee04ace7e22f4ddc1ebd63899894",
                   "bytes": 826607360 + 450107392, "tensor_pipe_pct": 58.8},
    ("fwd", 128): {"file": "fm_fwd.cu", "workload": "share_question32k",
                   "sha256": "bd5dfdf503256e367b6c6cc8b760315ba7e2299dfdde74e014a5dd77b4ded650",
                   "bytes": 265070080 + 217337088, "tensor_pipe_pct": 49.4},
    ("bwd", 256): {"file": "fm_bwd256.cu", "workload": "share_question32k",
                   "sha256": "4a74f10607bb3fe9ddb3bce855a37e863781ea99a6210d9179ccd704351b296f",
                   "bytes": 2578204928 + 1447225856, "tensor_pipe_pct": 42.3},
    ("fwd", 256): {"file": "fm_fwd256.cu", "workload": "share_question32k",
                   "sha256": "43a49b7ecbde286dd8dc56ffcc166e1b7199fb9e19b95c5e838eeaa05480071a",
                   "bytes": 527136512 + 485024256, "tensor_pipe_pct": 48.5},
}


def ncu_traffic(kind: str, workload: str, d: int, key: str = "bytes"):
    """A counter of the ncu capture of main kernel `kind` on this workload
    (DRAM bytes per launch, or the tensor pipe's active % of elapsed cycles),
    or None when the kernel source has changed since the capture."""
    import hashlib

    ent = NCU_TRAFFIC.get((kind, d))
    if not ent or ent["workload"] != workload:
        return None
    src = os.path.join(ROOT, "mask_aware_sparse_gb300", "csrc", ent["file"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return ent.get(key) if h == ent["sha256"] else None


# ------------------------------------------------------ FP8 forward
def _time_steps(fn, steps, flush):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / 1e3 / steps


def run_fp8(args, cfg):
    """The FP8 forward on the workload: one step = classify + fm_attn_fwd_fp8 on
    e4m3 Q / K / V (per-tensor scales), beside the bf16 forward on the same
    (dequantized) inputs. Metric: effective forward TFLOP/s (4 d FLOPs per
    unmasked pair), against the fp8 peak taken as the measured bf16 peak x 2
    (the nominal dense fp8 : bf16 ratio, 4.5 : 2.25 PFLOP/s)."""
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    from mask_aware_sparse_gb300 import build as fmbuild

    fmbuild.build()
    import mask_aware_sparse_gb300 as fm

    dev = torch.device("cuda", 0)
    q, k, v, _ = tensors.make_qkvdo(cfg, device=dev)

    def quant(x):
        sc = float(x.float().abs().max()) / 448.0
        return (x.float() / sc).to(torch.float8_e4m3fn), sc

    (q8, sq), (k8, sk), (v8, sv) = quant(q), quant(k), quant(v)
    qd, kd, vd = ((x.float() * s_).to(torch.bfloat16) for x, s_ in ((q8, sq), (k8, sk), (v8, sv)))
    vec = [torch.from_numpy(np.ascontiguousarray(cfg[n])).to(dev) for n in ("lts", "lte", "uts", "ute")]
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    c = cfg

    def step8():
        qs = fm.fm_classify_tiles(*vec, causal=c["causal"])
        fm.fm_attn_fwd_fp8(q8, k8, v8, *vec, qs, q_scale=sq, k_scale=sk, v_scale=sv, scale=c["scale"],
                           causal=c["causal"], o=o, lse=lse)

    def step16():
        qs = fm.fm_classify_tiles(*vec, causal=c["causal"])
        fm.fm_attn_fwd(qd, kd, vd, *vec, qs, scale=c["scale"], causal=c["causal"], o=o, lse=lse)

    for _ in range(max(3, args.warmup)):
        step8()
        step16()
    torch.cuda.synchronize()
    st, bits = fm.fm_device_status()
    if st != fm.FM_OK:
        print(json.dumps({"error": f"device status {st} bits {bits} after warm-up"}))
        return 1
    sampler = ClockSampler(0)
    time.sleep(0.3)
    t0 = time.time()
    t8 = _time_steps(step8, args.steps, flush)
    t1 = time.time()
    sampler.stop()
    t16 = _time_steps(step16, args.steps, flush)
    fm.fm_profile_read()
    fm.fm_profile_enable(True)
    for _ in range(min(args.steps, 10)):
        flush.zero_()
        step8()
    torch.cuda.synchronize()
    fm.fm_profile_enable(False)
    prof = fm.fm_profile_read()
    k8_ms = prof["fwd_ms"] / max(1, prof["fwd_launches"])
    work = workload_flops(cfg)
    peaks, src = read_peaks()
    peak8 = 2 * peaks["bf16_tflops"]
    value = work["fwd"] / t8 / 1e12
    achieved = work["fwd"] / (k8_ms / 1e3) / 1e12
    cfgd = config_dict(cfg, note="Q, K, V e4m3 with per-tensor scales (amax / 448); step = classify + forward")
    line = {"metric": "effective TFLOP/s (unmasked FLOPs) fwd, FP8 (e4m3) inputs", "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": t8 * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": cfgd, "bf16_forward_same_inputs": {"value": work["fwd"] / t16 / 1e12, "ms_per_step": t16 * 1e3},
            "roofline": {"kernel": "fm_attn_fwd_fp8 main", "bound": "tensor", "achieved": achieved, "peak": peak8,
                         "unit": "TFLOP/s", "frac": achieved / peak8, "traffic": None,
                         "peak_source": f"{src} bf16_tflops {peaks['bf16_tflops']} x 2 (nominal fp8 : bf16)",
                         "algorithmic": f"4*d FLOPs x {work['pairs']} unmasked pairs x {cfg['H_q']} heads per launch"},
            "kernel_ms": {"fwd_main": k8_ms}, "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line))
    return 0


# --------------------------------------------- mask-form compositions
def run_compose(args, cfg):
    """Forward + backward through one of the binding's compositions, on the
    workload's own mask written in that form (so the work and the metric are
    the workload's): `per_head` gives every query head its own copy of the
    vectors (fm_attn_per_head: one classification over the B * H_q vector
    rows, one forward and one backward launch over every head);
    `per_head_distinct` (share-question only) lets every query head pack its
    own eight samples (lengths drawn per head from seed 1000 + h), so the
    heads' masks and queues differ, and counts each head's own unmasked pairs;
    `multi_interval` writes each key column's visible
    rows [j, LTS_j) as two inclusive intervals split at their midpoint
    (fm_attn_multi_interval: one classification of the intervals' union,
    one forward and one backward launch). The latter needs a causal mask with LTE = N and no upper
    interval."""
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    from mask_aware_sparse_gb300 import build as fmbuild

    fmbuild.build()
    import mask_aware_sparse_gb300 as fm

    dev = torch.device("cuda", 0)
    q, k, v, do = tensors.make_qkvdo(cfg, device=dev)
    names = ("lts", "lte", "uts", "ute")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    c = cfg
    work = workload_flops(cfg)
    if args.compose == "per_head":
        vec = [torch.from_numpy(np.ascontiguousarray(np.repeat(cfg[n][:, None], cfg["H_q"], axis=1))).to(dev)
               for n in names]

        def step():
            fm.fm_attn_per_head(q, k, v, *vec, causal=c["causal"], scale=c["scale"], do=do)
    elif args.compose == "per_head_distinct":
        if "samples" not in cfg or cfg["B"] != 1:
            print(json.dumps({"error": "per_head_distinct needs the share-question workload (B = 1)"}))
            return 1
        from workloads import masks as wmasks

        per = [tuple(np.asarray(x, np.int32) for x in
                     wmasks.share_question(wmasks.draw_share_question(np.random.default_rng(1000 + h)), cfg["N"]))
               for h in range(cfg["H_q"])]
        vec = [torch.from_numpy(np.ascontiguousarray(np.stack([p[i] for p in per])[None])).to(dev) for i in range(4)]
        pairs = sum(visible_pairs(*p, cfg["causal"]) for p in per)   # summed over the heads
        d = cfg["d"]
        work = dict(pairs=pairs, fwd=pairs * 4 * d, bwd=pairs * 10 * d)

        def step():
            fm.fm_attn_per_head(q, k, v, *vec, causal=c["causal"], scale=c["scale"], do=do)
    else:
        lts, lte, uts, ute = (cfg[n].astype(np.int64) for n in names)
        n = cfg["N"]
        if not (cfg["causal"] and (lte == n).all() and (uts >= ute).all()):
            print(json.dumps({"error": "multi_interval needs a causal mask with LTE = N and no upper interval"}))
            return 1
        j = np.broadcast_to(np.arange(n), lts.shape)
        last = lts - 1                       # visible rows of column j: [j, LTS_j - 1]
        mid = (j + last) // 2
        fms = np.stack([j, mid + 1]).astype(np.int32)
        fme = np.stack([mid, last]).astype(np.int32)   # empty where start > end
        fms_t, fme_t = torch.from_numpy(fms).to(dev), torch.from_numpy(fme).to(dev)

        def step():
            fm.fm_attn_multi_interval(q, k, v, fms_t, fme_t, scale=c["scale"], do=do)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st, bits = fm.fm_device_status()
    if st != fm.FM_OK:
        print(json.dumps({"error": f"device status {st} bits {bits} after warm-up"}))
        return 1
    sampler = ClockSampler(0)
    time.sleep(0.3)
    t0 = time.time()
    t = _time_steps(step, args.steps, flush)
    t1 = time.time()
    sampler.stop()
    value = (work["fwd"] + work["bwd"]) / t / 1e12
    peaks, src = read_peaks()
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(cfg, note=f"composition: {args.compose} (eager library calls per step)"),
            "pct_of_bf16_peak": 100.0 * value / peaks["bf16_tflops"], "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------- chunk balancer
BAL_COSTS = (13, 10)  # partial, unmasked tile: the pages' illustrative 1.3 : 1
BAL_WORKLOADS = ("doc8k", "share_question32k", "prefix_lm64k", "sliding_window64k", "eviction128k")


def _rank_peak(w, owner, P):
    return float(np.bincount(owner, weights=w, minlength=P).max())


def _zigzag_owner(P, kappa):
    """Chunk owners of the zigzag split (kappa = 2: the dual-chunk split):
    pass p hands chunks p*P .. p*P + P - 1 to ranks 0..P-1, every other pass reversed."""
    owner = np.empty(P * kappa, dtype=np.int64)
    for p in range(kappa):
        for r in range(P):
            owner[p * P + (r if p % 2 == 0 else P - 1 - r)] = r
    return owner


def _time_call(fn, reps=5):
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        out = fn()
        ts.append(time.perf_counter() - t0)
    return out, 1e3 * float(np.median(ts))


def run_balance(args):
    import mask_aware_sparse_gb300 as fm
    from mask_aware_sparse_gb300 import build as fmbuild
    from workloads import chunks

    fmbuild.build()

    cp, cu = BAL_COSTS
    cases = []
    if torch.cuda.is_available():
        for name in BAL_WORKLOADS:
            cfg = configs.make(name)
            vec = [torch.from_numpy(np.ascontiguousarray(cfg[k])).cuda() for k in ("lts", "lte", "uts", "ute")]
            qs = fm.fm_classify_tiles(*vec, causal=cfg["causal"])
            cls = qs.tile_class.cpu().numpy()
            nq = cls.shape[1]
            for P in (4, 8, 16):
                kappa = 4
                bpc = nq // (P * kappa)
                if bpc < 1 or nq % (P * kappa):
                    continue
                w = fm.fm_chunk_loads(cls, bpc, cp, cu)
                (owner, rep), ms = _time_call(lambda: fm.fm_balance_chunks(w, P, kappa))
                avg = float(w.sum()) / P
                contiguous = np.repeat(np.arange(P), kappa)
                # mask-aware pruning of the K / V exchange: remote chunks a rank's rows never see
                need = fm.fm_needed_chunks(cls, owner, P, bpc)
                remote = np.ones(need.shape, dtype=bool)
                remote[owner, np.arange(owner.size)] = False
                pruned = 1.0 - float(need[remote].sum()) / float(remote.sum())
                cases.append(dict(workload=name, P=P, kappa=kappa, q_blocks_per_chunk=bpc,
                                  peak_over_avg=dict(contiguous=_rank_peak(w, contiguous, P) / avg,
                                                     zigzag=_rank_peak(w, _zigzag_owner(P, kappa), P) / avg,
                                                     lpt=rep["makespan_lpt"] / avg, ipo=rep["makespan"] / avg,
                                                     lower_bound=rep["lower_bound"] / avg,
                                                     lower_bound_kappa=rep["lower_bound_kappa"] / avg),
                                  certified=rep["certified"], ms_per_call=ms,
                                  pruned_remote_chunk_fraction=pruned))
    table = {}
    for name, (kind, n, P, kappa, w_max, inst) in chunks.TABLE.items():
        rng = np.random.default_rng(0)
        cert = lsub = psub = 0
        lgap, pgap, fgap, ms = [], [], [], []
        for _ in range(inst):
            w = chunks.random_loads(rng, kind, n, w_max)
            t0 = time.perf_counter()
            owner, rep = fm.fm_balance_chunks(w, P, kappa)
            ms.append(1e3 * (time.perf_counter() - t0))
            lb = rep["lower_bound_kappa"]
            fgap.append((rep["makespan"] - lb) / lb)
            if rep["certified"]:
                cert += 1
                lsub += rep["makespan_lpt"] > lb
                psub += rep["makespan_pair"] > lb
                lgap.append((rep["makespan_lpt"] - lb) / lb)
                pgap.append((rep["makespan_pair"] - lb) / lb)
        pct = lambda a: round(100.0 * a / max(cert, 1), 1)  # noqa: E731
        table[name] = dict(n=n, P=P, kappa=kappa, w_max=w_max, instances=inst, lb_certified=cert,
                           lpt_subopt_pct_of_certified=pct(lsub), lpt_gap_pct=round(100 * float(np.mean(lgap or [0])), 3),
                           pair_subopt_pct_of_certified=pct(psub),
                           pair_gap_pct=round(100 * float(np.mean(pgap or [0])), 3),
                           final_gap_to_lb_pct=round(100 * float(np.mean(fgap)), 4),
                           ms_per_call_median=round(float(np.median(ms)), 3), ms_per_call_max=round(max(ms), 3))
    ipo = [c["peak_over_avg"]["ipo"] for c in cases]
    line = {"metric": "chunk balancer: peak / average rank load (CP split of the query axis)",
            "value": float(np.exp(np.mean(np.log(ipo)))) if ipo else None, "unit": "ratio",
            "higher_is_better": False, "dtype": "int64", "data": "synthetic",
            "config": {"workload": "workloads' chunk loads (tile costs partial 13, unmasked 10) + ablation table "
                                   "families", "kappa": 4, "P": [4, 8, 16]},
            "cases": cases, "table": table}
    if not args.no_cpu_baseline:
        from oracle import balance as ob  # the CPU baseline leg: the oracle, as it stands
        kind, n, P, kappa, w_max, _ = chunks.TABLE["causal"]
        rng = np.random.default_rng(0)
        ws = [chunks.random_loads(rng, kind, n, w_max) for _ in range(3)]
        t0 = time.perf_counter()
        for w in ws:
            ob.ipo(w, P, kappa, phases=2)
        dt = (time.perf_counter() - t0) / len(ws)
        line["cpu_baseline"] = {"value": 1e3 * dt, "unit": "ms per call", "cores": 1, "kind": "oracle",
                                "sample": "3 causal-family instances (64 chunks, 8 ranks, kappa 8), LPT + pairwise"}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=configs.NAMES)
    ap.add_argument("--head-dim", type=int, default=None, choices=(64, 128, 256),
                    help="run the workload's mask and shapes at another head dimension")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--balance", action="store_true", help="measure the chunk balancer instead")
    ap.add_argument("--fp8", action="store_true", help="measure the FP8 forward instead")
    ap.add_argument("--compose", choices=("per_head", "per_head_distinct", "multi_interval"), default=None,
                    help="measure a mask-form composition of the binding instead")
    args = ap.parse_args()
    if args.balance:
        return run_balance(args)
    if args.warmup < 3:
        args.warmup = 3
    cfg = configs.make(args.workload) if args.head_dim is None else configs.make(args.workload, d=args.head_dim)
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.fp8:
        return run_fp8(args, cfg)
    if args.compose:
        return run_compose(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
