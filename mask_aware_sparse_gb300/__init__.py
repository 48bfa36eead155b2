"""Python binding of libfm (include/fm.h): FlashMask column-wise masked attention on GB300.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels of libfm.so; torch supplies device memory and the current stream.
Importing works without a GPU; the first call loads libfm.so and raises if it
is missing (build it with `mask_aware_sparse_gb300.build.build()`), so there
is no silent fallback.

Functions carry the names of the C entry points:
  fm_classify_tiles, fm_attn_fwd, fm_attn_fwd_fp8, fm_attn_bwd, fm_attn_fwd_heads and
  fm_attn_bwd_heads (per-head mask vectors), fm_attn_fwd_multi and fm_attn_bwd_multi
  (multi-interval masks), fm_attn_fwd_bwd_host (host buffers in
  and out, device workspace), fm_localize, fm_device_status,
  fm_selftest_wait_timeout, fm_profile_enable, fm_profile_read, fm_launch_count,
  fm_from_fms_fme, fm_merge_parts, fm_sum_parts, fm_chunk_loads,
  fm_balance_chunks, fm_needed_chunks (host code: the chunk balancer and the
  K / V exchange plan for context parallelism);
plus fm_classify_tiles_heads (fm_classify_tiles over the B * H_q rows of
per-head vectors), fm_attn_multi_interval and fm_attn_per_head (the library
calls of a multi-interval / per-head forward and backward in sequence) and
flashmask_attention (autograd wrapper: the classification, forward and
backward calls in one differentiable op).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# FM_LIBRARY=debug selects the range-checked debug build (build.build(debug=True))
LIB_PATH = os.path.join(_HERE, "libfm_debug.so" if os.environ.get("FM_LIBRARY") == "debug" else "libfm.so")

FM_OK, FM_ERR_INVALID_ARG, FM_ERR_UNSUPPORTED, FM_ERR_WORKSPACE, FM_ERR_CUDA, FM_ERR_TIMEOUT, FM_ERR_DEVICE = range(7)
FM_DEVERR_TIMEOUT, FM_DEVERR_RANGE, FM_DEVERR_QUEUE, FM_DEVERR_DEBUG = 1, 2, 4, 8


class fm_problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("N", ctypes.c_int32),
                ("d", ctypes.c_int32), ("scale", ctypes.c_float), ("causal", ctypes.c_int32), ("N_kv", ctypes.c_int32)]


class fm_tiling(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int32), ("block_n", ctypes.c_int32)]


class fm_balance_report(ctypes.Structure):
    _fields_ = [("lower_bound", ctypes.c_int64), ("lower_bound_kappa", ctypes.c_int64),
                ("makespan_lpt", ctypes.c_int64), ("makespan_pair", ctypes.c_int64),
                ("makespan", ctypes.c_int64), ("certified", ctypes.c_int32), ("pair_moves", ctypes.c_int32),
                ("triple_moves", ctypes.c_int32), ("budget_exhausted", ctypes.c_int32)]


class FMError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_SIGS = {
    "fm_abi_version": (ctypes.c_int32, []),
    "fm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fm_attn_tiling": (ctypes.c_int, [ctypes.POINTER(fm_tiling)]),
    "fm_tile_counts": (ctypes.c_int, [ctypes.POINTER(fm_problem), ctypes.POINTER(fm_tiling),
                                      ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "fm_classify_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem), ctypes.POINTER(fm_tiling)]),
    "fm_classify_tiles": (ctypes.c_int, [ctypes.POINTER(fm_problem), ctypes.POINTER(fm_tiling)] + [_P] * 9
                          + [_P, ctypes.c_size_t, _P]),
    "fm_attn_fwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem)]),
    "fm_attn_fwd": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 11 + [_P, ctypes.c_size_t, _P]),
    "fm_attn_fwd_noalloc": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 11 + [_P]),
    "fm_attn_fwd_fp8": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 3 + [ctypes.c_float] * 3 + [_P] * 8
                        + [_P, ctypes.c_size_t, _P]),
    "fm_attn_bwd_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem)]),
    "fm_attn_fwd_heads_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem)]),
    "fm_attn_fwd_heads": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 11 + [_P, ctypes.c_size_t, _P]),
    "fm_attn_bwd_heads": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 15 + [_P, ctypes.c_size_t, _P]),
    "fm_classify_multi_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem), ctypes.POINTER(fm_tiling),
                                                            ctypes.c_int32]),
    "fm_classify_tiles_multi": (ctypes.c_int, [ctypes.POINTER(fm_problem), ctypes.POINTER(fm_tiling),
                                               ctypes.c_int32] + [_P] * 7 + [_P, ctypes.c_size_t, _P]),
    "fm_attn_fwd_multi": (ctypes.c_int, [ctypes.POINTER(fm_problem), ctypes.c_int32] + [_P] * 9 +
                          [_P, ctypes.c_size_t, _P]),
    "fm_attn_bwd_multi": (ctypes.c_int, [ctypes.POINTER(fm_problem), ctypes.c_int32] + [_P] * 13 +
                          [_P, ctypes.c_size_t, _P]),
    "fm_attn_host_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(fm_problem)]),
    "fm_attn_fwd_bwd_host": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 13 + [_P, ctypes.c_size_t, _P]),
    "fm_attn_bwd": (ctypes.c_int, [ctypes.POINTER(fm_problem)] + [_P] * 15 + [_P, ctypes.c_size_t, _P]),
    "fm_localize": (ctypes.c_int, [_P, ctypes.c_int64, _P, ctypes.c_int32, ctypes.c_int32, _P, _P]),
    "fm_from_fms_fme": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P]),
    "fm_merge_parts": (ctypes.c_int, [ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
    "fm_sum_parts": (ctypes.c_int, [ctypes.c_int32, _P, ctypes.c_int64, _P, _P]),
    "fm_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "fm_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, _P]),
    "fm_profile_enable": (ctypes.c_int, [ctypes.c_int32]),
    "fm_profile_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32)]),
    "fm_launch_count": (ctypes.c_int64, []),
    "fm_chunk_loads": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int64, ctypes.c_int64, _P]),
    "fm_balance_chunks": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int64, _P, ctypes.POINTER(fm_balance_report)]),
    "fm_needed_chunks": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, _P]),
}
EXPORTS = tuple(_SIGS)


def lib():
    """The loaded libfm.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with mask_aware_sparse_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(s: int) -> str:
    try:
        return lib().fm_status_string(int(s)).decode()
    except Exception:  # library not loadable: still give a message
        return "status"


def _check(st: int, what: str):
    if st != FM_OK:
        raise FMError(st, what)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _problem(B, H_q, H_kv, N, d, scale, causal, N_kv=0) -> fm_problem:
    return fm_problem(int(B), int(H_q), int(H_kv), int(N), int(d), float(scale), 1 if causal else 0, int(N_kv))


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _like(t, name, shape, dtype):
    """t is a contiguous torch tensor of this shape and dtype (device checked separately)."""
    _need(isinstance(t, torch.Tensor), f"{name} must be a torch tensor")
    _need(tuple(t.shape) == tuple(shape), f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def _same_cuda(**ts):
    """Every given tensor lives on one CUDA device (the library computes on the GPU only)."""
    dev = None
    for name, t in ts.items():
        if t is None:
            continue
        _need(t.is_cuda, f"{name} must be a CUDA tensor: the library computes on the GPU only")
        dev = t.device if dev is None else dev
        _need(t.device == dev, f"{name} is on {t.device}, the other tensors on {dev}")


def _vec_ok(*vs, shape=None):
    """Mask vectors: contiguous int32 CUDA tensors of one (B, N_kv) shape."""
    shape = tuple(vs[0].shape) if shape is None else tuple(shape)
    _need(len(shape) == 2, "mask vectors must be (B, N_kv)")
    for i, v in enumerate(vs):
        _like(v, f"mask vector {i}", shape, torch.int32)
    _same_cuda(**{f"mask vector {i}": v for i, v in enumerate(vs)})


def _bf16_ok(*ts):
    for t in ts:
        _need(isinstance(t, torch.Tensor) and t.dim() == 4,
              "Q/K/V/O/dO must be contiguous bf16 CUDA tensors of shape (B, H, N, d)")
        _like(t, "Q/K/V/O/dO", t.shape, torch.bfloat16)
    _same_cuda(**{f"tensor {i}": t for i, t in enumerate(ts)})


def _attn_args(q, k, v, vec, queues, *, backward, o=None, lse=None, do=None, dq=None, dk=None, dv=None, ws=None,
               heads=False, intervals=0):
    """Shapes, dtypes and devices of an attention call, checked before the library
    sees any pointer (the C ABI receives bare pointers and cannot check them).
    Shape checks come first, so a mismatch is reported as such. heads: per-head
    mask vectors (B, H_q, N_kv) and queues over B * H_q rows; intervals = M > 0:
    multi-interval FMS / FME (M, B, N_kv) (vec holds the two) and the union
    classification's queues over B rows."""
    _need(isinstance(q, torch.Tensor) and q.dim() == 4, "q must be a (B, H_q, N, d) tensor")
    B, Hq, N, d = q.shape
    _need(isinstance(k, torch.Tensor) and k.dim() == 4 and k.shape[0] == B and k.shape[3] == d,
          f"k has shape {tuple(k.shape)}, expected (B={B}, H_kv, N_kv, d={d})")
    Hkv, Nk = k.shape[1], k.shape[2]
    _need(Hkv > 0 and Hq % Hkv == 0, f"H_q={Hq} must be a multiple of H_kv={Hkv}")
    _like(q, "q", (B, Hq, N, d), torch.bfloat16)
    _like(k, "k", (B, Hkv, Nk, d), torch.bfloat16)
    _like(v, "v", (B, Hkv, Nk, d), torch.bfloat16)
    vshape = (B, Hq, Nk) if heads else (intervals, B, Nk) if intervals else (B, Nk)
    for i, x in enumerate(vec):
        _like(x, f"mask vector {i}", vshape, torch.int32)
    for name, t in (("o", o), ("do", do), ("dq", dq)):
        if t is not None:
            _like(t, name, (B, Hq, N, d), torch.bfloat16)
    if lse is not None:
        _like(lse, "lse", (B, Hq, N), torch.float32)
    for name, t in (("dk", dk), ("dv", dv)):
        if t is not None:
            _like(t, name, (B, Hkv, Nk, d), torch.bfloat16)
    if ws is not None:
        _need(isinstance(ws, torch.Tensor) and ws.is_contiguous(), "ws must be a contiguous tensor")
    _need(isinstance(queues, TileQueues), "queues must come from fm_classify_tiles")
    bm, bn = attn_tiling()
    _need((queues.block_m, queues.block_n) == (bm, bn),
          f"queues were built with {queues.block_m} x {queues.block_n} tiles; the kernels need {bm} x {bn}")
    nq, nk = -(-N // bm), -(-Nk // bn)
    R = B * Hq if heads else B  # queue rows per Q (K) block
    off, qu, nrows = (queues.k_off, queues.k_queue, R * nk) if backward else (queues.q_off, queues.q_queue, R * nq)
    _like(off, "queue offsets", (nrows + 1,), torch.int32)
    _need(isinstance(qu, torch.Tensor) and qu.dtype == torch.int32 and qu.is_contiguous()
          and qu.numel() >= max(1, R * nq * nk),
          f"queue entries must be int32 with capacity {R} * nQ * nK")
    _same_cuda(q=q, k=k, v=v, o=o, lse=lse, do=do, dq=dq, dk=dk, dv=dv, ws=ws, queue_offsets=off, queue=qu,
               **{f"mask vector {i}": x for i, x in enumerate(vec)})


def attn_tiling():
    t = fm_tiling()
    _check(lib().fm_attn_tiling(ctypes.byref(t)), "fm_attn_tiling")
    return t.block_m, t.block_n


@dataclass
class TileQueues:
    """Outputs of fm_classify_tiles (device tensors) and the tiling they were built with."""
    tile_class: torch.Tensor  # (B, nQ, nK) uint8: 0 skip, 1 partial, 2 unmasked
    q_off: torch.Tensor       # (B*nQ + 1,) int32
    q_queue: torch.Tensor     # (capacity,) int32, (kb << 1) | partial, kb descending per row
    k_off: torch.Tensor       # (B*nK + 1,) int32
    k_queue: torch.Tensor     # (capacity,) int32, (qb << 1) | partial, qb ascending per column
    block_m: int
    block_n: int


def fm_classify_tiles(lts, lte, uts, ute, *, causal: bool, block_m: int = 128, block_n: int = 128, n_rows=None,
                      stream=None):
    """Classify every (Q-block, KV-block) tile and build both compacted queues.

    The vectors are (B, N_kv); n_rows is the number of query rows N (default
    N_kv: the square problem)."""
    _vec_ok(lts, lte, uts, ute)
    B, Nk = lts.shape
    N = Nk if n_rows is None else int(n_rows)
    prob = _problem(B, 1, 1, N, 128, 1.0, causal, Nk)
    til = fm_tiling(block_m, block_n)
    nq, nk = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().fm_tile_counts(ctypes.byref(prob), ctypes.byref(til), ctypes.byref(nq), ctypes.byref(nk)),
           "fm_tile_counts")
    nq, nk = nq.value, nk.value
    dev = lts.device
    cap = max(1, B * nq * nk)
    cls = torch.empty((B, nq, nk), dtype=torch.uint8, device=dev)
    q_off = torch.empty(B * nq + 1, dtype=torch.int32, device=dev)
    k_off = torch.empty(B * nk + 1, dtype=torch.int32, device=dev)
    q_queue = torch.empty(cap, dtype=torch.int32, device=dev)
    k_queue = torch.empty(cap, dtype=torch.int32, device=dev)
    wsb = lib().fm_classify_workspace_bytes(ctypes.byref(prob), ctypes.byref(til))
    ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=dev)
    _check(lib().fm_classify_tiles(ctypes.byref(prob), ctypes.byref(til), _ptr(lts), _ptr(lte), _ptr(uts), _ptr(ute),
                                   _ptr(cls), _ptr(q_off), _ptr(q_queue), _ptr(k_off), _ptr(k_queue), _ptr(ws),
                                   ctypes.c_size_t(wsb), _stream(stream)), "fm_classify_tiles")
    return TileQueues(cls, q_off, q_queue, k_off, k_queue, block_m, block_n)


def fm_attn_fwd(q, k, v, lts, lte, uts, ute, queues: TileQueues, *, scale: float, causal: bool, o=None, lse=None,
                ws=None, stream=None):
    """Forward: returns (O bf16 (B,H_q,N,d), LSE fp32 (B,H_q,N)); K, V may hold N_kv != N rows."""
    _attn_args(q, k, v, (lts, lte, uts, ute), queues, backward=False, o=o, lse=lse, ws=ws)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wsb = lib().fm_attn_fwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(lts), _ptr(lte), _ptr(uts),
                             _ptr(ute), _ptr(queues.q_off), _ptr(queues.q_queue), _ptr(o), _ptr(lse), _ptr(ws),
                             ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_fwd")
    return o, lse


def fm_attn_fwd_fp8(q, k, v, lts, lte, uts, ute, queues: TileQueues, *, q_scale: float, k_scale: float,
                    v_scale: float, scale: float, causal: bool, o=None, lse=None, ws=None, stream=None):
    """FP8 forward: q, k, v are float8_e4m3fn (B, H, N, 128) tensors standing for
    stored x q_scale (k_scale, v_scale). Returns (O bf16, LSE fp32)."""
    e4 = torch.float8_e4m3fn
    _need(isinstance(q, torch.Tensor) and q.dim() == 4, "q must be a (B, H_q, N, d) tensor")
    B, Hq, N, d = q.shape
    _need(isinstance(k, torch.Tensor) and k.dim() == 4 and k.shape[0] == B and k.shape[3] == d,
          f"k has shape {tuple(k.shape)}, expected (B={B}, H_kv, N_kv, d={d})")
    Hkv, Nk = k.shape[1], k.shape[2]
    _need(Hkv > 0 and Hq % Hkv == 0, f"H_q={Hq} must be a multiple of H_kv={Hkv}")
    _like(q, "q", (B, Hq, N, d), e4)
    _like(k, "k", (B, Hkv, Nk, d), e4)
    _like(v, "v", (B, Hkv, Nk, d), e4)
    for i, x in enumerate((lts, lte, uts, ute)):
        _like(x, f"mask vector {i}", (B, Nk), torch.int32)
    if o is not None:
        _like(o, "o", (B, Hq, N, d), torch.bfloat16)
    if lse is not None:
        _like(lse, "lse", (B, Hq, N), torch.float32)
    _need(isinstance(queues, TileQueues) and (queues.block_m, queues.block_n) == attn_tiling(),
          "queues must come from fm_classify_tiles with the attention tiling")
    nq = -(-N // queues.block_m)
    _like(queues.q_off, "queue offsets", (B * nq + 1,), torch.int32)
    _same_cuda(q=q, k=k, v=v, o=o, lse=lse, ws=ws, queue_offsets=queues.q_off, queue=queues.q_queue,
               **{f"mask vector {i}": x for i, x in enumerate((lts, lte, uts, ute))})
    prob = _problem(B, Hq, Hkv, N, d, scale, causal, Nk)
    o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=q.device) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wsb = lib().fm_attn_fwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_fwd_fp8(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), float(q_scale), float(k_scale),
                                 float(v_scale), _ptr(lts), _ptr(lte), _ptr(uts), _ptr(ute), _ptr(queues.q_off),
                                 _ptr(queues.q_queue), _ptr(o), _ptr(lse), _ptr(ws), ctypes.c_size_t(wsb),
                                 _stream(stream)), "fm_attn_fwd_fp8")
    return o, lse


def fm_attn_bwd(q, k, v, o, lse, do, lts, lte, uts, ute, queues: TileQueues, *, scale: float, causal: bool,
                dq=None, dk=None, dv=None, ws=None, stream=None):
    """Backward: returns (dQ, dK, dV) bf16."""
    _attn_args(q, k, v, (lts, lte, uts, ute), queues, backward=True, o=o, lse=lse, do=do, dq=dq, dk=dk, dv=dv,
               ws=ws)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    wsb = lib().fm_attn_bwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_bwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(lts),
                             _ptr(lte), _ptr(uts), _ptr(ute), _ptr(queues.k_off), _ptr(queues.k_queue), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(ws), ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_bwd")
    return dq, dk, dv


def fm_attn_fwd_bwd_host(q, k, v, do, lts, lte, uts, ute, *, scale: float, causal: bool, o=None, lse=None,
                         dq=None, dk=None, dv=None, ws=None, stream=None):
    """Forward + backward from HOST tensors (page-locked for asynchronous copies):
    the library copies the inputs to its device workspace `ws` (a CUDA uint8
    tensor of fm_attn_host_workspace_bytes bytes, allocated here if None),
    classifies, runs forward and backward, and copies O, LSE, dQ, dK, dV back
    into host tensors, all enqueued on `stream`. Returns (o, lse, dq, dk, dv)
    without waiting: synchronize the stream before reading them."""
    _need(isinstance(q, torch.Tensor) and q.dim() == 4, "q must be a (B, H_q, N, d) tensor")
    B, Hq, N, d = q.shape
    _need(isinstance(k, torch.Tensor) and k.dim() == 4 and k.shape[0] == B and k.shape[3] == d,
          f"k has shape {tuple(k.shape)}, expected (B={B}, H_kv, N_kv, d={d})")
    Hkv, Nk = k.shape[1], k.shape[2]
    bf = torch.bfloat16
    for name, t, shape, dt in (("q", q, (B, Hq, N, d), bf), ("k", k, (B, Hkv, Nk, d), bf), ("v", v, (B, Hkv, Nk, d), bf),
                               ("do", do, (B, Hq, N, d), bf)):
        _like(t, name, shape, dt)
    for i, x in enumerate((lts, lte, uts, ute)):
        _like(x, f"mask vector {i}", (B, Nk), torch.int32)
    host = dict(q=q, k=k, v=v, do=do, lts=lts, lte=lte, uts=uts, ute=ute)
    o = torch.empty((B, Hq, N, d), dtype=bf, pin_memory=True) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=True) if lse is None else lse
    dq = torch.empty((B, Hq, N, d), dtype=bf, pin_memory=True) if dq is None else dq
    dk = torch.empty((B, Hkv, Nk, d), dtype=bf, pin_memory=True) if dk is None else dk
    dv = torch.empty((B, Hkv, Nk, d), dtype=bf, pin_memory=True) if dv is None else dv
    for name, t, shape, dt in (("o", o, (B, Hq, N, d), bf), ("lse", lse, (B, Hq, N), torch.float32),
                               ("dq", dq, (B, Hq, N, d), bf), ("dk", dk, (B, Hkv, Nk, d), bf),
                               ("dv", dv, (B, Hkv, Nk, d), bf)):
        _like(t, name, shape, dt)
        host[name] = t
    for name, t in host.items():
        _need(not t.is_cuda, f"{name} must be a host tensor for the host-buffer entry point")
    prob = _problem(B, Hq, Hkv, N, d, scale, causal, Nk)
    wsb = lib().fm_attn_host_workspace_bytes(ctypes.byref(prob))
    if ws is None:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device="cuda")
    _need(isinstance(ws, torch.Tensor) and ws.is_cuda and ws.dtype == torch.uint8 and ws.numel() >= wsb,
          f"ws must be a CUDA uint8 tensor of at least {wsb} bytes")
    _check(lib().fm_attn_fwd_bwd_host(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lts), _ptr(lte),
                                      _ptr(uts), _ptr(ute), _ptr(o), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _ptr(ws), ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_fwd_bwd_host")
    return o, lse, dq, dk, dv


def fm_localize(x, chunk_off, C: int, out=None, stream=None):
    """Rank-local boundaries of any int32 boundary values x for chunks at chunk_off (ascending)."""
    _like(x, "x", x.shape, torch.int32)
    _need(chunk_off.dim() == 1, "chunk_off must be one-dimensional")
    _like(chunk_off, "chunk_off", chunk_off.shape, torch.int32)
    if out is not None:
        _like(out, "out", x.shape, torch.int32)
    _same_cuda(x=x, chunk_off=chunk_off, out=out)
    out = torch.empty_like(x) if out is None else out
    _check(lib().fm_localize(_ptr(x), ctypes.c_int64(x.numel()), _ptr(chunk_off), int(chunk_off.numel()), int(C),
                             _ptr(out), _stream(stream)), "fm_localize")
    return out


def fm_from_fms_fme(fms, fme, n_rows=None, stream=None):
    """(lts, lte, uts, ute) for the FlashMask Guide's inclusive visible intervals
    [FMS_j, FME_j] (int32 CUDA tensors of one shape, e.g. (B, N_kv)); use the
    result with causal=False. n_rows: query rows N (default: the last dimension)."""
    _need(isinstance(fms, torch.Tensor) and isinstance(fme, torch.Tensor) and fms.shape == fme.shape,
          "fms and fme must be tensors of the same shape")
    _need(fms.dtype == torch.int32 and fme.dtype == torch.int32, "fms and fme must be int32")
    _same_cuda(fms=fms, fme=fme)
    fms, fme = fms.contiguous(), fme.contiguous()
    n = fms.shape[-1] if n_rows is None else int(n_rows)
    out = [torch.empty_like(fms) for _ in range(4)]
    _check(lib().fm_from_fms_fme(_ptr(fms), _ptr(fme), ctypes.c_int64(fms.numel()), n, *(_ptr(x) for x in out),
                                 _stream(stream)), "fm_from_fms_fme")
    return tuple(out)


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def fm_merge_parts(o_parts, lse_parts, o=None, lse=None, stream=None):
    """Log-sum-exp merge of M partial attentions (bf16 O_m, fp32 LSE_m of one shape each)."""
    _need(len(o_parts) == len(lse_parts) and len(o_parts) > 0, "one LSE per O part")
    oshape = tuple(o_parts[0].shape)
    _need(len(oshape) >= 1, "O parts must have a head dimension")
    for i, t in enumerate(o_parts):
        _like(t, f"O part {i}", oshape, torch.bfloat16)
    for i, t in enumerate(lse_parts):
        _like(t, f"LSE part {i}", oshape[:-1], torch.float32)
    if o is not None:
        _like(o, "o", oshape, torch.bfloat16)
    if lse is not None:
        _like(lse, "lse", oshape[:-1], torch.float32)
    _same_cuda(o=o, lse=lse, **{f"O part {i}": t for i, t in enumerate(o_parts)},
               **{f"LSE part {i}": t for i, t in enumerate(lse_parts)})
    o = torch.empty_like(o_parts[0]) if o is None else o
    lse = torch.empty_like(lse_parts[0]) if lse is None else lse
    d = oshape[-1]
    _check(lib().fm_merge_parts(len(o_parts), _ptr_array(o_parts), _ptr_array(lse_parts),
                                ctypes.c_int64(lse_parts[0].numel()), d, _ptr(o), _ptr(lse), _stream(stream)),
           "fm_merge_parts")
    return o, lse


def fm_sum_parts(parts, out=None, stream=None):
    """Elementwise sum of bf16 tensors of one shape (fp32 accumulation, one rounding)."""
    _need(len(parts) > 0, "at least one part")
    shape = tuple(parts[0].shape)
    for i, t in enumerate(parts):
        _like(t, f"part {i}", shape, torch.bfloat16)
    if out is not None:
        _like(out, "out", shape, torch.bfloat16)
    _same_cuda(out=out, **{f"part {i}": t for i, t in enumerate(parts)})
    out = torch.empty_like(parts[0]) if out is None else out
    _check(lib().fm_sum_parts(len(parts), _ptr_array(parts), ctypes.c_int64(parts[0].numel()), _ptr(out),
                              _stream(stream)), "fm_sum_parts")
    return out


def fm_classify_tiles_multi(fms, fme, *, causal: bool, n_rows=None, block_m: int = 128, block_n: int = 128,
                            stream=None):
    """Tile classes and queues of a multi-interval mask: fms, fme are
    (M, B, N_kv) int32 CUDA tensors (M <= 4), key j visible to rows
    [fms[m, b, j], fme[m, b, j]] for some m. Each column's visible rows are
    taken as their maximal runs (overlapping or touching intervals joined) and
    every tile gets the most visible of the runs' own classes; the queues have
    the layout of fm_classify_tiles for B batch entries."""
    _need(isinstance(fms, torch.Tensor) and fms.dim() == 3, "fms, fme must be (M, B, N_kv)")
    M, B, Nk = fms.shape
    for i, x in enumerate((fms, fme)):
        _like(x, ("fms", "fme")[i], (M, B, Nk), torch.int32)
    _same_cuda(fms=fms, fme=fme)
    N = Nk if n_rows is None else int(n_rows)
    prob = _problem(B, 1, 1, N, 128, 1.0, causal, Nk)
    til = fm_tiling(block_m, block_n)
    nq, nk = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().fm_tile_counts(ctypes.byref(prob), ctypes.byref(til), ctypes.byref(nq), ctypes.byref(nk)),
           "fm_tile_counts")
    nq, nk = nq.value, nk.value
    dev = fms.device
    cap = max(1, B * nq * nk)
    cls = torch.empty((B, nq, nk), dtype=torch.uint8, device=dev)
    q_off = torch.empty(B * nq + 1, dtype=torch.int32, device=dev)
    k_off = torch.empty(B * nk + 1, dtype=torch.int32, device=dev)
    q_queue = torch.empty(cap, dtype=torch.int32, device=dev)
    k_queue = torch.empty(cap, dtype=torch.int32, device=dev)
    wsb = lib().fm_classify_multi_workspace_bytes(ctypes.byref(prob), ctypes.byref(til), M)
    ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=dev)
    _check(lib().fm_classify_tiles_multi(ctypes.byref(prob), ctypes.byref(til), M, _ptr(fms), _ptr(fme), _ptr(cls),
                                         _ptr(q_off), _ptr(q_queue), _ptr(k_off), _ptr(k_queue), _ptr(ws),
                                         ctypes.c_size_t(wsb), _stream(stream)), "fm_classify_tiles_multi")
    return TileQueues(cls, q_off, q_queue, k_off, k_queue, block_m, block_n)


def _multi_args(fms, fme):
    _need(isinstance(fms, torch.Tensor) and fms.dim() == 3, "multi-interval fms, fme must be (M, B, N_kv)")
    _need(isinstance(fme, torch.Tensor) and fme.shape == fms.shape, "fms and fme must have one shape")
    return fms.shape[0]


def fm_attn_fwd_multi(q, k, v, fms, fme, queues: TileQueues, *, scale: float, causal: bool, o=None, lse=None,
                      ws=None, stream=None):
    """Forward with a multi-interval mask (fms, fme (M, B, N_kv)) and the
    queues of fm_classify_tiles_multi. Returns (O bf16, LSE fp32)."""
    M = _multi_args(fms, fme)
    _attn_args(q, k, v, (fms, fme), queues, backward=False, o=o, lse=lse, ws=ws, intervals=M)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wsb = lib().fm_attn_fwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_fwd_multi(ctypes.byref(prob), M, _ptr(q), _ptr(k), _ptr(v), _ptr(fms), _ptr(fme),
                                   _ptr(queues.q_off), _ptr(queues.q_queue), _ptr(o), _ptr(lse), _ptr(ws),
                                   ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_fwd_multi")
    return o, lse


def fm_attn_bwd_multi(q, k, v, o, lse, do, fms, fme, queues: TileQueues, *, scale: float, causal: bool, dq=None,
                      dk=None, dv=None, ws=None, stream=None):
    """Backward with a multi-interval mask (fms, fme (M, B, N_kv)): returns
    (dQ, dK, dV) bf16."""
    M = _multi_args(fms, fme)
    _attn_args(q, k, v, (fms, fme), queues, backward=True, o=o, lse=lse, do=do, dq=dq, dk=dk, dv=dv, ws=ws,
               intervals=M)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    wsb = lib().fm_attn_bwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_bwd_multi(ctypes.byref(prob), M, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                   _ptr(fms), _ptr(fme), _ptr(queues.k_off), _ptr(queues.k_queue), _ptr(dq),
                                   _ptr(dk), _ptr(dv), _ptr(ws), ctypes.c_size_t(wsb), _stream(stream)),
           "fm_attn_bwd_multi")
    return dq, dk, dv


def fm_attn_multi_interval(q, k, v, fms, fme, *, scale: float, do=None, causal: bool = False, stream=None):
    """Attention under a multi-interval mask: fms, fme are (M, B, N_kv) int32
    CUDA tensors (M <= 4), key j visible to rows [fms[m, b, j], fme[m, b, j]]
    (inclusive) for some m (intervals may overlap), and to no row before j
    when causal. Library calls only: fm_classify_tiles_multi, then
    fm_attn_fwd_multi and, with do, fm_attn_bwd_multi (each block computed
    once, masked by the union of the intervals).
    Returns (o, lse) or (o, lse, dq, dk, dv)."""
    qs = fm_classify_tiles_multi(fms, fme, causal=causal, n_rows=q.shape[2], stream=stream)
    o, lse = fm_attn_fwd_multi(q, k, v, fms, fme, qs, scale=scale, causal=causal, stream=stream)
    if do is None:
        return o, lse
    dq, dk, dv = fm_attn_bwd_multi(q, k, v, o, lse, do, fms, fme, qs, scale=scale, causal=causal, stream=stream)
    return o, lse, dq, dk, dv


def fm_classify_tiles_heads(lts, lte, uts, ute, *, causal: bool, n_rows=None, stream=None):
    """Queues for per-head mask vectors (B, H_q, N_kv): fm_classify_tiles over
    the B * H_q rows, row b * H_q + h holding query head h of batch entry b."""
    _need(isinstance(lts, torch.Tensor) and lts.dim() == 3, "per-head mask vectors must be (B, H_q, N_kv)")
    B, Hq, Nk = lts.shape
    for i, x in enumerate((lts, lte, uts, ute)):
        _like(x, f"mask vector {i}", (B, Hq, Nk), torch.int32)
    return fm_classify_tiles(*(x.view(B * Hq, Nk) for x in (lts, lte, uts, ute)), causal=causal, n_rows=n_rows,
                             stream=stream)


def fm_attn_fwd_heads(q, k, v, lts, lte, uts, ute, queues: TileQueues, *, scale: float, causal: bool, o=None,
                      lse=None, ws=None, stream=None):
    """Forward with per-head mask vectors (B, H_q, N_kv) and the queues of
    fm_classify_tiles_heads: returns (O bf16, LSE fp32)."""
    _attn_args(q, k, v, (lts, lte, uts, ute), queues, backward=False, o=o, lse=lse, ws=ws, heads=True)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    wsb = lib().fm_attn_fwd_heads_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_fwd_heads(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(lts), _ptr(lte), _ptr(uts),
                                   _ptr(ute), _ptr(queues.q_off), _ptr(queues.q_queue), _ptr(o), _ptr(lse),
                                   _ptr(ws), ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_fwd_heads")
    return o, lse


def fm_attn_bwd_heads(q, k, v, o, lse, do, lts, lte, uts, ute, queues: TileQueues, *, scale: float, causal: bool,
                      dq=None, dk=None, dv=None, ws=None, stream=None):
    """Backward with per-head mask vectors: returns (dQ, dK, dV) bf16."""
    _attn_args(q, k, v, (lts, lte, uts, ute), queues, backward=True, o=o, lse=lse, do=do, dq=dq, dk=dk, dv=dv,
               ws=ws, heads=True)
    B, Hq, N, d = q.shape
    prob = _problem(B, Hq, k.shape[1], N, d, scale, causal, k.shape[2])
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    wsb = lib().fm_attn_bwd_workspace_bytes(ctypes.byref(prob))
    if ws is None or ws.numel() < wsb:
        ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=q.device)
    _check(lib().fm_attn_bwd_heads(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                   _ptr(lts), _ptr(lte), _ptr(uts), _ptr(ute), _ptr(queues.k_off),
                                   _ptr(queues.k_queue), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                   ctypes.c_size_t(wsb), _stream(stream)), "fm_attn_bwd_heads")
    return dq, dk, dv


def fm_attn_per_head(q, k, v, lts, lte, uts, ute, *, causal: bool, scale: float, do=None, stream=None):
    """Attention with one set of mask vectors per query head: lts..ute are
    (B, H_q, N_kv) int32 CUDA tensors. One classification over the B * H_q
    vector rows, one forward and (with do) one backward, each a single launch
    over every head. Returns (o, lse) or (o, lse, dq, dk, dv)."""
    qs = fm_classify_tiles_heads(lts, lte, uts, ute, causal=causal, n_rows=q.shape[2] if q.dim() == 4 else None,
                                 stream=stream)
    o, lse = fm_attn_fwd_heads(q, k, v, lts, lte, uts, ute, qs, scale=scale, causal=causal, stream=stream)
    if do is None:
        return o, lse
    dq, dk, dv = fm_attn_bwd_heads(q, k, v, o, lse, do, lts, lte, uts, ute, qs, scale=scale, causal=causal,
                                   stream=stream)
    return o, lse, dq, dk, dv


def fm_device_status(stream=None):
    """(status, bits) of the device error word; synchronizes the stream and clears the word."""
    bits = ctypes.c_int32(0)
    st = lib().fm_device_status(_stream(stream), ctypes.byref(bits))
    return st, bits.value


def fm_selftest_wait_timeout(limit_us: int, stream=None):
    _check(lib().fm_selftest_wait_timeout(ctypes.c_int64(limit_us), _stream(stream)), "fm_selftest_wait_timeout")


def fm_profile_enable(on: bool):
    _check(lib().fm_profile_enable(1 if on else 0), "fm_profile_enable")


def fm_profile_read():
    """{'fwd_ms', 'fwd_launches', 'bwd_ms', 'bwd_launches'} since the last read (synchronizes)."""
    fm_, fl, bm_, bl = ctypes.c_double(), ctypes.c_int32(), ctypes.c_double(), ctypes.c_int32()
    _check(lib().fm_profile_read(ctypes.byref(fm_), ctypes.byref(fl), ctypes.byref(bm_), ctypes.byref(bl)),
           "fm_profile_read")
    return dict(fwd_ms=fm_.value, fwd_launches=fl.value, bwd_ms=bm_.value, bwd_launches=bl.value)


def fm_launch_count() -> int:
    return int(lib().fm_launch_count())


def _host_array(x, dtype):
    """A contiguous host numpy array of `dtype` holding x (numpy array or torch tensor, any device)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        raise ValueError(f"expected {np.dtype(dtype).name} values, got {a.dtype}")
    return a


def fm_chunk_loads(tile_class, blocks_per_chunk: int, cost_partial: int, cost_unmasked: int) -> np.ndarray:
    """Per-chunk loads (int64) from the (B, nQ, nK) tile classes (copied to the host if on a GPU)."""
    cls = _host_array(tile_class, np.uint8)
    if cls.ndim != 3:
        raise ValueError("tile_class must be (B, nQ, nK)")
    B, nq, nk = cls.shape
    w = np.empty(-(-nq // int(blocks_per_chunk)) if blocks_per_chunk > 0 else 0, dtype=np.int64)
    _check(lib().fm_chunk_loads(ctypes.c_void_p(cls.ctypes.data), B, nq, nk, int(blocks_per_chunk),
                                int(cost_partial), int(cost_unmasked), ctypes.c_void_p(w.ctypes.data)),
           "fm_chunk_loads")
    return w


def fm_needed_chunks(tile_class, owner, P: int, blocks_per_chunk: int) -> np.ndarray:
    """(P, n_chunks) uint8: 1 where rank r's rows can see some key of chunk c."""
    cls = _host_array(tile_class, np.uint8)
    own = _host_array(np.asarray(owner, dtype=np.int32) if not isinstance(owner, torch.Tensor) else owner, np.int32)
    if cls.ndim != 3:
        raise ValueError("tile_class must be (B, nQ, nK)")
    B, nq, nk = cls.shape
    need = np.empty((int(P), own.size), dtype=np.uint8)
    _check(lib().fm_needed_chunks(ctypes.c_void_p(cls.ctypes.data), B, nq, nk, ctypes.c_void_p(own.ctypes.data),
                                  own.size, int(P), int(blocks_per_chunk), ctypes.c_void_p(need.ctypes.data)),
           "fm_needed_chunks")
    return need


def fm_balance_chunks(w, P: int, kappa: int, phases: int = 3, node_budget: int = 0):
    """HCC-IPO Stage 1 on chunk loads w: returns (owner int32 array, report dict)."""
    wa = _host_array(w, np.int64)
    owner = np.empty(wa.size, dtype=np.int32)
    rep = fm_balance_report()
    _check(lib().fm_balance_chunks(ctypes.c_void_p(wa.ctypes.data), int(wa.size), int(P), int(kappa), int(phases),
                                   int(node_budget), ctypes.c_void_p(owner.ctypes.data), ctypes.byref(rep)),
           "fm_balance_chunks")
    return owner, {name: int(getattr(rep, name)) for name, _ in fm_balance_report._fields_}


class _FlashMaskFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, lts, lte, uts, ute, scale, causal):
        bm, bn = attn_tiling()
        queues = fm_classify_tiles(lts, lte, uts, ute, causal=causal, block_m=bm, block_n=bn, n_rows=q.shape[2])
        o, lse = fm_attn_fwd(q, k, v, lts, lte, uts, ute, queues, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse, lts, lte, uts, ute)
        ctx.queues, ctx.scale, ctx.causal = queues, scale, causal
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, lts, lte, uts, ute = ctx.saved_tensors
        dq, dk, dv = fm_attn_bwd(q, k, v, o, lse, do.contiguous(), lts, lte, uts, ute, ctx.queues, scale=ctx.scale,
                                 causal=ctx.causal)
        return dq, dk, dv, None, None, None, None, None, None


def flashmask_attention(q, k, v, lts, lte, uts, ute, *, causal: bool, scale: float | None = None):
    """Masked SDPA with the FlashMask column-wise mask; differentiable in q, k, v."""
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    return _FlashMaskFn.apply(q, k, v, lts, lte, uts, ute, float(scale), bool(causal))
