"""The C ABI library: it builds, loads, exports every declared symbol, and its
host-side validation rejects bad calls without touching a GPU."""
import ctypes
import os
import re

import pytest

import mask_aware_sparse_gb300 as fm
from mask_aware_sparse_gb300 import build as fmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fmbuild.build()
    return fm.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "fm.h")).read()
    return sorted(set(re.findall(r"\b(fm_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = _declared()
    assert "fm_attn_fwd" in names and "fm_classify_tiles" in names
    for n in names:
        assert hasattr(lib, n), n
    # the binding declares exactly the header's entry points
    assert sorted(fm.EXPORTS) == names


def test_abi_version(lib):
    assert lib.fm_abi_version() == 3


def test_status_strings(lib):
    for s in range(7):
        assert len(fm.status_string(s)) > 0


def test_tile_counts_host_only(lib):
    p = fm._problem(2, 4, 2, 1000, 128, 0.1, 1)
    t = fm.fm_tiling(128, 64)
    nq, nk = ctypes.c_int32(), ctypes.c_int32()
    assert lib.fm_tile_counts(ctypes.byref(p), ctypes.byref(t), ctypes.byref(nq), ctypes.byref(nk)) == fm.FM_OK
    assert (nq.value, nk.value) == (8, 16)
    bad = fm.fm_tiling(100, 64)
    assert lib.fm_tile_counts(ctypes.byref(p), ctypes.byref(bad), ctypes.byref(nq), ctypes.byref(nk)) == \
        fm.FM_ERR_INVALID_ARG


def test_attn_tiling(lib):
    assert fm.attn_tiling() == (128, 128)


def test_validation_rejects_before_any_launch(lib):
    P = ctypes.POINTER(fm.fm_problem)
    nul = ctypes.c_void_p(0)
    # H_q not a multiple of H_kv
    p = fm._problem(1, 6, 4, 256, 128, 0.1, 1)
    args = [nul] * 11 + [nul, ctypes.c_size_t(0), nul]
    assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_ERR_INVALID_ARG
    # unsupported head dim
    p = fm._problem(1, 4, 2, 256, 96, 0.1, 1)
    assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_ERR_UNSUPPORTED
    # null tensors
    p = fm._problem(1, 4, 2, 256, 128, 0.1, 1)
    assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_ERR_INVALID_ARG
    bargs = [nul] * 15 + [nul, ctypes.c_size_t(0), nul]
    assert lib.fm_attn_bwd(ctypes.byref(p), *bargs) == fm.FM_ERR_INVALID_ARG
    # negative sizes
    p = fm._problem(1, 4, 2, -5, 128, 0.1, 1)
    assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_ERR_INVALID_ARG
    # non-finite scale
    p = fm._problem(1, 4, 2, 256, 128, float("nan"), 1)
    assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_ERR_INVALID_ARG
    # null problem
    assert lib.fm_attn_fwd(P(), *args) == fm.FM_ERR_INVALID_ARG


def test_empty_problems_are_noops(lib):
    nul = ctypes.c_void_p(0)
    for shape in ((0, 4, 2, 256), (1, 0, 2, 256), (1, 4, 2, 0)):
        p = fm._problem(*shape, 128, 0.1, 1)
        args = [nul] * 11 + [nul, ctypes.c_size_t(0), nul]
        assert lib.fm_attn_fwd(ctypes.byref(p), *args) == fm.FM_OK
        bargs = [nul] * 15 + [nul, ctypes.c_size_t(0), nul]
        assert lib.fm_attn_bwd(ctypes.byref(p), *bargs) == fm.FM_OK
    assert lib.fm_localize(nul, 0, nul, 1, 4, nul, nul) == fm.FM_OK
    assert lib.fm_localize(nul, 10, nul, 0, 4, nul, nul) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_from_fms_fme(nul, nul, 0, 16, nul, nul, nul, nul, nul) == fm.FM_OK
    assert lib.fm_from_fms_fme(nul, nul, 8, 16, nul, nul, nul, nul, nul) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_from_fms_fme(nul, nul, -1, 16, nul, nul, nul, nul, nul) == fm.FM_ERR_INVALID_ARG
    # merge / sum of parts: 1..8 parts, rows and elements >= 0, d a multiple of 8
    assert lib.fm_merge_parts(2, nul, nul, 0, 128, nul, nul, nul) == fm.FM_OK
    for M, rows, d in ((0, 4, 128), (9, 4, 128), (2, -1, 128), (2, 4, 12), (2, 4, 0)):
        assert lib.fm_merge_parts(M, nul, nul, rows, d, nul, nul, nul) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_merge_parts(2, nul, nul, 4, 128, nul, nul, nul) == fm.FM_ERR_INVALID_ARG  # null arrays
    assert lib.fm_sum_parts(3, nul, 0, nul, nul) == fm.FM_OK
    assert lib.fm_sum_parts(0, nul, 8, nul, nul) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_sum_parts(9, nul, 8, nul, nul) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_sum_parts(2, nul, 8, nul, nul) == fm.FM_ERR_INVALID_ARG


def test_rectangular_problem_shapes(lib):
    # N query rows, N_kv keys: tile counts follow each axis; N_kv = 0 is N
    t = fm.fm_tiling(128, 64)
    nq, nk = ctypes.c_int32(), ctypes.c_int32()
    p = fm._problem(1, 4, 2, 300, 128, 0.1, 0, 1000)
    assert lib.fm_tile_counts(ctypes.byref(p), ctypes.byref(t), ctypes.byref(nq), ctypes.byref(nk)) == fm.FM_OK
    assert (nq.value, nk.value) == (3, 16)
    p = fm._problem(1, 4, 2, 300, 128, 0.1, 0, 0)
    assert lib.fm_tile_counts(ctypes.byref(p), ctypes.byref(t), ctypes.byref(nq), ctypes.byref(nk)) == fm.FM_OK
    assert (nq.value, nk.value) == (3, 5)
    p = fm._problem(1, 4, 2, 300, 128, 0.1, 0, -1)
    assert lib.fm_tile_counts(ctypes.byref(p), ctypes.byref(t), ctypes.byref(nq), ctypes.byref(nk)) == \
        fm.FM_ERR_INVALID_ARG
    # workspaces follow the axes too: the backward's dQ accumulator by rows,
    # its launch-order table by key blocks
    a = fm._problem(1, 4, 2, 256, 128, 0.1, 0, 65536)
    b = fm._problem(1, 4, 2, 256, 128, 0.1, 0, 256)
    assert lib.fm_attn_bwd_workspace_bytes(ctypes.byref(a)) > lib.fm_attn_bwd_workspace_bytes(ctypes.byref(b))
    assert lib.fm_attn_fwd_workspace_bytes(ctypes.byref(a)) == lib.fm_attn_fwd_workspace_bytes(ctypes.byref(b))


def test_workspace_queries(lib):
    p = fm._problem(1, 32, 8, 32768, 128, 0.1, 1)
    t = fm.fm_tiling(128, 128)
    assert lib.fm_classify_workspace_bytes(ctypes.byref(p), ctypes.byref(t)) > 0
    assert lib.fm_attn_fwd_workspace_bytes(ctypes.byref(p)) >= 4 * 256
    assert lib.fm_attn_bwd_workspace_bytes(ctypes.byref(p)) > 0


def test_binding_refuses_host_tensors(lib):
    # the product path runs on the GPU only: host tensors are refused up front,
    # never computed some other way
    import torch

    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    vec = [torch.zeros(1, 128, dtype=torch.int32) for _ in range(4)]
    with pytest.raises(ValueError):
        fm.fm_classify_tiles(*vec, causal=True)
    with pytest.raises(ValueError):
        fm.fm_attn_fwd(q, k, k, *vec, None, scale=0.125, causal=True)
    with pytest.raises(ValueError):
        fm.fm_attn_per_head(q, k, k, *[torch.zeros(1, 2, 128, dtype=torch.int32)] * 4, causal=True, scale=0.125)
    with pytest.raises(ValueError):
        fm.fm_from_fms_fme(vec[0], vec[1])
    with pytest.raises(ValueError):
        fm.fm_merge_parts([q], [torch.zeros(1, 2, 127)])  # LSE shape must be O's without d
    with pytest.raises(ValueError):
        fm.fm_sum_parts([q, k])  # parts of different shapes


def test_binding_checks_shapes_before_any_library_call(lib):
    # The C ABI receives bare pointers and cannot see shapes: the binding must
    # refuse every mismatch before a pointer reaches the library. Shape checks
    # run before the device check, so these host tensors fail on the shape.
    import torch

    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    B, Hq, Hkv, N, d = 1, 4, 2, 256, 64
    q = torch.zeros(B, Hq, N, d, dtype=bf)
    k = torch.zeros(B, Hkv, N, d, dtype=bf)
    vec = [torch.zeros(B, N, dtype=i32) for _ in range(4)]
    cases = [
        dict(k=torch.zeros(B, Hkv, N, 2 * d, dtype=bf)),          # K head dim differs from Q
        dict(k=torch.zeros(B + 1, Hkv, N, d, dtype=bf)),           # K batch differs
        dict(v=torch.zeros(B, Hkv, N // 2, d, dtype=bf)),          # V rows differ from K
        dict(k=torch.zeros(B, 3, N, d, dtype=bf), v=torch.zeros(B, 3, N, d, dtype=bf)),  # H_q % H_kv
        dict(vec=[torch.zeros(B, N + 1, dtype=i32)] * 4),          # vectors not (B, N_kv)
        dict(vec=[torch.zeros(B, N, dtype=torch.int64)] * 4),      # vectors not int32
        dict(o=torch.zeros(B, Hq, N + 128, d, dtype=bf)),          # output larger than Q
        dict(lse=torch.zeros(B, Hq, 2 * N, dtype=f32)),            # LSE larger than (B, H_q, N)
    ]
    for c in cases:
        kk = c.get("k", k)
        vv = c.get("v", kk if "k" in c else k)
        with pytest.raises(ValueError, match="shape|multiple|must be torch|expected|int32"):
            fm.fm_attn_fwd(q, kk, vv, *c.get("vec", vec), None, scale=0.1, causal=True, o=c.get("o"),
                           lse=c.get("lse"))
    lse = torch.zeros(B, Hq, N, dtype=f32)
    bwd_cases = [
        dict(do=torch.zeros(B, Hq, N, d // 2, dtype=bf)),
        dict(dq=torch.zeros(B, Hq, N + 1, d, dtype=bf)),
        dict(dk=torch.zeros(B, Hq, N, d, dtype=bf)),               # dK with H_q heads instead of H_kv
        dict(dv=torch.zeros(B, Hkv, N, d, dtype=f32)),
    ]
    for c in bwd_cases:
        with pytest.raises(ValueError, match="shape|must be torch"):
            fm.fm_attn_bwd(q, k, k, q, lse, c.get("do", q), *vec, None, scale=0.1, causal=True,
                           dq=c.get("dq"), dk=c.get("dk"), dv=c.get("dv"))
    # all shapes right: the queues object is checked next, then the device
    with pytest.raises(ValueError, match="fm_classify_tiles"):
        fm.fm_attn_fwd(q, k, k, *vec, None, scale=0.1, causal=True)
    nq = N // 128
    queues = fm.TileQueues(torch.zeros(B, nq, nq, dtype=torch.uint8), torch.zeros(B * nq + 1, dtype=i32),
                           torch.zeros(B * nq * nq, dtype=i32), torch.zeros(B * nq + 1, dtype=i32),
                           torch.zeros(B * nq * nq, dtype=i32), 128, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_fwd(q, k, k, *vec, queues, scale=0.1, causal=True)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_bwd(q, k, k, q, lse, q, *vec, queues, scale=0.1, causal=True)
    short = fm.TileQueues(queues.tile_class, torch.zeros(B * nq, dtype=i32), queues.q_queue, queues.k_off,
                          queues.k_queue, 128, 128)
    with pytest.raises(ValueError, match="queue offsets"):
        fm.fm_attn_fwd(q, k, k, *vec, short, scale=0.1, causal=True)
    other_tiling = fm.TileQueues(*[getattr(queues, f) for f in ("tile_class", "q_off", "q_queue", "k_off",
                                                                "k_queue")], 64, 64)
    with pytest.raises(ValueError, match="tiles"):
        fm.fm_attn_fwd(q, k, k, *vec, other_tiling, scale=0.1, causal=True)


def test_binding_refuses_host_and_mismatched_parts(lib):
    import torch

    o = torch.zeros(2, 3, 16, 8, dtype=torch.bfloat16)
    lse = torch.zeros(2, 3, 16, dtype=torch.float32)
    # host-memory parts: never handed to a kernel as raw pointers
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_merge_parts([o, o], [lse, lse])
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_sum_parts([o, o])
    # outputs larger or smaller than the parts: the row / element count comes
    # from the parts, and a mismatched output is refused
    with pytest.raises(ValueError, match="shape"):
        fm.fm_merge_parts([o, o], [lse, lse], o=torch.zeros(2, 3, 32, 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="shape"):
        fm.fm_merge_parts([o, o], [lse, lse], lse=torch.zeros(2, 3, 32, dtype=torch.float32))
    with pytest.raises(ValueError, match="shape"):
        fm.fm_sum_parts([o, o], out=torch.zeros(2, 3, 16, 16, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="bfloat16"):
        fm.fm_sum_parts([o, o], out=torch.zeros(2, 3, 16, 8, dtype=torch.float32))
    # localization and the FMS / FME converter: host tensors are refused
    x = torch.zeros(64, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_localize(x, torch.zeros(2, dtype=torch.int32), 16)
    with pytest.raises(ValueError, match="shape"):
        fm.fm_localize(x, torch.zeros(2, dtype=torch.int32), 16, out=torch.zeros(32, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_from_fms_fme(x, x)
    with pytest.raises(ValueError, match="same shape"):
        fm.fm_from_fms_fme(x, x[:32])


def test_binding_checks_per_head_shapes(lib):
    # per-head entry points: vectors are (B, H_q, N_kv) and the queues have
    # B * H_q rows per Q (K) block; shared-shape vectors or shared-shape queues
    # are refused before any pointer reaches the library
    import torch

    bf, i32 = torch.bfloat16, torch.int32
    B, Hq, Hkv, N, d = 2, 4, 2, 256, 64
    q = torch.zeros(B, Hq, N, d, dtype=bf)
    k = torch.zeros(B, Hkv, N, d, dtype=bf)
    lse = torch.zeros(B, Hq, N, dtype=torch.float32)
    shared = [torch.zeros(B, N, dtype=i32) for _ in range(4)]
    per = [torch.zeros(B, Hq, N, dtype=i32) for _ in range(4)]
    nq = N // 128

    def queues(rows):
        return fm.TileQueues(torch.zeros(rows, nq, nq, dtype=torch.uint8), torch.zeros(rows * nq + 1, dtype=i32),
                             torch.zeros(rows * nq * nq, dtype=i32), torch.zeros(rows * nq + 1, dtype=i32),
                             torch.zeros(rows * nq * nq, dtype=i32), 128, 128)

    with pytest.raises(ValueError, match="shape"):
        fm.fm_attn_fwd_heads(q, k, k, *shared, queues(B * Hq), scale=0.1, causal=True)
    with pytest.raises(ValueError, match="queue offsets"):
        fm.fm_attn_fwd_heads(q, k, k, *per, queues(B), scale=0.1, causal=True)
    with pytest.raises(ValueError, match="queue offsets"):
        fm.fm_attn_bwd_heads(q, k, k, q, lse, q, *per, queues(B), scale=0.1, causal=True)
    with pytest.raises(ValueError, match="H_q, N_kv"):
        fm.fm_classify_tiles_heads(*shared, causal=True)
    # right shapes: only the device is left to refuse
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_fwd_heads(q, k, k, *per, queues(B * Hq), scale=0.1, causal=True)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_bwd_heads(q, k, k, q, lse, q, *per, queues(B * Hq), scale=0.1, causal=True)


def test_binding_checks_multi_interval_shapes(lib):
    # multi-interval entry points: FMS / FME are (M, B, N_kv) and the queues
    # (from fm_classify_tiles_multi) have B rows per Q (K) block; anything
    # else is refused before any pointer reaches the library
    import torch

    bf, i32 = torch.bfloat16, torch.int32
    M, B, Hq, Hkv, N, d = 3, 2, 4, 2, 256, 64
    q = torch.zeros(B, Hq, N, d, dtype=bf)
    k = torch.zeros(B, Hkv, N, d, dtype=bf)
    lse = torch.zeros(B, Hq, N, dtype=torch.float32)
    flat = torch.zeros(B, N, dtype=i32)
    fms = torch.zeros(M, B, N, dtype=i32)
    nq = N // 128

    def queues(rows):
        return fm.TileQueues(torch.zeros(rows, nq, nq, dtype=torch.uint8), torch.zeros(rows * nq + 1, dtype=i32),
                             torch.zeros(rows * nq * nq, dtype=i32), torch.zeros(rows * nq + 1, dtype=i32),
                             torch.zeros(rows * nq * nq, dtype=i32), 128, 128)

    with pytest.raises(ValueError, match=r"\(M, B, N_kv\)"):
        fm.fm_attn_fwd_multi(q, k, k, flat, flat, queues(B), scale=0.1, causal=False)
    with pytest.raises(ValueError, match="one shape"):
        fm.fm_attn_fwd_multi(q, k, k, fms, fms[:2], queues(B), scale=0.1, causal=False)
    with pytest.raises(ValueError, match="queue offsets"):
        fm.fm_attn_fwd_multi(q, k, k, fms, fms, queues(M * B), scale=0.1, causal=False)
    with pytest.raises(ValueError, match="queue offsets"):
        fm.fm_attn_bwd_multi(q, k, k, q, lse, q, fms, fms, queues(M * B), scale=0.1, causal=False)
    with pytest.raises(ValueError, match=r"\(M, B, N_kv\)"):
        fm.fm_classify_tiles_multi(flat, flat, causal=False)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_fwd_multi(q, k, k, fms, fms, queues(B), scale=0.1, causal=False)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fm.fm_attn_bwd_multi(q, k, k, q, lse, q, fms, fms, queues(B), scale=0.1, causal=False)


def test_multi_interval_entry_points_validate_before_any_launch(lib):
    # 1 <= M <= 4 intervals, then the usual checks, all before any launch
    nul = ctypes.c_void_p(0)
    args = [nul] * 9 + [nul, ctypes.c_size_t(0), nul]
    bargs = [nul] * 13 + [nul, ctypes.c_size_t(0), nul]
    cargs = [nul] * 7 + [nul, ctypes.c_size_t(0), nul]
    til = fm.fm_tiling(128, 128)
    p = fm._problem(1, 4, 2, 256, 128, 0.1, 0)
    for M, want in ((0, fm.FM_ERR_INVALID_ARG), (5, fm.FM_ERR_INVALID_ARG), (2, fm.FM_ERR_INVALID_ARG)):
        assert lib.fm_attn_fwd_multi(ctypes.byref(p), M, *args) == want
        assert lib.fm_attn_bwd_multi(ctypes.byref(p), M, *bargs) == want
        assert lib.fm_classify_tiles_multi(ctypes.byref(p), ctypes.byref(til), M, *cargs) == want
    q = fm._problem(1, 4, 2, 256, 96, 0.1, 0)
    assert lib.fm_attn_fwd_multi(ctypes.byref(q), 2, *args) == fm.FM_ERR_UNSUPPORTED
    e = fm._problem(0, 4, 2, 256, 128, 0.1, 0)
    assert lib.fm_attn_fwd_multi(ctypes.byref(e), 2, *args) == fm.FM_OK
    assert lib.fm_attn_bwd_multi(ctypes.byref(e), 9, *bargs) == fm.FM_ERR_INVALID_ARG
    # the classification workspace grows with the intervals
    a = fm._problem(1, 1, 1, 4096, 128, 0.1, 0)
    w1 = lib.fm_classify_multi_workspace_bytes(ctypes.byref(a), ctypes.byref(til), 1)
    w4 = lib.fm_classify_multi_workspace_bytes(ctypes.byref(a), ctypes.byref(til), 4)
    assert 0 < w1 < w4 and lib.fm_classify_multi_workspace_bytes(ctypes.byref(a), ctypes.byref(til), 5) == 0


def test_per_head_entry_points_validate_before_any_launch(lib):
    # the C side refuses groups of more than 64 query heads per kv head and
    # null tensors before touching a pointer; its workspace
    # query counts one order entry per (batch, head, Q block)
    nul = ctypes.c_void_p(0)
    args = [nul] * 11 + [nul, ctypes.c_size_t(0), nul]
    bargs = [nul] * 15 + [nul, ctypes.c_size_t(0), nul]
    for shape, want in (((1, 130, 2, 256, 128), fm.FM_ERR_UNSUPPORTED),   # 65 heads per kv head
                        ((1, 4, 2, 256, 96), fm.FM_ERR_UNSUPPORTED),      # d = 96
                        ((1, 4, 2, 256, 256), fm.FM_ERR_INVALID_ARG),     # d = 256, null tensors
                        ((1, 4, 2, 256, 128), fm.FM_ERR_INVALID_ARG)):    # null tensors
        p = fm._problem(*shape, 0.1, 1)
        assert lib.fm_attn_fwd_heads(ctypes.byref(p), *args) == want
        assert lib.fm_attn_bwd_heads(ctypes.byref(p), *bargs) == want
    p = fm._problem(0, 4, 2, 256, 128, 0.1, 1)
    assert lib.fm_attn_fwd_heads(ctypes.byref(p), *args) == fm.FM_OK
    a = fm._problem(2, 64, 8, 32768, 128, 0.1, 1)
    assert lib.fm_attn_fwd_heads_workspace_bytes(ctypes.byref(a)) >= 4 * 2 * 64 * 256
    assert lib.fm_attn_fwd_heads_workspace_bytes(ctypes.byref(a)) > lib.fm_attn_fwd_workspace_bytes(ctypes.byref(a))
