"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every symbol the header declares, and its argument checks and host-only
functions behave as documented.  No call here reaches the GPU: every error
case is rejected by the host checks before anything is enqueued."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp_fused.h")


@pytest.fixture(scope="module")
def tp():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import gemm_reduce_fusion_gb300 as tp
    return tp


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["tp_row_linear_fwd_allreduce", "tp_row_linear_fwd_reducescatter", "tp_col_linear_fwd",
              "tp_col_linear_bwd", "tp_ag_matmul", "tp_row_linear_bwd", "tp_workspace_size",
              "tp_choose_chunk_m_measured",
              "tp_pipeline_time", "tp_choose_chunk_m", "tp_get_device_status", "tp_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(tp):
    lib = ctypes.CDLL(tp.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tp.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (tp_\w+)", out))
    assert set(declared_functions()) <= exported


def test_status_strings(tp):
    for s in range(8):
        assert tp.tp_status_string(s)
    assert "unknown" in tp.tp_status_string(99)


def test_pipeline_time_matches_oracle(tp):
    for c, m, n in [(3, 2, 4), (1, 5, 4), (2, 2, 1), (0.5, 0.25, 128), (3, 2, 0)]:
        assert tp.tp_pipeline_time(c, m, n) == oracle.pipeline_time(c, m, n)
    assert tp.tp_pipeline_time(3, 2, 4) == 14.0   # M027 §03


def test_num_chunks_matches_oracle(tp):
    for M, c in [(128, 32), (130, 32), (16, 2048), (2048, 16), (2048, 64), (0, 32), (7, 7)]:
        assert tp.tp_num_chunks(M, c) == oracle.n_chunks(M, c)


def test_choose_chunk_m_is_valid(tp):
    for op in range(6):
        for p, M, N, K in [(2, 128, 2048, 1024), (4, 4096, 4096, 4096), (8, 16, 6144, 12288),
                           (8, 2048, 12288, 6144), (1, 1, 8, 8)]:
            c = tp.tp_choose_chunk_m(op, p, M, N, K)
            assert 1 <= c <= M
    assert tp.tp_choose_chunk_m(0, 2, 0, 8, 8) == 0
    assert tp.tp_choose_chunk_m(tp.TP_OP_COL_FWD, 8, 16, 6144, 12288) == 16


def test_choose_chunk_m_from_measured_times(tp):
    """The page's two-engine example: M = 128 in 4 chunks of 32 with c = 3,
    m = 2 gives 14 against 20 unchunked (c = 12, m = 8 for one chunk of
    128); the shortest timeline wins, checked against the oracle's closed
    form."""
    chunks, c, m = [128, 32], [12.0, 3.0], [8.0, 2.0]
    assert tp.tp_choose_chunk_m_measured(128, chunks, c, m) == 32
    ts = [oracle.pipeline_time(ci, mi, oracle.n_chunks(128, k)) for k, ci, mi in zip(chunks, c, m)]
    assert ts == [20.0, 14.0]
    # small chunks whose compute no longer shrinks lose (the page's warning)
    assert tp.tp_choose_chunk_m_measured(128, [128, 16], [12.0, 3.0], [8.0, 2.0]) == 128
    assert tp.tp_choose_chunk_m_measured(128, [], [], []) == 0
    assert tp.tp_choose_chunk_m_measured(0, [32], [1.0], [1.0]) == 0


def test_trace_set_argument_checks(tp):
    lib = tp._lib
    assert lib.tp_trace_set(None, 5) == tp.TP_ERR_INVALID_ARG       # size without a buffer
    assert lib.tp_trace_set(A, 0) == tp.TP_ERR_INVALID_ARG          # buffer without a size
    assert lib.tp_trace_set(A, -1) == tp.TP_ERR_INVALID_ARG
    assert lib.tp_trace_set(A + 8, 16) == tp.TP_ERR_ALIGNMENT
    assert lib.tp_trace_set(None, 0) == tp.TP_OK                    # off


def test_workspace_size(tp):
    assert tp.tp_workspace_size(tp.TP_OP_ROW_AR, 4, 4096, 4096, 4096, 0) >= 256
    # a skinny call plans an operand-swapped split-K whose fp32 partials,
    # one copy of Y per split, go to the second-stage kernel
    small = tp.tp_workspace_size(tp.TP_OP_ROW_AR, 8, 16, 12288, 6144, 16)
    assert small > 256 and (small - 256) % (16 * 12288 * 4) == 0
    # invalid requests still return the minimum
    assert tp.tp_workspace_size(tp.TP_OP_ROW_AR, 0, 16, 16, 16, 0) == 256


def test_split_plan_and_forced_split(tp):
    """The split-K factor of launches below one wave: the largest that keeps
    every unit in one wave, none for a GEMM too small to repay the second
    stage, the SM-filling split for HBM-bound skinny calls over long
    contractions; TP_DEBUG_SPLIT_K overrides it (fp32 partials: one copy of
    the output per split)."""
    def splits(op, p, M, N, K, chunk):
        return (tp.tp_workspace_size(op, p, M, N, K, chunk) - 256) / (M * N * 4)
    AR = tp.TP_OP_ROW_AR
    # [128, 2048] output in 64 swapped tiles of 32 tokens, 32 k-blocks: 2 splits fill one wave
    assert splits(AR, 2, 128, 2048, 1024, 32) == 2
    # 32 tiles of 128 x 256, 64 k-blocks: 4 splits
    assert splits(AR, 4, 1024, 1024, 1024, 0) == 4
    # 9 tiles x 8 k-blocks: not split
    assert splits(AR, 2, 300, 520, 200, 0) == 0
    # decode: 96 swapped tiles of 16 tokens over 768 k-blocks fill the SMs over several waves
    assert splits(AR, 8, 16, 12288, 6144, 0) == 11
    try:
        assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 3) == tp.TP_OK
        assert splits(AR, 2, 300, 520, 200, 0) == 3
        assert splits(AR, 2, 128, 2048, 1024, 32) == 3
        # clamped to one k-block per split: 1 x [64, 64] per rank, p = 2
        assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 16) == tp.TP_OK
        assert splits(AR, 2, 64, 64, 64, 0) == 2
        # launches of a wave or more are not split
        assert tp.tp_workspace_size(AR, 2, 4864, 2048, 1024, 0, tp.TP_BF16) == 256
        assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 17) == tp.TP_ERR_INVALID_ARG
        assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, -1) == tp.TP_ERR_INVALID_ARG
    finally:
        tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 0)
    assert splits(AR, 2, 300, 520, 200, 0) == 0


def test_workspace_holds_the_last_wave_slices(tp):
    """bf16 outputs on CTA pairs: 4096 x 4096 is 256 pair tiles, 3 full waves
    of 76 clusters and 28 tiles cut into 2 k-slices: one fp32 256 x 256 tile
    per slice, after the 8-byte slice counters (one per tile, CTA and epilogue warp)."""
    bf = tp.tp_workspace_size(tp.TP_OP_ROW_AR, 4, 4096, 4096, 4096, 0, tp.TP_BF16)
    assert bf == 256 + 28 * 2 * 8 * 8 + 28 * 2 * 256 * 256 * 4
    # a whole number of waves (152 tiles) needs no slices
    assert tp.tp_workspace_size(tp.TP_OP_ROW_AR, 2, 4864, 2048, 1024, 0, tp.TP_BF16) == 256


def test_fp32_workspace_holds_the_precise_splits(tp):
    """fp32 outputs: no accumulator takes more than 2048 of the contraction.
    p = 4 ranks of K = 4096 (16384 in all) need 8 fp32 copies of Y; a
    contraction of 2048 or less needs none."""
    f32 = tp.tp_workspace_size(tp.TP_OP_ROW_AR, 4, 4096, 4096, 4096, 0, tp.TP_FP32)
    assert f32 == 256 + 8 * 4096 * 4096 * 4
    # (a short contraction plans as with bf16 outputs: CTA pairs with last-wave slices)
    assert tp.tp_workspace_size(tp.TP_OP_ROW_AR, 4, 4096, 4096, 512, 0, tp.TP_FP32) == \
        tp.tp_workspace_size(tp.TP_OP_ROW_AR, 4, 4096, 4096, 512, 0, tp.TP_BF16)
    # column backward with enough tiles to need no split for occupancy: dX
    # contracts over p * N = 8192 (4 splits), dW over M = 4096 (2 splits)
    cb = tp.tp_workspace_size(tp.TP_OP_COL_BWD, 4, 4096, 2048, 2048, 0, tp.TP_FP32)
    assert cb == 256 + max(4 * 4096 * 2048 * 4, 2 * 4 * 2048 * 2048 * 4)


# ---------------------------------------------------------------- host argument checks

A = 1 << 20          # fake, 16-byte aligned "device" addresses: never dereferenced
B = 1 << 30


def arr(*ptrs):
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


def row_ar(tp, x, w, y, n_out, p, M, N, K, chunk=0, dt=0, ws=B + (1 << 28), wsb=1 << 20, bias=None):
    return tp._lib.tp_row_linear_fwd_allreduce(x, w, bias, y, n_out, p, M, N, K, chunk, dt, ws, wsb, None)


def test_row_ar_argument_checks(tp):
    x = arr(A, A + 4096)
    w = arr(A + 8192, A + 12288)
    y = arr(A + (1 << 24))
    M, N, K = 16, 8, 8
    assert row_ar(tp, x, w, y, 1, 0, M, N, K) == tp.TP_ERR_INVALID_ARG          # p = 0
    assert row_ar(tp, x, w, y, 1, 9, M, N, K) == tp.TP_ERR_INVALID_ARG          # p > 8
    assert row_ar(tp, x, w, y, 1, 2, -1, N, K) == tp.TP_ERR_INVALID_ARG         # negative M
    assert row_ar(tp, x, w, y, 1, 2, M, 12, K) == tp.TP_ERR_ALIGNMENT           # N % 8
    assert row_ar(tp, x, w, y, 1, 2, M, N, 4) == tp.TP_ERR_ALIGNMENT            # K % 8
    assert row_ar(tp, x, w, y, 3, 2, M, N, K) == tp.TP_ERR_INVALID_ARG          # n_out not 1 or p
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, dt=5) == tp.TP_ERR_INVALID_ARG    # dtype
    assert row_ar(tp, arr(A, 0), w, y, 1, 2, M, N, K) == tp.TP_ERR_INVALID_ARG  # null shard
    assert row_ar(tp, arr(A, A + 3), w, y, 1, 2, M, N, K) == tp.TP_ERR_ALIGNMENT
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, ws=0) == tp.TP_ERR_INVALID_ARG
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, ws=B + 8) == tp.TP_ERR_ALIGNMENT
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, wsb=16) == tp.TP_ERR_WORKSPACE_TOO_SMALL
    # output overlapping an input shard
    assert row_ar(tp, x, w, arr(A + 4096 + 64), 1, 2, M, N, K) == tp.TP_ERR_INVALID_ARG
    # a misaligned bias, and a bias overlapping the output
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, bias=A + (1 << 22) + 2) == tp.TP_ERR_ALIGNMENT
    assert row_ar(tp, x, w, y, 1, 2, M, N, K, bias=A + (1 << 24) + 32) == tp.TP_ERR_INVALID_ARG
    # M == 0: nothing to do, accepted without touching the device
    assert row_ar(tp, x, w, y, 1, 2, 0, N, K) == tp.TP_OK


def test_rs_and_ag_need_m_divisible_by_p(tp):
    x = arr(A, A + 4096, A + 8192)
    w = arr(A + 65536, A + 69632, A + 73728)
    y = arr(B, B + 4096, B + 8192)
    st = tp._lib.tp_row_linear_fwd_reducescatter(x, w, None, y, 3, 16, 8, 8, 0, 0, B + (1 << 28), 1 << 20, None)
    assert st == tp.TP_ERR_UNSUPPORTED_SHAPE
    st = tp._lib.tp_ag_matmul(x, w, None, y, None, 0, None, 3, 16, 8, 8, 0, 0, B + (1 << 28), 1 << 20, None)
    assert st == tp.TP_ERR_UNSUPPORTED_SHAPE


def test_col_and_bwd_argument_checks(tp):
    w = arr(A, A + 4096)
    y = arr(B, B + 4096)
    ws = B + (1 << 28)
    # bad epilogue for the forward
    assert tp._lib.tp_col_linear_fwd(A + 65536, w, None, y, None, 2, 2, 16, 8, 8, 0, 0, ws, 1 << 20, None) \
        == tp.TP_ERR_INVALID_ARG
    # GeLU with a preact list holding a null pointer
    assert tp._lib.tp_col_linear_fwd(A + 65536, w, None, y, arr(B + 65536, 0), 1, 2, 16, 8, 8, 0, 0, ws,
                                     1 << 20, None) == tp.TP_ERR_INVALID_ARG
    # a bias list holding a null pointer
    assert tp._lib.tp_col_linear_fwd(A + 65536, w, arr(A + 98304, 0), y, None, 0, 2, 16, 8, 8, 0, 0, ws,
                                     1 << 20, None) == tp.TP_ERR_INVALID_ARG
    # column backward with no output at all
    assert tp._lib.tp_col_linear_bwd(A + 65536, w, arr(A + 131072, A + 135168), None, None, None, 2, 16, 8,
                                     8, 0, 0, ws, 1 << 20, None) == tp.TP_ERR_INVALID_ARG
    # row backward with no output at all
    assert tp._lib.tp_row_linear_bwd(None, w, A + 65536, None, None, None, None, 2, 16, 8, 8, 0, 0, ws,
                                     1 << 20, None) == tp.TP_ERR_INVALID_ARG
    # a bias gradient overlapping the output gradient it is summed from
    assert tp._lib.tp_row_linear_bwd(None, w, A + 65536, None, None, A + 65536 + 64, None, 2, 16, 8, 8, 0,
                                     0, ws, 1 << 20, None) == tp.TP_ERR_INVALID_ARG
    # status query needs a workspace
    assert tp._lib.tp_get_device_status(None, None) == tp.TP_ERR_INVALID_ARG
