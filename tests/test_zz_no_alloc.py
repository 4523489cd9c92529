"""The allocation-free row-parallel AllReduce entry point.

Some callers cannot allocate device memory: a host plugin interface that
hands over only input and output buffers, or an engine that has reserved all
of device memory for its own pool.  tp_row_linear_fwd_allreduce_noalloc
serves them from a static device array inside the library.  These tests call
it through the C-ABI, two calls in a row with different inputs each time (so
that stale scratch from the first call cannot leak into the second), and
check its output
  - against the CPU oracle: bit for bit on integer inputs (every fp32 partial
    sum exact; bf16 outputs equal the oracle rounded to bf16), within the
    parity tolerance on normal inputs;
  - against the workspace entry point, bit for bit: both plan the same
    launches for these shapes, and the kernels are deterministic.
The cases reach the split-K second stage (fp32 partials in the scratch), the
operand-swapped token tiles, single-CTA tiles and the CTA-pair kernel whose
last partial wave runs as k-slices (slice partials and launch-numbered
counters in the scratch).  The file runs last (its name) so that a failure
here never hides the other GPU tests.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import BF16_TOL, FP32_TOL, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import gemm_reduce_fusion_gb300 as tp
    return tp


# (p, M, N, K, chunk_m): a skinny split-K case (fp32 partials in the scratch),
# a 32-row-chunk case (the worked example's shape), a ragged 128x256-tile
# case, and an 80-tile CTA-pair case whose last wave of 4 tiles runs as
# k-slices (about 4 MiB of slice partials and counters in the scratch).
CASES = [(8, 16, 2048, 512, 16), (2, 128, 2048, 1024, 32), (4, 300, 520, 200, 0), (2, 2048, 2560, 1024, 0)]


def _inputs(kind, call, p, M, N, K):
    if kind == "int":
        xs = [synth.integer_bf16((M, K), synth.seed_for(44 + call, r), 4) for r in range(p)]
        ws = [synth.integer_bf16((K, N), synth.seed_for(44 + call, 8 + r), 4) for r in range(p)]
    else:
        xs = [synth.normal_bf16((M, K), synth.seed_for(40 + call, r), 1.0 / np.sqrt(K)) for r in range(p)]
        ws = [synth.normal_bf16((K, N), synth.seed_for(40 + call, 8 + r)) for r in range(p)]
    return xs, ws


@pytest.mark.parametrize("kind", ["int", "normal"])
@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("p,M,N,K,chunk", CASES)
def test_noalloc_matches_oracle_and_workspace_entry_point(tp, p, M, N, K, chunk, f32, kind):
    import torch
    dt = torch.float32 if f32 else torch.bfloat16
    wsp = tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk, out_dtype=tp.TP_FP32 if f32 else tp.TP_BF16)
    for call in range(2):
        xs, ws = _inputs(kind, call, p, M, N, K)
        X, W = [dev(a) for a in xs], [dev(b) for b in ws]
        got = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        tp.tp_row_linear_fwd_allreduce_noalloc(X, W, [got], chunk)
        assert tp.tp_noalloc_device_status() == tp.TP_OK
        want = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        tp.tp_row_linear_fwd_allreduce(X, W, [want], wsp, chunk)
        assert tp.tp_get_device_status(wsp) == tp.TP_OK
        assert torch.equal(got.view(torch.int32 if f32 else torch.int16),
                           want.view(torch.int32 if f32 else torch.int16)), f"call {call}: differs from workspace call"
        ref = oracle.row_fwd_allreduce(xs, ws)
        if kind == "int":
            exp = ref if f32 else oracle.widen(oracle.round_bf16(ref))
            assert np.array_equal(host_f64(got), exp), f"call {call}: not exact"
        else:
            e = rel_err(host_f64(got), ref)
            assert e <= (FP32_TOL if f32 else BF16_TOL), f"call {call}: rel err {e:.3e}"


def test_noalloc_rejects_calls_beyond_its_scratch(tp):
    """A call whose plan needs more than the static scratch is refused on the
    host, before any pointer is looked at: every tensor pointer here is NULL,
    so a check that ever moved behind the pointer checks would return
    TP_ERR_INVALID_ARG instead, and nothing can reach the GPU either way."""
    import ctypes
    p, M, N, K, chunk = 8, 640, 5120, 8192, 640   # 100 tiles: split-K partials of ~39 MB
    need = tp.tp_workspace_size(tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    assert need > (16 << 20)
    fn = tp._lib.tp_row_linear_fwd_allreduce_noalloc
    fn.restype = ctypes.c_int
    nulls = (ctypes.c_void_p * p)(*([None] * p))
    y = (ctypes.c_void_p * 1)(None)
    st = fn(nulls, nulls, y, 1, p, ctypes.c_int64(M), ctypes.c_int64(N), ctypes.c_int64(K), ctypes.c_int64(chunk),
            0, None)
    assert st == tp.TP_ERR_WORKSPACE_TOO_SMALL
    # within the limit, the same NULL pointers are refused by the pointer checks
    st = fn(nulls, nulls, y, 1, 2, ctypes.c_int64(128), ctypes.c_int64(256), ctypes.c_int64(256),
            ctypes.c_int64(0), 0, None)
    assert st == tp.TP_ERR_INVALID_ARG


def test_noalloc_timeout_is_reported_then_next_call_is_exact(tp):
    """A device wait that runs out of time inside a no-alloc call is latched in
    the static scratch's status word and read (and cleared) by
    tp_noalloc_device_status; the next call is exact.  The wait is made to run
    out by the library's test hook (one k-block left unarmed, 200 ms limit)."""
    import torch
    p, M, N, K = 2, 2048, 2560, 1024
    xs, ws = _inputs("int", 0, p, M, N, K)
    X, W = [dev(a) for a in xs], [dev(b) for b in ws]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert tp.tp_noalloc_device_status() == tp.TP_OK
    assert tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 200) == tp.TP_OK
    assert tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, 3) == tp.TP_OK
    try:
        tp.tp_row_linear_fwd_allreduce_noalloc(X, W, [y])
        st = tp.tp_noalloc_device_status()
    finally:
        tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, -1)
        tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 0)
    assert st == tp.TP_ERR_DEVICE_TIMEOUT
    assert tp.tp_noalloc_device_status() == tp.TP_OK
    tp.tp_row_linear_fwd_allreduce_noalloc(X, W, [y])
    assert tp.tp_noalloc_device_status() == tp.TP_OK
    assert np.array_equal(host_f64(y), oracle.row_fwd_allreduce(xs, ws))
