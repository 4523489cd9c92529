"""Failure detection on the GPU without a fault: a device-side wait that runs
out of time is latched in the workspace status word, the kernel stops its
other roles and drains its own copies and MMAs before returning, and the
context stays usable for the next call.

The wait is made to run out through the library's test hook: CTA 0 leaves
one k-block of its ring unarmed (nothing ever signals it), with a 200 ms
limit on every wait."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_close, dev, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import gemm_reduce_fusion_gb300 as tp
    return tp


@pytest.mark.parametrize("chunk", [0, 32])
def test_timeout_latched_then_next_call_succeeds(tp, chunk):
    import time
    import torch
    p, M, N, K = 2, 512, 512, 512
    xs = [synth.normal_bf16((M, K), synth.seed_for(70, r), 1.0 / np.sqrt(K)) for r in range(p)]
    ws = [synth.normal_bf16((K, N), synth.seed_for(71, r)) for r in range(p)]
    X, W = [dev(a) for a in xs], [dev(b) for b in ws]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    wsp = tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    assert tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 200) == tp.TP_OK
    assert tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, 3) == tp.TP_OK
    try:
        t0 = time.time()
        tp.tp_row_linear_fwd_allreduce(X, W, [y], wsp, chunk)
        st = tp.tp_get_device_status(wsp)
        elapsed = time.time() - t0
    finally:
        tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, -1)
        tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 0)
    assert st == tp.TP_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    # status was cleared by the read; the context is healthy
    assert tp.tp_get_device_status(wsp) == tp.TP_OK
    tp.tp_row_linear_fwd_allreduce(X, W, [y], wsp, chunk)
    assert tp.tp_get_device_status(wsp) == tp.TP_OK
    assert_close(host_f64(y), oracle.row_fwd_allreduce(xs, ws), False, "after recovery")


@pytest.mark.parametrize("shape,tile_mode", [((2, 512, 512, 512), 2), ((2, 2048, 2560, 1024), 0)])
def test_timeout_on_cta_pairs_then_next_call_succeeds(tp, shape, tile_mode):
    """The same on the CTA-pair kernel: CTA 0 of the first cluster leaves a
    k-block unarmed, its peer's waits run out too, both meet at the cluster
    barrier and free their tensor memory.  The second shape also runs its
    last wave as k-slices: the stopped launch leaves some slice counters
    part-way, and the next launch on the same workspace must read them as
    zero (they carry the stopped launch's number) and be exact."""
    import time
    import torch
    p, M, N, K = shape
    xs = [synth.integer_bf16((M, K), synth.seed_for(72, r), 4) for r in range(p)]
    ws = [synth.integer_bf16((K, N), synth.seed_for(73, r), 4) for r in range(p)]
    X, W = [dev(a) for a in xs], [dev(b) for b in ws]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    wsp = tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, 0)
    assert tp.tp_debug_set(tp.TP_DEBUG_TILE_MODE, tile_mode) == tp.TP_OK
    assert tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 200) == tp.TP_OK
    assert tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, 3) == tp.TP_OK
    try:
        t0 = time.time()
        tp.tp_row_linear_fwd_allreduce(X, W, [y], wsp)
        st = tp.tp_get_device_status(wsp)
        elapsed = time.time() - t0
        tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, -1)
        tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 0)
        assert st == tp.TP_ERR_DEVICE_TIMEOUT
        assert elapsed < 10.0
        assert tp.tp_get_device_status(wsp) == tp.TP_OK
        tp.tp_row_linear_fwd_allreduce(X, W, [y], wsp)
        assert tp.tp_get_device_status(wsp) == tp.TP_OK
    finally:
        tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, -1)
        tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, 0)
        tp.tp_debug_set(tp.TP_DEBUG_TILE_MODE, 0)
    assert np.array_equal(host_f64(y), oracle.row_fwd_allreduce(xs, ws))


def test_debug_hook_argument_checks(tp):
    assert tp.tp_debug_set(9, 0) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_K_ALTERNATE, 2) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_NO_BWD_FUSION, 2) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_TMA_STORE, 2) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_L2_HINTS, -1) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_TIMEOUT_MS, -5) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_DROP_LOAD, -2) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_NO_TAIL_SLICES, 2) == tp.TP_ERR_INVALID_ARG
    assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 17) == tp.TP_ERR_INVALID_ARG
