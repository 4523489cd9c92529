"""The allocation-free row-parallel AllReduce entry point.

Some callers cannot allocate device memory: a host plugin interface that
hands over only input and output buffers, or an engine that has reserved all
of device memory for its own pool.  tp_row_linear_fwd_allreduce_noalloc
serves them from a static device array inside the library.  This test calls
it through the C-ABI and checks, on two calls in a row with different
inputs (so stale scratch from the first call cannot leak into the second),
that its output matches the workspace entry point's within the tolerance
the parity tests use.  It runs last (file name) so that a failure here never
hides the other GPU tests.
"""
import numpy as np
import pytest

import synth
from gpu_util import BF16_TOL, FP32_TOL, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    import gemm_reduce_fusion_gb300 as tp
    return tp


# (p, M, N, K, chunk_m): a split-K skinny case that uses the scratch for
# fp32 partials, a 32-row-chunk case, and a 128x256-tile case.
CASES = [(8, 16, 2048, 512, 16), (2, 128, 2048, 1024, 32), (4, 300, 520, 200, 0)]


@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("p,M,N,K,chunk", CASES)
def test_noalloc_matches_workspace_entry_point(tp, p, M, N, K, chunk, f32):
    import torch
    dt = torch.float32 if f32 else torch.bfloat16
    tol = FP32_TOL if f32 else BF16_TOL
    for call in range(2):
        xs = [dev(synth.normal_bf16((M, K), synth.seed_for(40 + call, r), 1.0 / np.sqrt(K))) for r in range(p)]
        ws = [dev(synth.normal_bf16((K, N), synth.seed_for(40 + call, 8 + r))) for r in range(p)]
        want = torch.empty((M, N), dtype=dt, device="cuda")
        tp.tp_row_linear_fwd_allreduce(xs, ws, [want], tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk), chunk)
        got = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        tp.tp_row_linear_fwd_allreduce_noalloc(xs, ws, [got], chunk)
        torch.cuda.synchronize()
        e = rel_err(host_f64(got), host_f64(want))
        assert e <= tol, f"call {call}: rel err {e:.3e}"


def test_noalloc_rejects_calls_beyond_its_scratch(tp):
    import ctypes
    p, M, N, K, chunk = 8, 640, 5120, 8192, 640   # 100 tiles: split-K partials of ~39 MB
    need = tp.tp_workspace_size(tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    assert need > (16 << 20)
    fn = tp._lib.tp_row_linear_fwd_allreduce_noalloc
    fn.restype = ctypes.c_int
    A = 1 << 20
    arr = (ctypes.c_void_p * p)(*[A + 4096 * i for i in range(p)])
    y = (ctypes.c_void_p * 1)(1 << 30)
    st = fn(arr, arr, y, 1, p, ctypes.c_int64(M), ctypes.c_int64(N), ctypes.c_int64(K), ctypes.c_int64(chunk),
            0, None)
    assert st == tp.TP_ERR_WORKSPACE_TOO_SMALL
