"""Python binding of the tp_fused C-ABI (argument marshalling only).

Every function here has the name of the C entry point it calls
(``include/tp_fused.h``).  It reads shapes from the torch tensors it is
given and checks that every shard, output and bias has the shape, dtype,
layout and device the call implies (the C ABI sees only pointers, so a
wrong-sized buffer would otherwise be read or written out of bounds on the
device); it then passes the device pointers and the current CUDA stream to
the shared library and raises :class:`TPError` on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback: if the
library is missing the import fails.

Tensors are torch CUDA tensors, contiguous, row-major; inputs bfloat16,
outputs bfloat16 or float32.  Lists hold one tensor per rank/shard.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtpfused.so")

# tp_status
TP_OK = 0
TP_ERR_INVALID_ARG = 1
TP_ERR_ALIGNMENT = 2
TP_ERR_UNSUPPORTED_SHAPE = 3
TP_ERR_WORKSPACE_TOO_SMALL = 4
TP_ERR_ARCH = 5
TP_ERR_CUDA = 6
TP_ERR_DEVICE_TIMEOUT = 7
# tp_dtype
TP_BF16 = 0
TP_FP32 = 1
# tp_epilogue
TP_EPI_NONE = 0
TP_EPI_GELU = 1
TP_EPI_DGELU = 2
# tp_op
TP_OP_ROW_AR = 0
TP_OP_ROW_RS = 1
TP_OP_COL_FWD = 2
TP_OP_COL_BWD = 3
TP_OP_ROW_BWD = 4
TP_OP_AG_MM = 5
TP_OP_ROW_AR_UNFUSED = 6
TP_OP_AG_MM_BWD = 7
TP_OP_ROW_RS_BWD = 8
# tp_debug_key
TP_DEBUG_TIMEOUT_MS = 0
TP_DEBUG_DROP_LOAD = 1
TP_DEBUG_TILE_MODE = 2
TP_DEBUG_NO_TAIL_SLICES = 3
TP_DEBUG_SPLIT_K = 4
TP_DEBUG_L2_HINTS = 5
TP_DEBUG_TMA_STORE = 6
TP_DEBUG_NO_BWD_FUSION = 7
TP_DEBUG_K_ALTERNATE = 8
# tp_row_linear_fwd_unfused flags
TP_UNFUSED_BF16_COLLECTIVE = 1


class TPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tp_status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python gemm_reduce_fusion_gb300/build.py` "
            "(nvcc, sm_103a); there is no non-CUDA fallback")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    PP = ctypes.POINTER(ctypes.c_void_p)
    I = ctypes.c_int
    L = ctypes.c_int64
    S = ctypes.c_size_t
    sig = {
        "tp_workspace_size": (S, [I, I, L, L, L, L, I]),
        "tp_row_linear_fwd_allreduce": (I, [PP, PP, P, PP, I, I, L, L, L, L, I, P, S, P]),
        "tp_row_linear_fwd_reducescatter": (I, [PP, PP, P, PP, I, L, L, L, L, I, P, S, P]),
        "tp_col_linear_fwd": (I, [P, PP, PP, PP, PP, I, I, L, L, L, L, I, P, S, P]),
        "tp_col_linear_bwd": (I, [P, PP, PP, P, PP, PP, I, L, L, L, L, I, P, S, P]),
        "tp_row_linear_bwd": (I, [PP, PP, P, PP, PP, P, PP, I, L, L, L, L, I, P, S, P]),
        "tp_ag_matmul": (I, [PP, PP, PP, PP, P, I, PP, I, L, L, L, L, I, P, S, P]),
        "tp_row_linear_fwd_unfused": (I, [PP, PP, P, I, L, L, L, L, I, I, I, P, S, P]),
        "tp_ag_matmul_bwd": (I, [PP, PP, PP, PP, PP, PP, I, L, L, L, L, I, P, S, P]),
        "tp_row_linear_bwd_reducescatter": (I, [PP, PP, PP, PP, PP, P, PP, I, L, L, L, L, I, P, S, P]),
        "tp_pipeline_time": (ctypes.c_double, [ctypes.c_double, ctypes.c_double, L]),
        "tp_num_chunks": (L, [L, L]),
        "tp_choose_chunk_m": (L, [I, I, L, L, L]),
        "tp_choose_chunk_m_measured": (L, [L, ctypes.POINTER(L), ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_double), I]),
        "tp_get_device_status": (I, [P, P]),
        "tp_status_string": (ctypes.c_char_p, [I]),
        "tp_debug_set": (I, [I, L]),
        "tp_trace_set": (I, [P, L]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


# ------------------------------------------------------------------ marshalling

def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous (row-major)")
    return t.data_ptr()


def _arr(ts) -> ctypes.Array | None:
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[_ptr(t) for t in ts])


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return TP_BF16
    if t.dtype == torch.float32:
        return TP_FP32
    raise ValueError(f"unsupported output dtype {t.dtype}")


def _out_dtype(*groups) -> int:
    """The single output dtype of a call: every output tensor must share it."""
    codes = {_dtype_code(t) for g in groups if g is not None
             for t in (g if isinstance(g, (list, tuple)) else [g])}
    if len(codes) != 1:
        raise ValueError("all outputs of one call must have the same dtype (bfloat16 or float32)")
    return codes.pop()


def _ws(ws):
    return _ptr(ws), ws.numel() * ws.element_size()


def _check(status: int, where: str) -> None:
    if status != TP_OK:
        raise TPError(status, where)


# ------------------------------------------------------------------ argument checks
#
# The C ABI takes one M, N, K for all shards and plain pointers: it cannot see
# how large a buffer is, so a shard of the wrong shape would be read or
# written out of bounds on the device.  The binding knows every tensor's
# shape and checks them on the host before anything is enqueued: shape,
# bfloat16 for inputs, row-major layout, and the calling thread's current
# CUDA device (the device the library runs the call on).  None stands for a
# NULL pointer; the library decides where NULL is allowed.

def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def _need(where: str, name: str, t, shape, bf16: bool, dev: int) -> None:
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{where}: {name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if bf16:
        import torch
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{where}: {name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{where}: {name} must be contiguous (row-major)")
    if t.get_device() != dev:
        raise TypeError(f"{where}: {name} is on {t.device}; the call runs on cuda:{dev}, "
                        "the calling thread's current device")


def _need_all(where: str, name: str, ts, counts, shape, bf16: bool, dev: int) -> None:
    if ts is None:
        return
    if len(ts) not in counts:
        raise ValueError(f"{where}: {name} holds {len(ts)} tensors, expected "
                         + " or ".join(str(c) for c in counts))
    for i, t in enumerate(ts):
        _need(where, f"{name}[{i}]", t, shape, bf16, dev)


def _need_ws(where: str, ws, dev: int) -> None:
    if ws.get_device() != dev:
        raise TypeError(f"{where}: the workspace is on {ws.device}; the call runs on cuda:{dev}")


# ------------------------------------------------------------------ host-only calls

def tp_status_string(status: int) -> str:
    return _lib.tp_status_string(int(status)).decode()


def tp_workspace_size(op: int, p: int, M: int, N: int, K: int, chunk_m: int = 0,
                      out_dtype: int = TP_BF16) -> int:
    return int(_lib.tp_workspace_size(op, p, M, N, K, chunk_m, out_dtype))


def tp_pipeline_time(c: float, m: float, n_chunks: int) -> float:
    return float(_lib.tp_pipeline_time(c, m, n_chunks))


def tp_num_chunks(M: int, chunk_m: int) -> int:
    return int(_lib.tp_num_chunks(M, chunk_m))


def tp_choose_chunk_m(op: int, p: int, M: int, N: int, K: int) -> int:
    return int(_lib.tp_choose_chunk_m(op, p, M, N, K))


def tp_choose_chunk_m_measured(M: int, chunks: Sequence[int], c: Sequence[float], m: Sequence[float]) -> int:
    """The candidate chunk_m whose timeline from measured per-chunk c and m is shortest."""
    n = len(chunks)
    if not (len(c) == len(m) == n):
        raise ValueError("one c and one m per candidate chunk")
    return int(_lib.tp_choose_chunk_m_measured(M, (ctypes.c_int64 * n)(*chunks), (ctypes.c_double * n)(*c),
                                               (ctypes.c_double * n)(*m), n))


def workspace(op: int, p: int, M: int, N: int, K: int, chunk_m: int = 0, device="cuda",
              out_dtype: int = TP_BF16):
    """A zero-filled device workspace of tp_workspace_size(...) bytes (torch-allocated)."""
    import torch
    n = tp_workspace_size(op, p, M, N, K, chunk_m, out_dtype)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def tp_trace_set(buf, cap_units: int = 0) -> None:
    """Trace the GEMM launches that follow into ``buf`` (a zeroed CUDA
    int64 tensor of cap_units x 4), or stop tracing with ``buf=None``."""
    _check(_lib.tp_trace_set(_ptr(buf), cap_units if buf is not None else 0), "tp_trace_set")


def tp_debug_set(key: int, value: int) -> int:
    """Test hook of the failure-detection path (see tp_fused.h)."""
    return int(_lib.tp_debug_set(key, value))


def tp_get_device_status(ws, stream=None) -> int:
    """Latched device status of ``ws`` (synchronises the stream, clears it)."""
    return int(_lib.tp_get_device_status(_ptr(ws), _stream(stream)))


# ------------------------------------------------------------------ the sharded Linear

def tp_row_linear_fwd_allreduce(x: Sequence, w: Sequence, y: Sequence, ws, chunk_m: int = 0,
                                stream=None, bias=None) -> None:
    """Y = sum_r X_r W_r (+ bias) written once (len(y) == 1) or as p replicas (len(y) == p)."""
    p = len(x)
    M, K = x[0].shape
    N = w[0].shape[1]
    W, dev = "tp_row_linear_fwd_allreduce", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "y", y, (1, p), (M, N), False, dev)
    _need(W, "bias", bias, (N,), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_row_linear_fwd_allreduce(_arr(x), _arr(w), _ptr(bias), _arr(y), len(y), p, M, N, K, chunk_m,
                                            _dtype_code(y[0]), wp, wb, _stream(stream)),
           "tp_row_linear_fwd_allreduce")


def tp_row_linear_fwd_reducescatter(x: Sequence, w: Sequence, y: Sequence, ws, chunk_m: int = 0,
                                    stream=None, bias=None) -> None:
    """Rank j's y[j] = rows [j M/p, (j+1) M/p) of sum_r X_r W_r (+ bias)."""
    p = len(x)
    M, K = x[0].shape
    N = w[0].shape[1]
    W, dev = "tp_row_linear_fwd_reducescatter", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "y", y, (p,), (M // p, N), False, dev)
    _need(W, "bias", bias, (N,), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_row_linear_fwd_reducescatter(_arr(x), _arr(w), _ptr(bias), _arr(y), p, M, N, K, chunk_m,
                                                _dtype_code(y[0]), wp, wb, _stream(stream)),
           "tp_row_linear_fwd_reducescatter")


def tp_col_linear_fwd(x, w: Sequence, y: Sequence, ws, epi: int = TP_EPI_NONE, preact=None,
                      chunk_m: int = 0, stream=None, bias=None) -> None:
    """y[k] = X A_k + b_k (or GeLU of it, with H_k into preact[k]); bias[k] = b_k or bias None."""
    p = len(w)
    M, K = x.shape
    N = w[0].shape[1]
    W, dev = "tp_col_linear_fwd", _current_device()
    _need(W, "x", x, (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "y", y, (p,), (M, N), False, dev)
    _need_all(W, "preact", preact, (p,), (M, N), False, dev)
    _need_all(W, "bias", bias, (p,), (N,), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_col_linear_fwd(_ptr(x), _arr(w), _arr(bias), _arr(y), _arr(preact), epi, p, M, N, K, chunk_m,
                                  _out_dtype(y, preact), wp, wb, _stream(stream)), "tp_col_linear_fwd")


def tp_col_linear_bwd(x, w: Sequence, dy: Sequence, dx, dw, ws, chunk_m: int = 0,
                      stream=None, db=None) -> None:
    """dX = sum_k dY_k A_k^T; dw[k] = X^T dY_k; db[k] = row sum of dY_k (dx, dw, db may be None)."""
    p = len(w)
    K, N = w[0].shape
    M = dy[0].shape[0]
    W, dev = "tp_col_linear_bwd", _current_device()
    _need(W, "x", x, (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "dy", dy, (p,), (M, N), True, dev)
    _need(W, "dx", dx, (M, K), False, dev)
    _need_all(W, "dw", dw, (p,), (K, N), False, dev)
    _need_all(W, "db", db, (p,), (N,), False, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_col_linear_bwd(_ptr(x), _arr(w), _arr(dy), _ptr(dx), _arr(dw), _arr(db), p, M, N, K,
                                  chunk_m, _out_dtype(dx, dw, db), wp, wb, _stream(stream)), "tp_col_linear_bwd")


def tp_row_linear_bwd(x, w: Sequence, dy, dx, dw, ws, preact=None, chunk_m: int = 0,
                      stream=None, db=None) -> None:
    """dx[k] = dY A_k^T (times GeLU'(preact[k])); dw[k] = X_k^T dY; db = row sum of dY."""
    p = len(w)
    K, N = w[0].shape
    M = dy.shape[0]
    W, dev = "tp_row_linear_bwd", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need(W, "dy", dy, (M, N), True, dev)
    _need_all(W, "dx", dx, (p,), (M, K), False, dev)
    _need_all(W, "dw", dw, (p,), (K, N), False, dev)
    _need(W, "db", db, (N,), False, dev)
    _need_all(W, "preact", preact, (p,), (M, K), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_row_linear_bwd(_arr(x), _arr(w), _ptr(dy), _arr(dx), _arr(dw), _ptr(db), _arr(preact), p,
                                  M, N, K, chunk_m, _out_dtype(dx, dw, db), wp, wb, _stream(stream)),
           "tp_row_linear_bwd")


def tp_ag_matmul(x: Sequence, w: Sequence, y: Sequence, ws, x_gathered=None,
                 epi: int = TP_EPI_NONE, preact=None, chunk_m: int = 0, stream=None, bias=None) -> None:
    """y[k] = [X_0; ...; X_{p-1}] A_k + b_k (optionally GeLU, H_k, gathered X)."""
    p = len(x)
    Mp, K = x[0].shape
    N = w[0].shape[1]
    W, dev = "tp_ag_matmul", _current_device()
    _need_all(W, "x", x, (p,), (Mp, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "y", y, (p,), (Mp * p, N), False, dev)
    _need(W, "x_gathered", x_gathered, (Mp * p, K), True, dev)
    _need_all(W, "preact", preact, (p,), (Mp * p, N), False, dev)
    _need_all(W, "bias", bias, (p,), (N,), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_ag_matmul(_arr(x), _arr(w), _arr(bias), _arr(y), _ptr(x_gathered), epi, _arr(preact), p,
                             Mp * p, N, K, chunk_m, _out_dtype(y, preact), wp, wb, _stream(stream)),
           "tp_ag_matmul")


def tp_ag_matmul_bwd(x, w: Sequence, dy: Sequence, dx, dw, ws, chunk_m: int = 0, stream=None,
                     db=None) -> None:
    """dx[s] = rows of sum_k dY_k A_k^T (ReduceScatter); dw[k] = [X_0;...]^T dY_k; db[k] = row sum of dY_k."""
    p = len(w)
    K, N = w[0].shape
    M = dy[0].shape[0]
    W, dev = "tp_ag_matmul_bwd", _current_device()
    _need_all(W, "x", x, (p,), (M // p, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "dy", dy, (p,), (M, N), True, dev)
    _need_all(W, "dx", dx, (p,), (M // p, K), False, dev)
    _need_all(W, "dw", dw, (p,), (K, N), False, dev)
    _need_all(W, "db", db, (p,), (N,), False, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_ag_matmul_bwd(_arr(x), _arr(w), _arr(dy), _arr(dx), _arr(dw), _arr(db), p, M, N, K, chunk_m,
                                 _out_dtype(dx, dw, db), wp, wb, _stream(stream)), "tp_ag_matmul_bwd")


def tp_row_linear_bwd_reducescatter(x, w: Sequence, dy: Sequence, dx, dw, ws, preact=None, chunk_m: int = 0,
                                    stream=None, db=None) -> None:
    """dx[r] = [dY_0;...] A_r^T (* GeLU'(preact[r])) (AllGather); dw[r] = X_r^T [dY_0;...];
    db = row sum of all the dY shards."""
    p = len(w)
    K, N = w[0].shape
    M = dy[0].shape[0] * p
    W, dev = "tp_row_linear_bwd_reducescatter", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "dy", dy, (p,), (M // p, N), True, dev)
    _need_all(W, "dx", dx, (p,), (M, K), False, dev)
    _need_all(W, "dw", dw, (p,), (K, N), False, dev)
    _need(W, "db", db, (N,), False, dev)
    _need_all(W, "preact", preact, (p,), (M, K), True, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_row_linear_bwd_reducescatter(_arr(x), _arr(w), _arr(dy), _arr(dx), _arr(dw), _ptr(db),
                                                _arr(preact), p, M, N, K, chunk_m, _out_dtype(dx, dw, db), wp, wb,
                                                _stream(stream)), "tp_row_linear_bwd_reducescatter")


def tp_row_linear_fwd_unfused(x: Sequence, w: Sequence, y, ws, chunk_m: int = 0, phases: int = 3,
                              flags: int = 0, stream=None) -> None:
    """Unfused baseline: per-rank fp32 partials (phase 1), rank-order reduce into y (phase 2);
    flags=TP_UNFUSED_BF16_COLLECTIVE sums bf16-rounded partials with a bf16 running sum."""
    p = len(x)
    M, K = x[0].shape
    N = w[0].shape[1]
    W, dev = "tp_row_linear_fwd_unfused", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need(W, "y", y, (M, N), False, dev)
    _need_ws(W, ws, dev)
    wp, wb = _ws(ws)
    _check(_lib.tp_row_linear_fwd_unfused(_arr(x), _arr(w), _ptr(y), p, M, N, K, chunk_m, _dtype_code(y),
                                          phases, flags, wp, wb, _stream(stream)), "tp_row_linear_fwd_unfused")


def tp_row_linear_fwd_allreduce_noalloc(x: Sequence, w: Sequence, y: Sequence, chunk_m: int = 0,
                                        stream=None) -> None:
    """tp_row_linear_fwd_allreduce without a workspace: for callers that
    cannot allocate device memory (the library uses its static scratch)."""
    fn = _lib.tp_row_linear_fwd_allreduce_noalloc
    fn.restype = ctypes.c_int
    PP = ctypes.POINTER(ctypes.c_void_p)
    L = ctypes.c_int64
    fn.argtypes = [PP, PP, PP, ctypes.c_int, ctypes.c_int, L, L, L, L, ctypes.c_int, ctypes.c_void_p]
    p = len(x)
    M, K = x[0].shape
    N = w[0].shape[1]
    W, dev = "tp_row_linear_fwd_allreduce_noalloc", _current_device()
    _need_all(W, "x", x, (p,), (M, K), True, dev)
    _need_all(W, "w", w, (p,), (K, N), True, dev)
    _need_all(W, "y", y, (1, p), (M, N), False, dev)
    _check(fn(_arr(x), _arr(w), _arr(y), len(y), p, M, N, K, chunk_m, _dtype_code(y[0]), _stream(stream)),
           "tp_row_linear_fwd_allreduce_noalloc")


def tp_noalloc_device_status(stream=None) -> int:
    """Read and clear the status word of the allocation-free entry point's
    static scratch (synchronises the stream): TP_OK or TP_ERR_DEVICE_TIMEOUT."""
    fn = _lib.tp_noalloc_device_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p]
    return fn(_stream(stream))
