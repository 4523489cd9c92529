"""PyTorch autograd wrappers over the sharded-Linear C-ABI.

The TP tutorial (§6.3, the autograd view of the duality) pairs the two
layouts with two communication regions:

* the column-parallel Linear copies its input to every rank in the forward
  pass (identity) and all-reduces the input gradient in the backward pass;
* the row-parallel Linear all-reduces the partial outputs in the forward
  pass and passes the output gradient through unchanged in the backward
  pass (each rank's dX_k is already its own shard).

Here all p ranks live in one GPU's memory and every reduction is fused into
the GEMM that produces it, so each layer is one ``torch.autograd.Function``
whose forward and backward are single library calls:

==========================  ===================================  ==========================================
Function                    forward                              backward
==========================  ===================================  ==========================================
column (copy region)        tp_col_linear_fwd                    tp_col_linear_bwd (fused dX reduce, dA_k)
row (reduce region)         tp_row_linear_fwd_allreduce          tp_row_linear_bwd (no reduction)
MLP block (§7.1)            column + GeLU, then row + AllReduce  row bwd with GeLU' epilogue, column bwd
sequence-parallel column    tp_ag_matmul (AllGather+MatMul)      tp_ag_matmul_bwd (ReduceScatter of dX)
sequence-parallel row       tp_row_linear_fwd_reducescatter      tp_row_linear_bwd_reducescatter (AllGather)
sequence-parallel MLP       AG+MatMul+GeLU, row + ReduceScatter  both sequence-parallel backwards
==========================  ===================================  ==========================================

GeLU exists only inside the MLP functions: its derivative is applied in the
epilogue of FC2's backward GEMM, so no separate elementwise kernel is
needed.  Biases are optional: a column layer adds rank k's block b_k before
the activation, a row layer adds its b once after the reduction (TP §三/§四),
and their gradients are the row sums of the output gradient, computed by
the backward call.  Tensors are bf16 CUDA tensors; weights are ``[in, out]``
row-major shards (rank k's column block for column layers, row block for
row layers).  Gradients are produced in bf16.  Nothing here computes: every
arithmetic step runs in the library's kernels.
"""
from __future__ import annotations

from typing import Sequence

import torch

from . import (TP_EPI_GELU, TP_OP_AG_MM, TP_OP_AG_MM_BWD, TP_OP_COL_BWD, TP_OP_COL_FWD, TP_OP_ROW_AR,
               TP_OP_ROW_BWD, TP_OP_ROW_RS, TP_OP_ROW_RS_BWD, tp_ag_matmul, tp_ag_matmul_bwd,
               tp_col_linear_bwd, tp_col_linear_fwd, tp_row_linear_bwd, tp_row_linear_bwd_reducescatter,
               tp_row_linear_fwd_allreduce, tp_row_linear_fwd_reducescatter, tp_workspace_size)

_WS: dict[int, torch.Tensor] = {}


def _workspace(device: torch.device, calls) -> torch.Tensor:
    """The device's shared workspace, grown (zero-filled) to fit every call
    in ``calls`` (tuples of tp_workspace_size arguments).  Calls that share
    it are ordered on the current stream."""
    need = max(tp_workspace_size(*c) for c in calls)
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _WS.get(idx)
    if ws is None or ws.numel() < need:
        ws = torch.zeros((need + 255) // 256 * 256, dtype=torch.uint8, device=device)
        _WS[idx] = ws
    return ws


def _bf16(t: torch.Tensor, what: str) -> torch.Tensor:
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{what}: expected a bfloat16 CUDA tensor, got {t.dtype} on {t.device}")
    return t if t.is_contiguous() else t.contiguous()


def _grad(g, like: torch.Tensor) -> torch.Tensor:
    """An output gradient as a contiguous bf16 tensor (zeros when autograd passes None)."""
    if g is None:
        return torch.zeros_like(like)
    return _bf16(g, "output gradient")


def _empty(shape, like):
    return torch.empty(shape, dtype=torch.bfloat16, device=like.device)


# ------------------------------------------------------------------ column parallel (copy region)

def _opt(ts):
    """A list of optional tensors -> None when absent, else bf16 contiguous."""
    if not ts or ts[0] is None:
        return None
    return [_bf16(t, "bias") for t in ts]


class _ColumnFn(torch.autograd.Function):
    """Y_k = X A_k + b_k for k < p.  Backward: dX = sum_k dY_k A_k^T (fused
    reduce), dA_k = X^T dY_k, db_k = row sum of dY_k."""

    @staticmethod
    def forward(ctx, p, x, *wb):
        x = _bf16(x, "x")
        w = [_bf16(a, "weight shard") for a in wb[:p]]
        b = _opt(wb[p:])
        (M, K), N = x.shape, w[0].shape[1]
        ws = _workspace(x.device, [(TP_OP_COL_FWD, p, M, N, K, 0), (TP_OP_COL_BWD, p, M, N, K, 0)])
        y = [_empty((M, N), x) for _ in range(p)]
        tp_col_linear_fwd(x, w, y, ws, bias=b)
        ctx.p = p
        ctx.save_for_backward(x, *w)
        return tuple(y)

    @staticmethod
    def backward(ctx, *dy):
        p = ctx.p
        x, *w = ctx.saved_tensors
        (M, K), N = x.shape, w[0].shape[1]
        dy = [_grad(g, x.new_empty((M, N))) for g in dy]
        need_x = ctx.needs_input_grad[1]
        need_w = any(ctx.needs_input_grad[2:2 + p])
        need_b = any(ctx.needs_input_grad[2 + p:])
        dx = _empty((M, K), x) if need_x else None
        dw = [_empty((K, N), x) for _ in range(p)] if need_w else None
        db = [_empty((N,), x) for _ in range(p)] if need_b else None
        if need_x or need_w or need_b:
            ws = _workspace(x.device, [(TP_OP_COL_BWD, p, M, N, K, 0)])
            tp_col_linear_bwd(x, w, dy, dx, dw, ws, db=db)
        return (None, dx, *(dw or [None] * p), *(db or [None] * p))


# ------------------------------------------------------------------ row parallel (reduce region)

class _RowFn(torch.autograd.Function):
    """Y = sum_r X_r A_r + b (fused AllReduce, b once).  Backward: dX_r = dY A_r^T,
    dA_r = X_r^T dY (no reduction), db = row sum of dY."""

    @staticmethod
    def forward(ctx, p, bias, *xw):
        x = [_bf16(a, "input shard") for a in xw[:p]]
        w = [_bf16(a, "weight shard") for a in xw[p:]]
        b = _bf16(bias, "bias") if bias is not None else None
        (M, K), N = x[0].shape, w[0].shape[1]
        ws = _workspace(x[0].device, [(TP_OP_ROW_AR, p, M, N, K, 0), (TP_OP_ROW_BWD, p, M, N, K, 0)])
        y = _empty((M, N), x[0])
        tp_row_linear_fwd_allreduce(x, w, [y], ws, bias=b)
        ctx.p = p
        ctx.save_for_backward(*x, *w)
        return y

    @staticmethod
    def backward(ctx, dy):
        p = ctx.p
        saved = ctx.saved_tensors
        x, w = list(saved[:p]), list(saved[p:])
        (M, K), N = x[0].shape, w[0].shape[1]
        dy = _grad(dy, x[0].new_empty((M, N)))
        need_b = ctx.needs_input_grad[1]
        need_x = any(ctx.needs_input_grad[2:2 + p])
        need_w = any(ctx.needs_input_grad[2 + p:])
        dx = [_empty((M, K), dy) for _ in range(p)] if need_x else None
        dw = [_empty((K, N), dy) for _ in range(p)] if need_w else None
        db = _empty((N,), dy) if need_b else None
        if need_x or need_w or need_b:
            ws = _workspace(dy.device, [(TP_OP_ROW_BWD, p, M, N, K, 0)])
            tp_row_linear_bwd(x, w, dy, dx, dw, ws, db=db)
        return (None, db, *(dx or [None] * p), *(dw or [None] * p))


# ------------------------------------------------------------------ the MLP block

class _MLPFn(torch.autograd.Function):
    """Y = sum_k GeLU(X A1_k + b1_k) A2_k + b2: column FC1 with GeLU, row FC2
    with the fused AllReduce (biases optional).

    Backward: dH_k = (dY A2_k^T) * GeLU'(H_k) in FC2's backward epilogue,
    dA2_k = Z_k^T dY, db2 = row sum of dY, then FC1's dX = sum_k dH_k A1_k^T
    (fused), dA1_k = X^T dH_k and db1_k = row sum of dH_k.  Saves X,
    Z_k = GeLU(H_k) and H_k (bf16)."""

    @staticmethod
    def forward(ctx, p, b2, x, *wb):
        x = _bf16(x, "x")
        w1 = [_bf16(a, "FC1 weight shard") for a in wb[:p]]
        w2 = [_bf16(a, "FC2 weight shard") for a in wb[p:2 * p]]
        b1 = _opt(wb[2 * p:])
        b2 = _bf16(b2, "FC2 bias") if b2 is not None else None
        (M, h), nk = x.shape, w1[0].shape[1]
        ws = _workspace(x.device, [(TP_OP_COL_FWD, p, M, nk, h, 0), (TP_OP_ROW_AR, p, M, h, nk, 0),
                                   (TP_OP_ROW_BWD, p, M, h, nk, 0), (TP_OP_COL_BWD, p, M, nk, h, 0)])
        z = [_empty((M, nk), x) for _ in range(p)]
        hh = [_empty((M, nk), x) for _ in range(p)]
        tp_col_linear_fwd(x, w1, z, ws, epi=TP_EPI_GELU, preact=hh, bias=b1)
        y = _empty((M, h), x)
        tp_row_linear_fwd_allreduce(z, w2, [y], ws, bias=b2)
        ctx.p = p
        ctx.save_for_backward(x, *w1, *w2, *z, *hh)
        return y

    @staticmethod
    def backward(ctx, dy):
        p = ctx.p
        s = ctx.saved_tensors
        x, w1, w2 = s[0], list(s[1:1 + p]), list(s[1 + p:1 + 2 * p])
        z, hh = list(s[1 + 2 * p:1 + 3 * p]), list(s[1 + 3 * p:])
        (M, h), nk = x.shape, w1[0].shape[1]
        dy = _grad(dy, x)
        need_b2 = ctx.needs_input_grad[1]
        need_b1 = any(ctx.needs_input_grad[3 + 2 * p:])
        ws = _workspace(x.device, [(TP_OP_ROW_BWD, p, M, h, nk, 0), (TP_OP_COL_BWD, p, M, nk, h, 0)])
        dz = [_empty((M, nk), x) for _ in range(p)]
        dw2 = [_empty((nk, h), x) for _ in range(p)]
        db2 = _empty((h,), x) if need_b2 else None
        tp_row_linear_bwd(z, w2, dy, dz, dw2, ws, preact=hh, db=db2)
        dx = _empty((M, h), x) if ctx.needs_input_grad[2] else None
        dw1 = [_empty((h, nk), x) for _ in range(p)]
        db1 = [_empty((nk,), x) for _ in range(p)] if need_b1 else None
        tp_col_linear_bwd(x, w1, dz, dx, dw1, ws, db=db1)
        return (None, db2, dx, *dw1, *dw2, *(db1 or [None] * p))


# ------------------------------------------------------------------ sequence parallel (§11.3)

class _AllGatherColumnFn(torch.autograd.Function):
    """Y_k = [X_0; ...; X_{p-1}] A_k + b_k.  Backward: dX_s = rows s of
    sum_k dY_k A_k^T (ReduceScatter), dA_k = X_gathered^T dY_k, db_k = row sum of dY_k."""

    @staticmethod
    def forward(ctx, p, *xwb):
        x = [_bf16(a, "token shard") for a in xwb[:p]]
        w = [_bf16(a, "weight shard") for a in xwb[p:2 * p]]
        b = _opt(xwb[2 * p:])
        (Mp, K), N = x[0].shape, w[0].shape[1]
        M = Mp * p
        ws = _workspace(x[0].device, [(TP_OP_AG_MM, p, M, N, K, 0), (TP_OP_AG_MM_BWD, p, M, N, K, 0)])
        y = [_empty((M, N), x[0]) for _ in range(p)]
        tp_ag_matmul(x, w, y, ws, bias=b)
        ctx.p = p
        ctx.save_for_backward(*x, *w)
        return tuple(y)

    @staticmethod
    def backward(ctx, *dy):
        p = ctx.p
        s = ctx.saved_tensors
        x, w = list(s[:p]), list(s[p:])
        (Mp, K), N = x[0].shape, w[0].shape[1]
        M = Mp * p
        dy = [_grad(g, x[0].new_empty((M, N))) for g in dy]
        need_x = any(ctx.needs_input_grad[1:1 + p])
        need_w = any(ctx.needs_input_grad[1 + p:1 + 2 * p])
        need_b = any(ctx.needs_input_grad[1 + 2 * p:])
        dx = [_empty((Mp, K), x[0]) for _ in range(p)] if need_x else None
        dw = [_empty((K, N), x[0]) for _ in range(p)] if need_w else None
        db = [_empty((N,), x[0]) for _ in range(p)] if need_b else None
        if need_x or need_w or need_b:
            ws = _workspace(x[0].device, [(TP_OP_AG_MM_BWD, p, M, N, K, 0)])
            tp_ag_matmul_bwd(x, w, dy, dx, dw, ws, db=db)
        return (None, *(dx or [None] * p), *(dw or [None] * p), *(db or [None] * p))


class _RowReduceScatterFn(torch.autograd.Function):
    """Y_j = rows j of sum_r X_r A_r + b (ReduceScatter).  Backward: dX_r = [dY_0; ...] A_r^T
    (AllGather of dY), dA_r = X_r^T [dY_0; ...], db = row sum of all dY shards."""

    @staticmethod
    def forward(ctx, p, bias, *xw):
        x = [_bf16(a, "input shard") for a in xw[:p]]
        w = [_bf16(a, "weight shard") for a in xw[p:]]
        b = _bf16(bias, "bias") if bias is not None else None
        (M, K), N = x[0].shape, w[0].shape[1]
        if M % p:
            raise ValueError(f"ReduceScatter needs M % p == 0 (M={M}, p={p})")
        ws = _workspace(x[0].device, [(TP_OP_ROW_RS, p, M, N, K, 0), (TP_OP_ROW_RS_BWD, p, M, N, K, 0)])
        y = [_empty((M // p, N), x[0]) for _ in range(p)]
        tp_row_linear_fwd_reducescatter(x, w, y, ws, bias=b)
        ctx.p = p
        ctx.save_for_backward(*x, *w)
        return tuple(y)

    @staticmethod
    def backward(ctx, *dy):
        p = ctx.p
        s = ctx.saved_tensors
        x, w = list(s[:p]), list(s[p:])
        (M, K), N = x[0].shape, w[0].shape[1]
        dy = [_grad(g, x[0].new_empty((M // p, N))) for g in dy]
        need_b = ctx.needs_input_grad[1]
        need_x = any(ctx.needs_input_grad[2:2 + p])
        need_w = any(ctx.needs_input_grad[2 + p:])
        dx = [_empty((M, K), x[0]) for _ in range(p)] if need_x else None
        dw = [_empty((K, N), x[0]) for _ in range(p)] if need_w else None
        db = _empty((N,), x[0]) if need_b else None
        if need_x or need_w or need_b:
            ws = _workspace(x[0].device, [(TP_OP_ROW_RS_BWD, p, M, N, K, 0)])
            tp_row_linear_bwd_reducescatter(x, w, dy, dx, dw, ws, db=db)
        return (None, db, *(dx or [None] * p), *(dw or [None] * p))


class _SequenceParallelMLPFn(torch.autograd.Function):
    """Token shards in, token shards out: Y_j = rows j of
    sum_k GeLU([X_0;...] A1_k + b1_k) A2_k + b2.

    Forward: AllGather+MatMul with GeLU, then the row layer with the fused
    ReduceScatter.  Backward: the row layer's AllGather of dY with GeLU' in
    the epilogue, then the AllGather+MatMul backward (ReduceScatter of dX)."""

    @staticmethod
    def forward(ctx, p, b2, *args):
        x = [_bf16(a, "token shard") for a in args[:p]]
        w1 = [_bf16(a, "FC1 weight shard") for a in args[p:2 * p]]
        w2 = [_bf16(a, "FC2 weight shard") for a in args[2 * p:3 * p]]
        b1 = _opt(args[3 * p:])
        b2 = _bf16(b2, "FC2 bias") if b2 is not None else None
        (Mp, h), nk = x[0].shape, w1[0].shape[1]
        M = Mp * p
        ws = _workspace(x[0].device, [(TP_OP_AG_MM, p, M, nk, h, 0), (TP_OP_ROW_RS, p, M, h, nk, 0),
                                      (TP_OP_ROW_RS_BWD, p, M, h, nk, 0), (TP_OP_AG_MM_BWD, p, M, nk, h, 0)])
        z = [_empty((M, nk), x[0]) for _ in range(p)]
        hh = [_empty((M, nk), x[0]) for _ in range(p)]
        tp_ag_matmul(x, w1, z, ws, epi=TP_EPI_GELU, preact=hh, bias=b1)
        y = [_empty((Mp, h), x[0]) for _ in range(p)]
        tp_row_linear_fwd_reducescatter(z, w2, y, ws, bias=b2)
        ctx.p = p
        ctx.save_for_backward(*x, *w1, *w2, *z, *hh)
        return tuple(y)

    @staticmethod
    def backward(ctx, *dy):
        p = ctx.p
        s = ctx.saved_tensors
        x, w1, w2 = list(s[:p]), list(s[p:2 * p]), list(s[2 * p:3 * p])
        z, hh = list(s[3 * p:4 * p]), list(s[4 * p:])
        (Mp, h), nk = x[0].shape, w1[0].shape[1]
        M = Mp * p
        dy = [_grad(g, x[0]) for g in dy]
        need_b2 = ctx.needs_input_grad[1]
        need_b1 = any(ctx.needs_input_grad[2 + 3 * p:])
        ws = _workspace(x[0].device, [(TP_OP_ROW_RS_BWD, p, M, h, nk, 0), (TP_OP_AG_MM_BWD, p, M, nk, h, 0)])
        dz = [_empty((M, nk), x[0]) for _ in range(p)]
        dw2 = [_empty((nk, h), x[0]) for _ in range(p)]
        db2 = _empty((h,), x[0]) if need_b2 else None
        tp_row_linear_bwd_reducescatter(z, w2, dy, dz, dw2, ws, preact=hh, db=db2)
        dx = [_empty((Mp, h), x[0]) for _ in range(p)]
        dw1 = [_empty((h, nk), x[0]) for _ in range(p)]
        db1 = [_empty((nk,), x[0]) for _ in range(p)] if need_b1 else None
        tp_ag_matmul_bwd(x, w1, dz, dx, dw1, ws, db=db1)
        return (None, db2, *dx, *dw1, *dw2, *(db1 or [None] * p))


# ------------------------------------------------------------------ functional API

def _blocks(b, p):
    return list(b) if b is not None else [None] * p


def column_parallel_linear(x: torch.Tensor, weights: Sequence[torch.Tensor], biases=None) -> tuple:
    """(Y_0, ..., Y_{p-1}) with Y_k = X A_k (+ b_k); differentiable in X, every A_k and b_k."""
    p = len(weights)
    return _ColumnFn.apply(p, x, *weights, *_blocks(biases, p))


def row_parallel_linear(xs: Sequence[torch.Tensor], weights: Sequence[torch.Tensor], bias=None) -> torch.Tensor:
    """Y = sum_r X_r A_r (+ b) (fused AllReduce); differentiable in every X_r, A_r and b."""
    if len(xs) != len(weights):
        raise ValueError("one input shard per weight shard")
    return _RowFn.apply(len(xs), bias, *xs, *weights)


def parallel_mlp(x: torch.Tensor, w1: Sequence[torch.Tensor], w2: Sequence[torch.Tensor],
                 b1=None, b2=None) -> torch.Tensor:
    """Y = sum_k GeLU(X A1_k + b1_k) A2_k + b2 (the TP tutorial's §7.1 block)."""
    if len(w1) != len(w2):
        raise ValueError("FC1 and FC2 need the same number of shards")
    p = len(w1)
    return _MLPFn.apply(p, b2, x, *w1, *w2, *_blocks(b1, p))


def allgather_column_parallel_linear(xs: Sequence[torch.Tensor], weights: Sequence[torch.Tensor],
                                     biases=None) -> tuple:
    """(Y_0, ..., Y_{p-1}) with Y_k = [X_0; ...; X_{p-1}] A_k (+ b_k) (AllGather+MatMul)."""
    if len(xs) != len(weights):
        raise ValueError("one token shard per weight shard")
    p = len(xs)
    return _AllGatherColumnFn.apply(p, *xs, *weights, *_blocks(biases, p))


def row_parallel_linear_reducescatter(xs: Sequence[torch.Tensor], weights: Sequence[torch.Tensor],
                                      bias=None) -> tuple:
    """(Y_0, ..., Y_{p-1}): rank j's rows of sum_r X_r A_r (+ b) (MatMul+ReduceScatter)."""
    if len(xs) != len(weights):
        raise ValueError("one input shard per weight shard")
    return _RowReduceScatterFn.apply(len(xs), bias, *xs, *weights)


def sequence_parallel_mlp(xs: Sequence[torch.Tensor], w1: Sequence[torch.Tensor],
                          w2: Sequence[torch.Tensor], b1=None, b2=None) -> tuple:
    """Token shards of sum_k GeLU([X_0; ...] A1_k + b1_k) A2_k + b2 (the TP tutorial's §11.3 pair)."""
    if not (len(xs) == len(w1) == len(w2)):
        raise ValueError("one token shard and one FC1/FC2 shard per rank")
    p = len(xs)
    return _SequenceParallelMLPFn.apply(p, b2, *xs, *w1, *w2, *_blocks(b1, p))


# ------------------------------------------------------------------ modules

def _shards(weight: torch.Tensor, p: int, dim: int) -> list:
    n = weight.shape[dim]
    if n % p:
        raise ValueError(f"dimension {dim} of size {n} does not split into {p} shards")
    return [c.contiguous() for c in torch.split(weight, n // p, dim=dim)]


def _params(ts):
    return torch.nn.ParameterList(torch.nn.Parameter(t) for t in ts)


class ColumnParallelLinear(torch.nn.Module):
    """X [M, in] -> p outputs Y_k [M, out/p]; weight [in, out] split into
    contiguous column blocks A_k (TP tutorial §2.3), and the optional bias
    [out] into the matching blocks b_k."""

    def __init__(self, weight: torch.Tensor, p: int, bias: torch.Tensor | None = None):
        super().__init__()
        self.p = p
        self.weights = _params(_shards(weight, p, 1))
        self.biases = _params(_shards(bias, p, 0)) if bias is not None else None

    def forward(self, x: torch.Tensor) -> tuple:
        return column_parallel_linear(x, list(self.weights), list(self.biases) if self.biases else None)


class RowParallelLinear(torch.nn.Module):
    """p input shards X_r [M, in/p] -> Y [M, out] = sum_r X_r A_r (+ b);
    weight [in, out] split into contiguous row blocks A_r (TP tutorial
    §2.4); the bias [out] is added once, after the reduction.  With
    ``sequence_parallel`` the output is the p token shards of Y
    (ReduceScatter) instead of the full Y."""

    def __init__(self, weight: torch.Tensor, p: int, bias: torch.Tensor | None = None,
                 sequence_parallel: bool = False):
        super().__init__()
        self.p = p
        self.sequence_parallel = sequence_parallel
        self.weights = _params(_shards(weight, p, 0))
        self.bias = torch.nn.Parameter(bias.contiguous()) if bias is not None else None

    def forward(self, xs: Sequence[torch.Tensor]):
        if self.sequence_parallel:
            return row_parallel_linear_reducescatter(xs, list(self.weights), self.bias)
        return row_parallel_linear(xs, list(self.weights), self.bias)


class ParallelMLP(torch.nn.Module):
    """Column FC1 [h, ffn] (+ b1 [ffn]) + GeLU, row FC2 [ffn, h] (+ b2 [h]),
    p shards each (TP tutorial §7.1).  Input X [M, h] -> Y [M, h]; with
    ``sequence_parallel`` the input and output are p token shards [M/p, h]
    (§11.3)."""

    def __init__(self, w1: torch.Tensor, w2: torch.Tensor, p: int, b1: torch.Tensor | None = None,
                 b2: torch.Tensor | None = None, sequence_parallel: bool = False):
        super().__init__()
        self.p = p
        self.sequence_parallel = sequence_parallel
        self.w1 = _params(_shards(w1, p, 1))
        self.w2 = _params(_shards(w2, p, 0))
        self.b1 = _params(_shards(b1, p, 0)) if b1 is not None else None
        self.b2 = torch.nn.Parameter(b2.contiguous()) if b2 is not None else None

    def forward(self, x):
        b1 = list(self.b1) if self.b1 is not None else None
        if self.sequence_parallel:
            return sequence_parallel_mlp(x, list(self.w1), list(self.w2), b1, self.b2)
        return parallel_mlp(x, list(self.w1), list(self.w2), b1, self.b2)
