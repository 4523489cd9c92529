"""CPU oracle for the tensor-parallel sharded Linear (fp64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The CUDA
library never calls it and shares no code with it.

Every function is the plain definition of what the sharded Linear computes,
written out in float64 with explicit per-rank partials.  Inputs are numpy
``uint16`` arrays holding bfloat16 bit patterns (exactly what the GPU reads);
they are widened exactly to float64.  A library matmul (numpy ``@`` in
float64) is the only primitive; there is no blocking, fusion or reordering.

Sources (web pages, cited by title and section):

* [M027] "compute-communication fusion" knowledge-base article,
  xuujii.github.io/ai-infra-kb/details/M027.html.
  §01 row-parallel Linear on two ranks (Y = Y0 + Y1; AllReduce vs the
  matching ReduceScatter layout; AllGather then MatMul), §02 chunked
  MatMul->AllReduce and AllGather->MatMul, §03 the worked example and the
  two-engine timeline, §07 the self-check exercises.
* [TP] "PyTorch 2.x tensor parallelism" tutorial,
  www.cnblogs.com/zuoyang/p/22340322.
  §2.3 column parallel, §2.4 row parallel, §2.5-2.7 the collectives,
  §四/§六 forward and backward of both layouts, §7.1 the MLP block
  (column FC1 -> GeLU -> row FC2), §九 the MHA projections, §11.3 the
  sequence-parallel pair.

Readings where the pages are silent (each one is also listed in the design
notes): partials are accumulated without intermediate rounding and summed in
rank order r = 0..p-1; GeLU is the exact erf form; the ReduceScatter splits
the rows of Y into p contiguous blocks; a bias is not part of any workload.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np
from scipy.special import erf as _erf


# ---------------------------------------------------------------- bf16 helpers

def widen(b16: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    b = np.asarray(b16, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bfloat16 bits, round to nearest even (via float32).

    Used only where a chained check feeds the oracle's own intermediate
    (for instance GeLU(H) between FC1 and FC2) into the next layer in the
    same storage type the library hands over.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    b = f.view(np.uint32)
    r = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------- activations

def gelu(h: np.ndarray) -> np.ndarray:
    """GeLU(x) = x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)).  [TP §7.1]"""
    h = np.asarray(h, dtype=np.float64)
    return 0.5 * h * (1.0 + _erf(h / math.sqrt(2.0)))


def gelu_prime(h: np.ndarray) -> np.ndarray:
    """d/dx GeLU(x) = Phi(x) + x * phi(x).  [TP §6.5, §7.1 backward]"""
    h = np.asarray(h, dtype=np.float64)
    cdf = 0.5 * (1.0 + _erf(h / math.sqrt(2.0)))
    pdf = np.exp(-0.5 * h * h) / math.sqrt(2.0 * math.pi)
    return cdf + h * pdf


# ---------------------------------------------------------------- row parallel

def row_partials(xs: Sequence[np.ndarray], ws: Sequence[np.ndarray]) -> list[np.ndarray]:
    """Per-rank partial products P_r = X_r . W_r.  [M027 §01; TP §2.4]

    ``xs[r]`` is X_r [M, K_r] (rank r's column block of X), ``ws[r]`` is
    W_r [K_r, N] (rank r's row block of W).
    """
    assert len(xs) == len(ws) and len(xs) >= 1
    return [widen(x) @ widen(w) for x, w in zip(xs, ws)]


def row_fwd_allreduce(xs, ws, bias=None) -> np.ndarray:
    """MatMul+AllReduce: full Y = sum_r X_r . W_r, summed r = 0, 1, ..., p-1.

    [M027 §01: Y = Y0 + Y1; the AllReduce layout leaves the whole Y on
    every rank.  TP §2.4 / §四: Y = sum_k X_k @ A_k.]
    With ``bias`` (b [N]) the bias is added once, after the reduction:
    Y = sum_k X_k A_k + b.  [TP §四, row-parallel forward]
    """
    parts = row_partials(xs, ws)
    y = parts[0].copy()
    for p_r in parts[1:]:
        y = y + p_r
    if bias is not None:
        y = y + widen(bias)[None, :]
    return y


def row_fwd_allreduce_bf16_collective(xs, ws) -> np.ndarray:
    """The row-parallel output an unfused bf16 AllReduce would produce.

    Each rank's partial P_r = X_r . W_r is handed to the collective as a
    bfloat16 tensor, and the collective adds those tensors in rank order
    r = 0, 1, ..., p-1, storing its running sum as bfloat16 after every
    addition:  acc = bf16(P_0);  acc = bf16(acc + bf16(P_r)).
    This is the separate baseline whose whole-layer output error the fused
    path (one rounding, after all p partials) is compared with.
    [M027 §04: compare the whole layer's output error against the baseline;
    §06: record the separate baseline and the output error.  The rounding
    points are the reading of "an AllReduce of bf16 partials" in rank order.]
    """
    parts = row_partials(xs, ws)
    acc = widen(round_bf16(parts[0]))
    for p_r in parts[1:]:
        acc = widen(round_bf16(acc + widen(round_bf16(p_r))))
    return acc


def row_fwd_reducescatter(xs, ws, bias=None) -> list[np.ndarray]:
    """MatMul+ReduceScatter: rank j holds rows [j*M/p, (j+1)*M/p) of Y
    (Y with the bias added once, as in :func:`row_fwd_allreduce`).

    [M027 §01: ReduceScatter in the layout that matches what follows;
    TP §2.7: reduce, then each rank keeps one slice.]
    """
    y = row_fwd_allreduce(xs, ws, bias)
    p = len(xs)
    m = y.shape[0]
    assert m % p == 0, "ReduceScatter needs M divisible by p"
    mp = m // p
    return [y[j * mp:(j + 1) * mp] for j in range(p)]


def row_bwd_dx(ws, dy, preacts=None) -> list[np.ndarray]:
    """Row-parallel backward, input gradient: dX_k = dY . A_k^T (no reduction).

    With ``preacts`` (the MLP case, FC2 fed by GeLU(H_k)) the gradient is
    carried through the activation: dH_k = (dY . A_k^T) * GeLU'(H_k).
    [TP §四/§六: dX_k = dY @ A_k^T needs no communication; §7.1.]
    """
    g = widen(dy)
    out = []
    for k, w in enumerate(ws):
        d = g @ widen(w).T
        if preacts is not None:
            d = d * gelu_prime(widen(preacts[k]))
        out.append(d)
    return out


def row_bwd_dw(xs, dy) -> list[np.ndarray]:
    """Row-parallel backward, weight gradient: dA_k = X_k^T . dY (local).  [TP §四]"""
    g = widen(dy)
    return [widen(x).T @ g for x in xs]


# ---------------------------------------------------------------- column parallel

def col_fwd(x, ws, apply_gelu: bool = False, biases=None):
    """Column-parallel forward: H_k = X . A_k (+ b_k) for every shard k.  [TP §2.3, §三]

    Returns ``(ys, hs)``: with ``apply_gelu`` ys[k] = GeLU(H_k) (the MLP
    FC1, TP §7.1) and hs[k] = H_k; otherwise ys[k] = H_k and hs is None.
    ``biases[k]`` (b_k [N_k], optional) is rank k's bias block, added before
    the activation.  [TP §三, column-parallel forward Y_k = X A_k + b_k]
    """
    xf = widen(x)
    hs = [xf @ widen(w) for w in ws]
    if biases is not None:
        hs = [h + widen(b)[None, :] for h, b in zip(hs, biases)]
    if apply_gelu:
        return [gelu(h) for h in hs], hs
    return hs, None


def col_bwd_dx(ws, dys) -> np.ndarray:
    """Column-parallel backward, input gradient with its AllReduce:
    dX = sum_k dY_k . A_k^T, summed k = 0, 1, ..., p-1.  [TP §三/§六]"""
    parts = [widen(d) @ widen(w).T for d, w in zip(dys, ws)]
    dx = parts[0].copy()
    for q in parts[1:]:
        dx = dx + q
    return dx


def col_bwd_dw(x, dys) -> list[np.ndarray]:
    """Column-parallel backward, weight gradient: dA_k = X^T . dY_k (local;
    X is replicated on every rank).  [TP §三]"""
    xt = widen(x).T
    return [xt @ widen(d) for d in dys]


# ---------------------------------------------------------------- AllGather + MatMul

def all_gather_rows(xs) -> np.ndarray:
    """AllGather of row shards: X = [X_0; X_1; ...; X_{p-1}].  [TP §2.6]"""
    return np.vstack([widen(x) for x in xs])


def ag_matmul(xs, ws, apply_gelu: bool = False, biases=None):
    """AllGather+MatMul: Y_k = [X_0; ...; X_{p-1}] . A_k (+ b_k).  [M027 §01-§02; TP §11.3]

    Returns ``(ys, hs, x_gathered)`` with ys/hs (and biases) as in :func:`col_fwd`.
    """
    xg = all_gather_rows(xs)
    hs = [xg @ widen(w) for w in ws]
    if biases is not None:
        hs = [h + widen(b)[None, :] for h, b in zip(hs, biases)]
    if apply_gelu:
        return [gelu(h) for h in hs], hs, xg
    return hs, None, xg


# ---------------------------------------------------------------- chunked pipeline

def n_chunks(m: int, chunk_m: int) -> int:
    """Chunks of ``chunk_m`` rows covering M rows; the last one may be short.
    ``chunk_m`` larger than M is clamped to M.  [M027 §03: M=128 in 4 chunks of 32]"""
    if m <= 0:
        return 0
    c = min(chunk_m, m)
    return -(-m // c)


def pipeline_time(c: float, m: float, n: int) -> float:
    """Ideal two-engine timeline of n chunks, compute c and communication m
    per chunk: the first compute, n-1 steps of the slower engine, the last
    communication.  [M027 §03: 3 + 3*max(3, 2) + 2 = 14 ms]"""
    if n <= 0:
        return 0.0
    return c + (n - 1) * max(c, m) + m


def serial_time(c: float, m: float, n: int) -> float:
    """Unpipelined timeline: every chunk computes then communicates.  [M027 §03: 20 ms]"""
    return n * (c + m)


# ---------------------------------------------------------------- collective volumes

def allreduce_bytes(p: int, msg_bytes: float) -> float:
    """Bandwidth-optimal AllReduce volume per rank, 2(p-1)/p * msg.  [TP §2.5]"""
    return 2.0 * (p - 1) / p * msg_bytes


def allgather_bytes(p: int, msg_bytes: float) -> float:
    """AllGather (and ReduceScatter) volume per rank, (p-1)/p * msg.  [TP §2.6-2.7]"""
    return (p - 1) / p * msg_bytes


# ---------------------------------------------------------------- sequence-parallel backward

def ag_matmul_bwd_dx(ws, dys) -> list[np.ndarray]:
    """Backward of AllGather+MatMul, input gradient: the column backward's
    dX = sum_k dY_k . A_k^T (k in order), then ReduceScatter of its rows:
    shard s keeps rows [s*M/p, (s+1)*M/p).  [TP §2.6-2.7: the AllGather's
    backward is a ReduceScatter; §11.3]"""
    dx = col_bwd_dx(ws, dys)
    p = len(ws)
    m = dx.shape[0]
    assert m % p == 0
    mp = m // p
    return [dx[s * mp:(s + 1) * mp] for s in range(p)]


def ag_matmul_bwd_dw(xs, dys) -> list[np.ndarray]:
    """Backward of AllGather+MatMul, weight gradient: dA_k = X^T . dY_k with
    X = [X_0; ...; X_{p-1}] the gathered input.  [TP §三, §11.3]"""
    return col_bwd_dw(np.vstack([np.asarray(x, dtype=np.uint16) for x in xs]), dys)


def row_rs_bwd_dx(ws, dys, preacts=None) -> list[np.ndarray]:
    """Backward of MatMul+ReduceScatter, input gradient: the output gradient
    is gathered, dY = [dY_0; ...; dY_{p-1}], then dX_r = dY . A_r^T
    (times GeLU'(H_r) with preacts).  [TP §2.6-2.7: the ReduceScatter's
    backward is an AllGather; §四; §11.3]"""
    return row_bwd_dx(ws, np.vstack([np.asarray(d, dtype=np.uint16) for d in dys]), preacts)


def row_rs_bwd_dw(xs, dys) -> list[np.ndarray]:
    """Backward of MatMul+ReduceScatter, weight gradient: dA_r = X_r^T . dY
    with dY the gathered output gradient.  [TP §四, §11.3]"""
    return row_bwd_dw(xs, np.vstack([np.asarray(d, dtype=np.uint16) for d in dys]))


# ---------------------------------------------------------------- bias gradients

def bias_grad(dys) -> np.ndarray:
    """Gradient of a bias added to every row: db = sum over rows of dY.

    ``dys`` is one output gradient [M, N] or a list of row blocks of one
    (the token shards of a ReduceScatter output), summed over all their
    rows.  For the column layer, rank k's db_k is bias_grad(dY_k); for the
    row layer, db = bias_grad(dY).  [TP §三/§四: Y_k = X A_k + b_k and
    Y = sum_k X_k A_k + b; b enters every row of Y with weight 1]
    """
    if isinstance(dys, (list, tuple)):
        g = np.vstack([widen(d) for d in dys])
    else:
        g = widen(dys)
    return g.sum(axis=0)
