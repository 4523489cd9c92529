"""GPU parity of every entry point against the CPU oracle, through the C-ABI.

Sizes span several 128x256 tiles, several 64-wide k-blocks and ragged tails
in M, N and K, for p = 1..8, both tile orientations (chunks of >= 128 rows
and the operand-swapped kernel for chunks of 16/32/64 rows) and split-K.

* integer-valued bf16 inputs (|v| <= 4): every fp32 partial sum is an exact
  integer, so fp32 outputs must equal the oracle exactly and bf16 outputs
  must equal the oracle's value rounded to bf16 bit for bit -- this pins
  shard offsets, RS slices, AG routing, chunk order and tile bounds;
* normal inputs through GeLU / GeLU': max|d|/max|ref| <= 5e-3 (bf16) or
  1e-5 (fp32);
* outputs sit between NaN guard bands that must survive the call.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import BF16_TOL, assert_close, dev, host_bits, host_f64

pytestmark = pytest.mark.gpu

PAD = 4096


@pytest.fixture(scope="module")
def tp():
    import gemm_reduce_fusion_gb300 as tp
    return tp


class Guarded:
    """An output tensor with NaN guard bands on both sides."""

    def __init__(self, shape, f32=False):
        import torch
        n = int(np.prod(shape))
        self.full = torch.full((n + 2 * PAD,), float("nan"),
                               dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
        self.t = self.full[PAD:PAD + n].view(*shape)
        self.n = n

    def check_bands(self):
        import torch
        lo = self.full[:PAD]
        hi = self.full[PAD + self.n:]
        assert bool(torch.isnan(lo).all()) and bool(torch.isnan(hi).all()), "write outside the output"


def outs(shapes, f32):
    return [Guarded(s, f32) for s in shapes]


def ints(shape, seed):
    return synth.integer_bf16(shape, seed, 4)


def check_exact(g, ref, f32):
    g.check_bands()
    if f32:
        got = host_f64(g.t)
        assert np.array_equal(got, ref), f"max|d| = {np.max(np.abs(got - ref))}"
    else:
        assert np.array_equal(host_bits(g.t), oracle.round_bf16(ref))


def ws_for(tp, op, p, M, N, K, chunk):
    """A workspace that serves the call with bf16 or fp32 outputs."""
    import torch
    n = max(tp.tp_workspace_size(op, p, M, N, K, chunk, dt) for dt in (tp.TP_BF16, tp.TP_FP32))
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


@pytest.fixture(params=[0, 3], ids=["planned_split", "split3"])
def split_k(tp, request):
    """The planner's split-K factor (0), or every single-CTA launch below one
    wave split 3 ways: the split-K partials and the second stage's epilogues
    then run on the small shapes the planner leaves whole."""
    assert tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, request.param) == tp.TP_OK
    yield request.param
    tp.tp_debug_set(tp.TP_DEBUG_SPLIT_K, 0)


ROW_CASES = [  # p, M, N, K, chunk_m
    (1, 128, 256, 64, 0),
    (2, 300, 520, 200, 0),
    (3, 300, 520, 200, 128),
    (4, 257, 264, 136, 256),
    (2, 300, 520, 200, 32),
    (2, 100, 264, 200, 16),
    (3, 77, 136, 72, 64),
    (8, 130, 72, 64, 0),
    (2, 128, 2048, 1024, 32),   # the worked example's shape, 4 chunks of 32 rows
]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", ROW_CASES)
def test_row_allreduce_exact(tp, split_k, p, M, N, K, chunk, f32):
    xs = [ints((M, K), 100 + r) for r in range(p)]
    ws = [ints((K, N), 200 + r) for r in range(p)]
    ref = oracle.row_fwd_allreduce(xs, ws)
    y = outs([(M, N)], f32)
    ws_ = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [y[0].t], ws_, chunk)
    check_exact(y[0], ref, f32)
    assert tp.tp_get_device_status(ws_) == tp.TP_OK


@pytest.mark.parametrize("p,M,N,K,chunk", [(2, 300, 520, 200, 0), (4, 130, 136, 72, 32)])
def test_row_allreduce_replicas_identical(tp, split_k, p, M, N, K, chunk):
    xs = [ints((M, K), 110 + r) for r in range(p)]
    ws = [ints((K, N), 210 + r) for r in range(p)]
    y = outs([(M, N)] * p, False)
    ws_ = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [g.t for g in y], ws_, chunk)
    ref = oracle.row_fwd_allreduce(xs, ws)
    first = host_bits(y[0].t)
    for g in y:
        check_exact(g, ref, False)
        assert np.array_equal(host_bits(g.t), first)


RS_CASES = [(2, 128, 2048, 1024, 32), (2, 300, 520, 200, 0), (4, 520, 264, 136, 128),
            (3, 450, 136, 72, 16), (8, 512, 72, 64, 64), (4, 4 * 150, 264, 200, 256)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", RS_CASES)
def test_row_reducescatter_exact(tp, split_k, p, M, N, K, chunk, f32):
    xs = [ints((M, K), 120 + r) for r in range(p)]
    ws = [ints((K, N), 220 + r) for r in range(p)]
    refs = oracle.row_fwd_reducescatter(xs, ws)
    y = outs([(M // p, N)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_ROW_RS, p, M, N, K, chunk)
    tp.tp_row_linear_fwd_reducescatter([dev(a) for a in xs], [dev(b) for b in ws], [g.t for g in y], ws_, chunk)
    for g, r in zip(y, refs):
        check_exact(g, r, f32)
    # the slices concatenate to the AllReduce output, bit for bit
    y_ar = outs([(M, N)], f32)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [y_ar[0].t],
                                   ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk), chunk)
    import torch
    assert torch.equal(torch.cat([g.t for g in y], 0), y_ar[0].t)


COL_CASES = [(1, 128, 256, 64, 0), (3, 300, 264, 136, 0), (4, 257, 520, 200, 128), (2, 100, 136, 200, 16),
             (3, 64, 72, 72, 32), (8, 130, 264, 64, 64), (2, 513, 256, 128, 256)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", COL_CASES)
def test_col_fwd_exact(tp, split_k, p, M, N, K, chunk, f32):
    x = ints((M, K), 130)
    ws = [ints((K, N), 230 + k) for k in range(p)]
    refs, _ = oracle.col_fwd(x, ws)
    y = outs([(M, N)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, chunk)
    tp.tp_col_linear_fwd(dev(x), [dev(b) for b in ws], [g.t for g in y], ws_, chunk_m=chunk)
    for g, r in zip(y, refs):
        check_exact(g, r, f32)


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", [(3, 300, 264, 136, 0), (2, 100, 136, 200, 16), (4, 260, 520, 72, 64)])
def test_col_fwd_gelu(tp, split_k, p, M, N, K, chunk, f32):
    # H ~ N(0, 1): the GeLU curve itself is exercised
    x = synth.normal_bf16((M, K), 131, sigma=1.0 / np.sqrt(K))
    ws = [synth.normal_bf16((K, N), 231 + k) for k in range(p)]
    refs, hs = oracle.col_fwd(x, ws, apply_gelu=True)
    y = outs([(M, N)] * p, f32)
    h = outs([(M, N)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, chunk)
    tp.tp_col_linear_fwd(dev(x), [dev(b) for b in ws], [g.t for g in y], ws_, epi=tp.TP_EPI_GELU,
                         preact=[g.t for g in h], chunk_m=chunk)
    for k in range(p):
        y[k].check_bands()
        h[k].check_bands()
        assert_close(host_f64(y[k].t), refs[k], f32, f"gelu y[{k}]")
        assert_close(host_f64(h[k].t), hs[k], f32, f"preact h[{k}]")
    # GeLU applied to the kernel's own H: the epilogue, not the GEMM, is what is checked
    if f32:
        for k in range(p):
            assert_close(host_f64(y[k].t), oracle.gelu(host_f64(h[k].t)), True, "gelu(H)")


def _bf16_grid(lo_exp=-20, hi=16.0):
    """Every bf16 value v with 2^lo_exp <= |v| <= hi, both signs, and 0."""
    b = np.arange(0, 0x8000, dtype=np.uint32)
    v = (b << 16).view(np.float32)
    keep = (v >= 2.0 ** lo_exp) & (v <= hi)
    pos = b[keep].astype(np.uint16)
    return np.concatenate([[0], pos, pos | 0x8000]).astype(np.uint16)


@pytest.mark.parametrize("chunk", [0, 32])
def test_gelu_epilogues_within_their_error_bound(tp, chunk):
    """The GeLU and GeLU' epilogues on every bf16 pre-activation in
    [-16, 16] (magnitudes down to 2^-20), fp32 outputs, against the exact
    functions.  The epilogue's normal CDF follows Abramowitz & Stegun 7.1.26
    (|error| <= 1.5e-7 on erf), so in fp32 |GeLU error| <= 4e-7 |h| and
    |GeLU' error| <= 4e-7.  H reaches the epilogue exactly: the column
    forward multiplies an identity by H, the row backward's product is all
    ones (dY's first column and A's first column are ones)."""
    import torch
    vals = _bf16_grid()
    M, N = 256, 256     # every value about ten times, on 128-row tiles (chunk 0) or 32-token tiles (chunk 32)
    hv = np.resize(vals, M * N).reshape(M, N)
    h = oracle.widen(hv)
    # column forward with GeLU: X = I [M, M], W = H
    eye = synth.f32_to_bf16_bits(np.eye(M, dtype=np.float32))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    pre = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tp.tp_col_linear_fwd(dev(eye), [dev(hv)], [y], ws_for(tp, tp.TP_OP_COL_FWD, 1, M, N, M, chunk),
                         epi=tp.TP_EPI_GELU, preact=[pre], chunk_m=chunk)
    assert np.array_equal(host_f64(pre), h)
    err = np.abs(host_f64(y) - oracle.gelu(h))
    assert np.all(err <= 4e-7 * np.abs(h)), f"GeLU: worst |d|/|h| = {np.max(err / np.maximum(np.abs(h), 1e-30)):.3e}"
    # row backward with GeLU': dX = (dY A^T) * GeLU'(H) with dY A^T = 1
    K, Nb = N, 16
    dy = np.zeros((M, Nb), dtype=np.float32)
    dy[:, 0] = 1.0
    a = np.zeros((K, Nb), dtype=np.float32)
    a[:, 0] = 1.0
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
    tp.tp_row_linear_bwd(None, [dev(synth.f32_to_bf16_bits(a))], dev(synth.f32_to_bf16_bits(dy)), [dx], None,
                         ws_for(tp, tp.TP_OP_ROW_BWD, 1, M, Nb, K, chunk), preact=[dev(hv)], chunk_m=chunk)
    err = np.abs(host_f64(dx) - oracle.gelu_prime(h))
    assert np.all(err <= 4e-7), f"GeLU': max |d| = {err.max():.3e}"


COLB_CASES = [(1, 128, 256, 64, 0), (3, 300, 136, 264, 0), (4, 257, 72, 520, 128), (2, 100, 200, 136, 16),
              (3, 77, 72, 72, 64), (2, 64, 64, 256, 32)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", COLB_CASES)
def test_col_bwd_exact(tp, split_k, p, M, N, K, chunk, f32):
    x = ints((M, K), 140)
    ws = [ints((K, N), 240 + k) for k in range(p)]
    dys = [ints((M, N), 340 + k) for k in range(p)]
    ref_dx = oracle.col_bwd_dx(ws, dys)
    ref_dw = oracle.col_bwd_dw(x, dys)
    dx = outs([(M, K)], f32)
    dw = outs([(K, N)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, chunk)
    tp.tp_col_linear_bwd(dev(x), [dev(b) for b in ws], [dev(d) for d in dys], dx[0].t, [g.t for g in dw],
                         ws_, chunk)
    check_exact(dx[0], ref_dx, f32)
    for g, r in zip(dw, ref_dw):
        check_exact(g, r, f32)


ROWB_CASES = [(1, 128, 256, 64, 0), (3, 300, 136, 264, 0), (4, 257, 520, 72, 128), (2, 100, 136, 200, 16),
              (2, 64, 72, 256, 32), (8, 130, 64, 72, 64)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", ROWB_CASES)
def test_row_bwd_exact(tp, split_k, p, M, N, K, chunk, f32):
    xs = [ints((M, K), 150 + k) for k in range(p)]
    ws = [ints((K, N), 250 + k) for k in range(p)]
    dy = ints((M, N), 350)
    ref_dx = oracle.row_bwd_dx(ws, dy)
    ref_dw = oracle.row_bwd_dw(xs, dy)
    dx = outs([(M, K)] * p, f32)
    dw = outs([(K, N)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, chunk)
    tp.tp_row_linear_bwd([dev(a) for a in xs], [dev(b) for b in ws], dev(dy), [g.t for g in dx],
                         [g.t for g in dw], ws_, chunk_m=chunk)
    for g, r in zip(dx, ref_dx):
        check_exact(g, r, f32)
    for g, r in zip(dw, ref_dw):
        check_exact(g, r, f32)


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", [(3, 300, 136, 264, 0), (2, 100, 136, 200, 16), (4, 130, 64, 72, 64)])
def test_row_bwd_dgelu(tp, split_k, p, M, N, K, chunk, f32):
    ws = [synth.normal_bf16((K, N), 251 + k, sigma=1.0 / np.sqrt(N)) for k in range(p)]
    dy = synth.normal_bf16((M, N), 351)
    hs = [synth.normal_bf16((M, K), 451 + k) for k in range(p)]
    refs = oracle.row_bwd_dx(ws, dy, preacts=hs)
    dx = outs([(M, K)] * p, f32)
    ws_ = ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, chunk)
    tp.tp_row_linear_bwd(None, [dev(b) for b in ws], dev(dy), [g.t for g in dx], None, ws_,
                         preact=[dev(h) for h in hs], chunk_m=chunk)
    for g, r in zip(dx, refs):
        g.check_bands()
        assert_close(host_f64(g.t), r, f32, "dgelu dx")


AG_CASES = [(2, 256, 264, 136, 0), (4, 512, 136, 200, 128), (4, 400, 72, 72, 0), (3, 300, 264, 64, 16),
            (8, 512, 64, 128, 64), (2, 128, 256, 64, 32)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", AG_CASES)
def test_ag_matmul_exact(tp, split_k, p, M, N, K, chunk, f32):
    Mp = M // p
    xs = [ints((Mp, K), 160 + s) for s in range(p)]
    ws = [ints((K, N), 260 + k) for k in range(p)]
    refs, _, xg_ref = oracle.ag_matmul(xs, ws)
    y = outs([(M, N)] * p, f32)
    xg = outs([(M, K)], False)
    ws_ = ws_for(tp, tp.TP_OP_AG_MM, p, M, N, K, chunk)
    tp.tp_ag_matmul([dev(a) for a in xs], [dev(b) for b in ws], [g.t for g in y], ws_, x_gathered=xg[0].t,
                    chunk_m=chunk)
    for g, r in zip(y, refs):
        check_exact(g, r, f32)
    check_exact(xg[0], xg_ref, False)


@pytest.mark.parametrize("p,M,N,K,chunk", [(4, 512, 264, 136, 0), (2, 100, 136, 64, 16)])
def test_ag_matmul_gelu(tp, split_k, p, M, N, K, chunk):
    Mp = M // p
    xs = [synth.normal_bf16((Mp, K), 161 + s, sigma=1.0 / np.sqrt(K)) for s in range(p)]
    ws = [synth.normal_bf16((K, N), 261 + k) for k in range(p)]
    refs, hs, _ = oracle.ag_matmul(xs, ws, apply_gelu=True)
    y = outs([(M, N)] * p, False)
    h = outs([(M, N)] * p, False)
    ws_ = ws_for(tp, tp.TP_OP_AG_MM, p, M, N, K, chunk)
    tp.tp_ag_matmul([dev(a) for a in xs], [dev(b) for b in ws], [g.t for g in y], ws_, epi=tp.TP_EPI_GELU,
                    preact=[g.t for g in h], chunk_m=chunk)
    for k in range(p):
        assert_close(host_f64(y[k].t), refs[k], False, "ag gelu")
        assert_close(host_f64(h[k].t), hs[k], False, "ag preact")


# ------------------------------------------------------------------ coordinate encoding

def test_onehot_routing_row_ar(tp):
    """X_r one-hot: Y[i] = sum_r W_r[c_r(i)] -- a transposed or misrouted tile
    would pick wrong rows."""
    p, M, N, K = 3, 260, 264, 200
    xs = [synth.onehot_bf16(M, K, 170 + r) for r in range(p)]
    ws = [synth.ramp_bf16(K, N, scale=float(r + 1)) for r in range(p)]
    ref = oracle.row_fwd_allreduce(xs, ws)
    for chunk in (0, 32):
        y = outs([(M, N)], True)
        tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [y[0].t],
                                       ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk), chunk)
        check_exact(y[0], ref, True)


# ------------------------------------------------------------------ determinism and chunking

def test_deterministic_and_chunk_invariant(tp):
    import torch
    p, M, N, K = 4, 520, 520, 264
    xs = [dev(synth.normal_bf16((M, K), 180 + r)) for r in range(p)]
    ws = [dev(synth.normal_bf16((K, N), 280 + r, 0.02)) for r in range(p)]
    res = {}
    for chunk in (0, 128, 256, 512, 32, 16):
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        tp.tp_row_linear_fwd_allreduce(xs, ws, [y], tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk), chunk)
        y2 = torch.empty_like(y)
        tp.tp_row_linear_fwd_allreduce(xs, ws, [y2], tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk), chunk)
        assert torch.equal(y, y2), f"run-to-run difference at chunk_m={chunk}"
        res[chunk] = y
    # chunks of >= 128 rows only reorder tiles: identical bits
    for c in (256, 512):
        assert torch.equal(res[c], res[128])
    ref = oracle.row_fwd_allreduce([host_bits(a) for a in xs], [host_bits(b) for b in ws])
    for c, y in res.items():
        assert_close(host_f64(y), ref, False, f"chunk {c}")


# ------------------------------------------------------------------ bias epilogues and bias gradients

def ibias(n, seed):
    return ints((1, n), seed)[0]


BIAS_ROW_CASES = [  # p, M, N, K, chunk_m: 128x256 tiles, operand-swapped, K == 0
    (2, 300, 520, 200, 0), (3, 130, 136, 72, 32), (4, 64, 264, 64, 16), (2, 40, 72, 0, 0)]


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K,chunk", BIAS_ROW_CASES)
def test_row_bias_exact(tp, split_k, p, M, N, K, chunk, f32):
    """Y = sum_r X_r W_r + b (b once, after the reduction), AllReduce with
    replicas and ReduceScatter."""
    xs = [ints((M, K), 600 + r) for r in range(p)]
    ws = [ints((K, N), 610 + r) for r in range(p)]
    b = ibias(N, 620)
    ref = oracle.row_fwd_allreduce(xs, ws, bias=b)
    dx_, dw_ = [dev(a) for a in xs], [dev(c) for c in ws]
    y = outs([(M, N)] * p, f32)
    wsp = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    tp.tp_row_linear_fwd_allreduce(dx_, dw_, [g.t for g in y], wsp, chunk, bias=dev(b))
    for g in y:
        check_exact(g, ref, f32)
    Mr = M - M % p
    ys = outs([(Mr // p, N)] * p, f32)
    tp.tp_row_linear_fwd_reducescatter([a[:Mr] for a in dx_], dw_, [g.t for g in ys],
                                       ws_for(tp, tp.TP_OP_ROW_RS, p, Mr, N, K, chunk), chunk, bias=dev(b))
    for g, r in zip(ys, oracle.row_fwd_reducescatter([a[:Mr] for a in xs], ws, bias=b)):
        check_exact(g, r, f32)
    assert tp.tp_get_device_status(wsp) == tp.TP_OK


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
def test_row_bias_direct_epilogue_both_tile_paths(tp, tile_mode):
    """Enough tiles for no split: the bias is added in the GEMM's own
    epilogue, on 128x256 tiles and on CTA-pair 256x256 tiles."""
    p, M, N, K = 2, 2048, 2560, 64
    xs = [ints((M, K), 630 + r) for r in range(p)]
    ws = [ints((K, N), 632 + r) for r in range(p)]
    b = ibias(N, 634)
    y = outs([(M, N)], True)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(c) for c in ws], [y[0].t],
                                   ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0), bias=dev(b))
    check_exact(y[0], oracle.row_fwd_allreduce(xs, ws, bias=b), True)


@pytest.mark.parametrize("p,M,N,K,chunk", [(2, 300, 264, 136, 0), (3, 77, 136, 72, 64), (2, 2048, 1280, 64, 0),
                                           (2, 24, 72, 0, 0)])
def test_column_and_allgather_bias(tp, split_k, p, M, N, K, chunk):
    """H_k = X A_k + b_k before the GeLU: H exact on integers, GeLU(H) within
    the fp32 tolerance; the AllGather+MatMul form routes b_k by shard k."""
    x = ints((M, K), 640)
    ws = [ints((K, N), 641 + k) for k in range(p)]
    bs = [ibias(N, 650 + k) for k in range(p)]
    W, Bs = [dev(c) for c in ws], [dev(c) for c in bs]
    # GeLU with the pre-activation saved (fp32 outputs, one dtype per call)
    zr, hr = oracle.col_fwd(x, ws, apply_gelu=True, biases=bs)
    yf = outs([(M, N)] * p, True)
    h = outs([(M, N)] * p, True)
    tp.tp_col_linear_fwd(dev(x), W, [g.t for g in yf], ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, chunk),
                         epi=tp.TP_EPI_GELU, preact=[g.t for g in h], chunk_m=chunk, bias=Bs)
    for k in range(p):
        check_exact(h[k], hr[k], True)
        yf[k].check_bands()
        assert_close(host_f64(yf[k].t), zr[k], True, f"GeLU(H_{k})")
    # no activation, bf16 outputs
    y = outs([(M, N)] * p, False)
    tp.tp_col_linear_fwd(dev(x), W, [g.t for g in y], ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, chunk),
                         chunk_m=chunk, bias=Bs)
    hplain, _ = oracle.col_fwd(x, ws, biases=bs)
    for k in range(p):
        check_exact(y[k], hplain[k], False)
    # AllGather+MatMul over the row shards of X
    Mr = M - M % p
    xs = [np.ascontiguousarray(x[s * (Mr // p):(s + 1) * (Mr // p)]) for s in range(p)]
    ya = outs([(Mr, N)] * p, True)
    tp.tp_ag_matmul([dev(a) for a in xs], W, [g.t for g in ya], ws_for(tp, tp.TP_OP_AG_MM, p, Mr, N, K, chunk),
                    chunk_m=chunk, bias=Bs)
    yr, _, _ = oracle.ag_matmul(xs, ws, biases=bs)
    for k in range(p):
        check_exact(ya[k], yr[k], True)


@pytest.mark.parametrize("f32", [True, False])
@pytest.mark.parametrize("p,M,N,K", [(2, 300, 72, 64), (4, 1024, 264, 136), (3, 96, 520, 72), (2, 0, 136, 64)])
def test_bias_gradients_exact(tp, split_k, p, M, N, K, f32):
    """db = the row sums of dY on integer inputs (exact in fp32): column
    backward (one per shard), row backward, AllGather+MatMul backward (with
    dW in the same call) and the ReduceScatter backward (summed over the
    token shards in order).  M == 0 gives zeros."""
    assert M % p == 0
    Mp = M // p
    dys = [ints((M, N), 660 + k) for k in range(p)]
    x = ints((M, K), 680)
    W = [dev(ints((K, N), 670 + k)) for k in range(p)]
    DY = [dev(d) for d in dys]
    db = outs([(N,)] * p, f32)
    tp.tp_col_linear_bwd(None, W, DY, None, None, ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0),
                         db=[g.t for g in db])
    for g, d in zip(db, dys):
        check_exact(g, oracle.bias_grad(d), f32)
    db1 = outs([(N,)], f32)
    tp.tp_row_linear_bwd(None, W, DY[0], None, None, ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0), db=db1[0].t)
    check_exact(db1[0], oracle.bias_grad(dys[0]), f32)
    xs = [np.ascontiguousarray(x[s * Mp:(s + 1) * Mp]) for s in range(p)]
    dw = outs([(K, N)] * p, f32)
    db = outs([(N,)] * p, f32)
    tp.tp_ag_matmul_bwd([dev(a) for a in xs], W, DY, None, [g.t for g in dw],
                        ws_for(tp, tp.TP_OP_AG_MM_BWD, p, M, N, K, 0), db=[g.t for g in db])
    for g, d in zip(db, dys):
        check_exact(g, oracle.bias_grad(d), f32)
    for g, r in zip(dw, oracle.ag_matmul_bwd_dw(xs, dys)):
        check_exact(g, r, f32)
    shards = [np.ascontiguousarray(dys[0][s * Mp:(s + 1) * Mp]) for s in range(p)]
    dbr = outs([(N,)], f32)
    tp.tp_row_linear_bwd_reducescatter(None, W, [dev(a) for a in shards], None, None,
                                       ws_for(tp, tp.TP_OP_ROW_RS_BWD, p, M, N, K, 0), db=dbr[0].t)
    check_exact(dbr[0], oracle.bias_grad(shards), f32)


# ------------------------------------------------------------------ last-wave k-slices (CTA pairs)
#
# A CTA-pair launch whose tile count leaves a last partial wave of R tiles
# (R <= half the clusters) runs those tiles as 2-4 k-slices; the warp that
# finishes a slice last sums the slices in slice order.  Integer inputs:
# exact, for every epilogue on the slice path.

def test_tail_slices_row_allreduce_and_reducescatter_exact(tp):
    p, M, N, K = 2, 2048, 2560, 1024      # 80 pair tiles: 4 in the last wave, 4 slices each
    xs = [ints((M, K), 700 + r) for r in range(p)]
    ws = [ints((K, N), 702 + r) for r in range(p)]
    b = ibias(N, 704)
    X, W = [dev(a) for a in xs], [dev(c) for c in ws]
    ref = oracle.row_fwd_allreduce(xs, ws, bias=b)
    for f32 in (True, False):
        y = outs([(M, N)] * p, f32)
        tp.tp_row_linear_fwd_allreduce(X, W, [g.t for g in y], ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0),
                                       bias=dev(b))
        for g in y:
            check_exact(g, ref, f32)
    p, M, N, K = 4, 2048, 2560, 512       # ReduceScatter: groups along M, 80 pair tiles
    xs = [ints((M, K), 706 + r) for r in range(p)]
    ws = [ints((K, N), 710 + r) for r in range(p)]
    ys = outs([(M // p, N)] * p, True)
    tp.tp_row_linear_fwd_reducescatter([dev(a) for a in xs], [dev(c) for c in ws], [g.t for g in ys],
                                       ws_for(tp, tp.TP_OP_ROW_RS, p, M, N, K, 0))
    for g, r in zip(ys, oracle.row_fwd_reducescatter(xs, ws)):
        check_exact(g, r, True)


def test_tail_slices_column_gelu_and_backward_exact(tp):
    """Ragged M and N inside the sliced tiles: column forward with bias,
    GeLU and the saved H; row backward with GeLU' (H read back); weight
    gradients (both operands MN-major)."""
    p, M, N, K = 4, 1000, 1240, 1024      # 4 x 4 x 5 = 80 pair tiles, 2 slices
    x = ints((M, K), 720)
    ws = [ints((K, N), 721 + k) for k in range(p)]
    bs = [ibias(N, 726 + k) for k in range(p)]
    y = outs([(M, N)] * p, True)
    h = outs([(M, N)] * p, True)
    tp.tp_col_linear_fwd(dev(x), [dev(c) for c in ws], [g.t for g in y], ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, 0),
                         epi=tp.TP_EPI_GELU, preact=[g.t for g in h], bias=[dev(c) for c in bs])
    zr, hr = oracle.col_fwd(x, ws, apply_gelu=True, biases=bs)
    for k in range(p):
        check_exact(h[k], hr[k], True)
        y[k].check_bands()
        assert_close(host_f64(y[k].t), zr[k], True, f"GeLU(H_{k})")
    # row backward: dX_k = dY W_k^T * GeLU'(H_k); here W_k is [K=1240, N=1024]
    Kr, Nr = 1240, 1024
    w2 = [ints((Kr, Nr), 730 + k) for k in range(p)]
    dy = ints((M, Nr), 735)
    hb = [synth.normal_bf16((M, Kr), synth.seed_for(61, k)) for k in range(p)]
    dx = outs([(M, Kr)] * p, True)
    tp.tp_row_linear_bwd(None, [dev(c) for c in w2], dev(dy), [g.t for g in dx], None,
                         ws_for(tp, tp.TP_OP_ROW_BWD, p, M, Nr, Kr, 0), preact=[dev(a) for a in hb])
    for g, r in zip(dx, oracle.row_bwd_dx(w2, dy, preacts=hb)):
        g.check_bands()
        assert_close(host_f64(g.t), r, True, "dX * GeLU'")
    # the same without GeLU': exact
    dx2 = outs([(M, Kr)] * p, True)
    tp.tp_row_linear_bwd(None, [dev(c) for c in w2], dev(dy), [g.t for g in dx2], None,
                         ws_for(tp, tp.TP_OP_ROW_BWD, p, M, Nr, Kr, 0))
    for g, r in zip(dx2, oracle.row_bwd_dx(w2, dy)):
        check_exact(g, r, True)
    # weight gradients dW_k = X_k^T dY: [1240, 1280] per k, 4 x 5 x 5 = 100 pair tiles
    Mw, Kw, Nw = 1024, 1240, 1280
    xw = [ints((Mw, Kw), 740 + k) for k in range(p)]
    dyw = ints((Mw, Nw), 745)
    ww = [ints((Kw, Nw), 746 + k) for k in range(p)]
    dw = outs([(Kw, Nw)] * p, True)
    tp.tp_row_linear_bwd([dev(a) for a in xw], [dev(c) for c in ww], dev(dyw), None, [g.t for g in dw],
                         ws_for(tp, tp.TP_OP_ROW_BWD, p, Mw, Nw, Kw, 0))
    for g, r in zip(dw, oracle.row_bwd_dw(xw, dyw)):
        check_exact(g, r, True)


def test_workspace_without_room_for_slices_runs_whole_tiles(tp):
    """A workspace smaller than tp_workspace_size() but large enough for the
    plan without last-wave slices is accepted: same result bit for bit on
    integer inputs, and a workspace below that is still rejected."""
    import torch
    p, M, N, K = 2, 2048, 2560, 1024
    xs = [ints((M, K), 750 + r) for r in range(p)]
    ws = [ints((K, N), 752 + r) for r in range(p)]
    X, W = [dev(a) for a in xs], [dev(c) for c in ws]
    full = tp.tp_workspace_size(tp.TP_OP_ROW_AR, p, M, N, K, 0)
    assert full > 256
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    y = outs([(M, N)], True)
    tp.tp_row_linear_fwd_allreduce(X, W, [y[0].t], small)
    check_exact(y[0], oracle.row_fwd_allreduce(xs, ws), True)
    assert tp.tp_get_device_status(small) == tp.TP_OK
    # a skinny call that needs split-K partials even without slices
    p, M, N, K = 8, 16, 2048, 1024
    x8 = [dev(ints((M, K), 760 + r)) for r in range(p)]
    w8 = [dev(ints((K, N), 770 + r)) for r in range(p)]
    y8 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_row_linear_fwd_allreduce(x8, w8, [y8], small, chunk_m=16)
    assert e.value.status == tp.TP_ERR_WORKSPACE_TOO_SMALL


def test_tail_slices_deterministic(tp):
    """Which warp finishes a slice last changes from run to run; the result
    does not (normal inputs, fp32 and bf16 outputs)."""
    import torch
    p, M, N, K = 2, 2048, 2560, 1024
    X = [dev(synth.normal_bf16((M, K), synth.seed_for(62, r))) for r in range(p)]
    W = [dev(synth.normal_bf16((K, N), synth.seed_for(62, 4 + r), 0.02)) for r in range(p)]
    wsp = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0)
    for dt in (torch.float32, torch.bfloat16):
        first = torch.empty((M, N), dtype=dt, device="cuda")
        tp.tp_row_linear_fwd_allreduce(X, W, [first], wsp)
        for _ in range(4):
            again = torch.empty_like(first)
            tp.tp_row_linear_fwd_allreduce(X, W, [again], wsp)
            assert torch.equal(first, again)
    ref = oracle.row_fwd_allreduce([host_bits(a) for a in X], [host_bits(b) for b in W])
    assert_close(host_f64(first), ref, False, "sliced AllReduce")


# ------------------------------------------------------------------ timeline trace

def test_timeline_trace_records_every_unit(tp):
    """A traced launch records each unit once, in order start <= full <=
    drained, tags every chunk, and leaves the result bit-identical."""
    import torch
    p, M, N, K, chunk = 2, 512, 520, 200, 128     # 4 chunks of 128 rows on 128x256 tiles
    xs = [dev(ints((M, K), 780 + r)) for r in range(p)]
    ws = [dev(ints((K, N), 782 + r)) for r in range(p)]
    wsp = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, chunk)
    plain = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tp.tp_row_linear_fwd_allreduce(xs, ws, [plain], wsp, chunk)
    buf = torch.zeros((4096, 4), dtype=torch.int64, device="cuda")
    traced = torch.empty_like(plain)
    tp.tp_trace_set(buf, 4096)
    try:
        tp.tp_row_linear_fwd_allreduce(xs, ws, [traced], wsp, chunk)
        torch.cuda.synchronize()
    finally:
        tp.tp_trace_set(None)
    assert torch.equal(plain, traced)
    rec = buf.cpu().numpy()
    used = rec[rec[:, 0] != 0]
    assert len(used) >= 4 * 3                              # 4 chunks x 3 column tiles (x splits)
    assert np.all(used[:, 0] <= used[:, 1]) and np.all(used[:, 1] <= used[:, 2])
    assert sorted(set((used[:, 3] >> 32).tolist())) == [0, 1, 2, 3]
    assert not np.any(rec[len(used):, 0])                  # units are numbered from 0, densely


# ------------------------------------------------------------------ concurrent streams

def test_two_streams_with_their_own_workspaces(tp):
    """Calls enqueued on two streams with no ordering between them, each with
    its own workspace (one a sliced CTA-pair launch, one a split-K skinny
    launch), both exact."""
    import torch
    p, M, N, K = 2, 2048, 2560, 512
    xa = [ints((M, K), 790 + r) for r in range(p)]
    wa = [ints((K, N), 792 + r) for r in range(p)]
    pb, Mb, Nb, Kb = 8, 16, 2048, 512
    xb = [ints((Mb, Kb), 794 + r) for r in range(pb)]
    wb = [ints((Kb, Nb), 803 + r) for r in range(pb)]
    XA, WA = [dev(a) for a in xa], [dev(b) for b in wa]
    XB, WB = [dev(a) for a in xb], [dev(b) for b in wb]
    ya = torch.empty((M, N), dtype=torch.float32, device="cuda")
    yb = torch.empty((Mb, Nb), dtype=torch.float32, device="cuda")
    wsa = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0)
    wsb = ws_for(tp, tp.TP_OP_ROW_AR, pb, Mb, Nb, Kb, 16)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            tp.tp_row_linear_fwd_allreduce(XA, WA, [ya], wsa)
        with torch.cuda.stream(s2):
            tp.tp_row_linear_fwd_allreduce(XB, WB, [yb], wsb, chunk_m=16)
    torch.cuda.synchronize()
    assert tp.tp_get_device_status(wsa) == tp.TP_OK and tp.tp_get_device_status(wsb) == tp.TP_OK
    assert np.array_equal(host_f64(ya), oracle.row_fwd_allreduce(xa, wa))
    assert np.array_equal(host_f64(yb), oracle.row_fwd_allreduce(xb, wb))


# ------------------------------------------------------------------ calls from other threads

def test_call_from_a_fresh_thread(tp):
    """A thread that made no CUDA call before (as autograd's worker threads)
    gets the same results as the main thread."""
    import threading
    import torch
    p, M, N, K = 2, 300, 264, 136
    x = ints((M, K), 560)
    ws = [ints((K, N), 561 + k) for k in range(p)]
    dys = [ints((M, N), 563 + k) for k in range(p)]
    X, W, DY = dev(x), [dev(a) for a in ws], [dev(a) for a in dys]
    wsp = ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0)
    res = {}

    def run():
        try:
            dx = outs([(M, K)], True)
            dw = outs([(K, N)] * p, True)
            tp.tp_col_linear_bwd(X, W, DY, dx[0].t, [g.t for g in dw], wsp)
            torch.cuda.synchronize()
            res["out"] = (dx, dw)
        except Exception as e:  # re-raised on the main thread
            res["err"] = e

    t = threading.Thread(target=run)
    t.start()
    t.join()
    if "err" in res:
        raise res["err"]
    dx, dw = res["out"]
    check_exact(dx[0], oracle.col_bwd_dx(ws, dys), True)
    for g, r in zip(dw, oracle.col_bwd_dw(x, dys)):
        check_exact(g, r, True)
    assert tp.tp_get_device_status(wsp) == tp.TP_OK


# ------------------------------------------------------------------ edge cases

def test_edge_sizes(tp):
    import torch
    p, N, K = 2, 72, 64
    # M == 0: accepted, nothing written
    w = [dev(ints((K, N), 5 + r)) for r in range(p)]
    x0 = [torch.empty((0, K), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    y0 = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    tp.tp_row_linear_fwd_allreduce(x0, w, [y0], tp.workspace(0, p, 0, N, K, 0))
    # K == 0: zeros
    xk = [torch.empty((5, 0), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    wk = [torch.empty((0, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    yk = torch.full((5, N), 7.0, dtype=torch.bfloat16, device="cuda")
    st = tp._lib.tp_row_linear_fwd_allreduce(tp._arr(xk), tp._arr(wk), None, tp._arr([yk]), 1, p, 5, N, 0, 0, 0,
                                             tp._ptr(tp.workspace(0, p, 5, N, 0)), 256,
                                             torch.cuda.current_stream().cuda_stream)
    assert st == tp.TP_OK
    assert bool((yk == 0).all())
    # M == 1, N == 8, K == 8, p == 8, chunk_m far above M
    p, M, N, K = 8, 1, 8, 8
    xs = [ints((M, K), 60 + r) for r in range(p)]
    ws = [ints((K, N), 70 + r) for r in range(p)]
    y = outs([(M, N)], True)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [y[0].t],
                                   tp.workspace(0, p, M, N, K, 4096), 4096)
    check_exact(y[0], oracle.row_fwd_allreduce(xs, ws), True)


def test_misaligned_pointer_rejected_on_device(tp):
    import torch
    p, M, N, K = 2, 16, 8, 8
    buf = torch.zeros(M * K + 8, dtype=torch.bfloat16, device="cuda")
    bad = buf[1:1 + M * K].view(M, K)    # 2-byte offset: not 16-byte aligned
    w = [torch.zeros((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_row_linear_fwd_allreduce([bad, bad], w, [y], tp.workspace(0, p, M, N, K, 0))
    assert e.value.status == tp.TP_ERR_ALIGNMENT


# ------------------------------------------------------------------ unfused baseline

@pytest.mark.parametrize("p,M,N,K,chunk", [(2, 300, 520, 200, 0), (4, 130, 136, 72, 32), (3, 64, 264, 64, 16)])
def test_unfused_baseline_exact(tp, p, M, N, K, chunk):
    """Per-rank fp32 partials then the rank-order reduce: run whole, and as
    its two phases separately; both equal the oracle exactly."""
    xs = [ints((M, K), 190 + r) for r in range(p)]
    ws = [ints((K, N), 290 + r) for r in range(p)]
    ref = oracle.row_fwd_allreduce(xs, ws)
    dx, dw = [dev(a) for a in xs], [dev(b) for b in ws]
    for split in (False, True):
        y = outs([(M, N)], True)
        wsp = ws_for(tp, tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, chunk)
        if split:
            tp.tp_row_linear_fwd_unfused(dx, dw, y[0].t, wsp, chunk, phases=1)
            tp.tp_row_linear_fwd_unfused(dx, dw, y[0].t, wsp, chunk, phases=2)
        else:
            tp.tp_row_linear_fwd_unfused(dx, dw, y[0].t, wsp, chunk, phases=3)
        check_exact(y[0], ref, True)


# ------------------------------------------------------------------ bf16-collective emulation

@pytest.mark.parametrize("p,M,N,K,chunk", [(2, 300, 520, 200, 0), (4, 130, 136, 72, 32), (8, 64, 264, 64, 16)])
def test_unfused_bf16_collective_exact(tp, p, M, N, K, chunk):
    """Integer inputs: every fp32 partial is an exact integer, many above 256
    where bf16 has to round, so each rounding of the emulated bf16 collective
    is decided the same way on both sides and the GPU equals the oracle bit
    for bit, with bf16 and with fp32 output buffers."""
    xs = [ints((M, K), 195 + r) for r in range(p)]
    ws = [ints((K, N), 295 + r) for r in range(p)]
    ref = oracle.row_fwd_allreduce_bf16_collective(xs, ws)
    assert not np.array_equal(ref, oracle.row_fwd_allreduce(xs, ws))  # rounding is exercised
    dx, dw = [dev(a) for a in xs], [dev(b) for b in ws]
    for f32 in (False, True):
        y = outs([(M, N)], f32)
        wsp = ws_for(tp, tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, chunk)
        tp.tp_row_linear_fwd_unfused(dx, dw, y[0].t, wsp, chunk, flags=tp.TP_UNFUSED_BF16_COLLECTIVE)
        check_exact(y[0], ref, f32)


def test_unfused_bf16_collective_normal_inputs(tp):
    """Normal inputs at p = 8: the emulation matches the oracle's bf16
    collective within the bf16 tolerance, and its error against the exact
    sum is at least that of the fused path (which rounds once)."""
    import torch
    from gpu_util import rel_err
    p, M, N, K = 8, 256, 512, 1024
    xs = [synth.normal_bf16((M, K), synth.seed_for(50, r)) for r in range(p)]
    ws = [synth.normal_bf16((K, N), synth.seed_for(50, 8 + r), 0.02) for r in range(p)]
    dx, dw = [dev(a) for a in xs], [dev(b) for b in ws]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tp.tp_row_linear_fwd_unfused(dx, dw, y, ws_for(tp, tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, 0), 0,
                                 flags=tp.TP_UNFUSED_BF16_COLLECTIVE)
    got = host_f64(y)
    assert_close(got, oracle.row_fwd_allreduce_bf16_collective(xs, ws), False, "bf16 collective")
    fused = torch.empty_like(y)
    tp.tp_row_linear_fwd_allreduce(dx, dw, [fused], ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0))
    exact = oracle.row_fwd_allreduce(xs, ws)
    assert rel_err(got, exact) >= rel_err(host_f64(fused), exact)


def test_unfused_rejects_unknown_flags(tp):
    import torch
    p, M, N, K = 2, 16, 8, 8
    x = [torch.zeros((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    w = [torch.zeros((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tp.TPError) as e:
        tp.tp_row_linear_fwd_unfused(x, w, y, ws_for(tp, tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, 0), flags=2)
    assert e.value.status == tp.TP_ERR_INVALID_ARG


# ------------------------------------------------------------------ fp32 outputs at long contractions

def test_fp32_mode_within_1e5_at_large_k(tp):
    """p = 4 ranks of K = 4096 (16384 in all): fp32 outputs stay within 1e-5
    of max|Y| of the exact sum, for the AllReduce (both chunk paths) and the
    ReduceScatter."""
    import torch
    p, M, N, K = 4, 256, 512, 4096
    xs = [synth.normal_bf16((M, K), synth.seed_for(51, r)) for r in range(p)]
    ws = [synth.normal_bf16((K, N), synth.seed_for(51, 8 + r)) for r in range(p)]
    dx, dw = [dev(a) for a in xs], [dev(b) for b in ws]
    ref = oracle.row_fwd_allreduce(xs, ws)
    for chunk in (0, 32):
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        wsp = tp.workspace(tp.TP_OP_ROW_AR, p, M, N, K, chunk, out_dtype=tp.TP_FP32)
        tp.tp_row_linear_fwd_allreduce(dx, dw, [y], wsp, chunk)
        assert_close(host_f64(y), ref, True, f"AllReduce chunk {chunk}")
    ys = [torch.empty((M // p, N), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_row_linear_fwd_reducescatter(dx, dw, ys, tp.workspace(tp.TP_OP_ROW_RS, p, M, N, K, 0,
                                                                out_dtype=tp.TP_FP32))
    for j in range(p):
        assert_close(host_f64(ys[j]), ref[j * (M // p):(j + 1) * (M // p)], True, f"ReduceScatter {j}")


def test_fp32_mode_column_long_contractions(tp):
    """Column forward with GeLU over K = 16384, and the column backward whose
    dX contracts over p * N = 8192 and whose dW contracts over M = 8192."""
    import torch
    p, M, N, K = 2, 256, 256, 16384
    x = synth.normal_bf16((M, K), synth.seed_for(52, 0))
    ws = [synth.normal_bf16((K, N), synth.seed_for(52, 1 + k), 0.02) for k in range(p)]
    y = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(p)]
    h = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_col_linear_fwd(dev(x), [dev(b) for b in ws], y,
                         tp.workspace(tp.TP_OP_COL_FWD, p, M, N, K, 0, out_dtype=tp.TP_FP32),
                         epi=tp.TP_EPI_GELU, preact=h)
    zr, hr = oracle.col_fwd(x, ws, apply_gelu=True)
    for k in range(p):
        assert_close(host_f64(h[k]), hr[k], True, f"H {k}")
        assert_close(host_f64(y[k]), zr[k], True, f"GeLU(H) {k}")
    p, M, N, K = 2, 8192, 4096, 256
    xb = synth.normal_bf16((M, K), synth.seed_for(53, 0))
    wb = [synth.normal_bf16((K, N), synth.seed_for(53, 1 + k), 0.02) for k in range(p)]
    dyb = [synth.normal_bf16((M, N), synth.seed_for(53, 4 + k)) for k in range(p)]
    dxo = torch.empty((M, K), dtype=torch.float32, device="cuda")
    dwo = [torch.empty((K, N), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_col_linear_bwd(dev(xb), [dev(b) for b in wb], [dev(d) for d in dyb], dxo, dwo,
                         tp.workspace(tp.TP_OP_COL_BWD, p, M, N, K, 0, out_dtype=tp.TP_FP32))
    rows = np.arange(0, M, 61)
    assert_close(host_f64(dxo)[rows], oracle.col_bwd_dx(wb, [d[rows] for d in dyb]), True, "dX")
    cols = np.arange(0, N, 37)
    dwr = oracle.col_bwd_dw(xb, [d[:, cols] for d in dyb])
    for k in range(p):
        assert_close(host_f64(dwo[k])[:, cols], dwr[k], True, f"dW {k}")


# ------------------------------------------------------------------ both tile paths

@pytest.fixture
def tile_mode(tp, request):
    """Force 128x256 single-CTA tiles (1) or 256x256 CTA-pair tiles (2)."""
    assert tp.tp_debug_set(tp.TP_DEBUG_TILE_MODE, request.param) == tp.TP_OK
    yield request.param
    tp.tp_debug_set(tp.TP_DEBUG_TILE_MODE, 0)


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K", [(1, 256, 256, 64), (2, 300, 520, 200), (3, 513, 264, 136), (4, 1300, 776, 72),
                                     (2, 300, 256, 192), (3, 130, 512, 320), (2, 640, 320, 448)])
def test_tile_paths_row_ops_exact(tp, tile_mode, p, M, N, K):
    xs = [ints((M, K), 500 + r) for r in range(p)]
    ws = [ints((K, N), 510 + r) for r in range(p)]
    y = outs([(M, N)], True)
    tp.tp_row_linear_fwd_allreduce([dev(a) for a in xs], [dev(b) for b in ws], [y[0].t],
                                   ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0), 0)
    check_exact(y[0], oracle.row_fwd_allreduce(xs, ws), True)
    Mr = M - M % p
    xr = [a[:Mr] for a in xs]
    ys = outs([(Mr // p, N)] * p, False)
    tp.tp_row_linear_fwd_reducescatter([dev(a) for a in xr], [dev(b) for b in ws], [g.t for g in ys],
                                       ws_for(tp, tp.TP_OP_ROW_RS, p, Mr, N, K, 0), 0)
    for g, r in zip(ys, oracle.row_fwd_reducescatter(xr, ws)):
        check_exact(g, r, False)
    dy = ints((M, N), 520)
    dx = outs([(M, K)] * p, True)
    dw = outs([(K, N)] * p, True)
    tp.tp_row_linear_bwd([dev(a) for a in xs], [dev(b) for b in ws], dev(dy), [g.t for g in dx],
                         [g.t for g in dw], ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0))
    for g, r in zip(dx, oracle.row_bwd_dx(ws, dy)):
        check_exact(g, r, True)
    for g, r in zip(dw, oracle.row_bwd_dw(xs, dy)):
        check_exact(g, r, True)


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K", [(1, 256, 256, 64), (3, 300, 264, 136), (2, 777, 520, 200), (2, 300, 320, 192),
                                     (4, 520, 256, 320)])
def test_tile_paths_col_ops_exact(tp, tile_mode, p, M, N, K):
    x = ints((M, K), 530)
    ws = [ints((K, N), 540 + k) for k in range(p)]
    y = outs([(M, N)] * p, False)
    tp.tp_col_linear_fwd(dev(x), [dev(b) for b in ws], [g.t for g in y], ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, 0))
    refs, _ = oracle.col_fwd(x, ws)
    for g, r in zip(y, refs):
        check_exact(g, r, False)
    dys = [ints((M, N), 550 + k) for k in range(p)]
    dx = outs([(M, K)], True)
    dw = outs([(K, N)] * p, True)
    tp.tp_col_linear_bwd(dev(x), [dev(b) for b in ws], [dev(d) for d in dys], dx[0].t, [g.t for g in dw],
                         ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0))
    check_exact(dx[0], oracle.col_bwd_dx(ws, dys), True)
    for g, r in zip(dw, oracle.col_bwd_dw(x, dys)):
        check_exact(g, r, True)
    Mg = M - M % p
    xs = [x[s * (Mg // p):(s + 1) * (Mg // p)] for s in range(p)]
    ya = outs([(Mg, N)] * p, True)
    tp.tp_ag_matmul([dev(a) for a in xs], [dev(b) for b in ws], [g.t for g in ya],
                    ws_for(tp, tp.TP_OP_AG_MM, p, Mg, N, K, 0))
    refa, _, _ = oracle.ag_matmul(xs, ws)
    for g, r in zip(ya, refa):
        check_exact(g, r, True)


@pytest.mark.parametrize("tile_mode", [2], indirect=True)
def test_pair_path_gelu_epilogues(tp, tile_mode):
    p, M, N, K = 2, 520, 264, 136
    x = synth.normal_bf16((M, K), 560, sigma=1.0 / np.sqrt(K))
    ws = [synth.normal_bf16((K, N), 561 + k) for k in range(p)]
    y = outs([(M, N)] * p, False)
    h = outs([(M, N)] * p, False)
    tp.tp_col_linear_fwd(dev(x), [dev(b) for b in ws], [g.t for g in y], ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, 0),
                         epi=tp.TP_EPI_GELU, preact=[g.t for g in h])
    refs, hs = oracle.col_fwd(x, ws, apply_gelu=True)
    for k in range(p):
        assert_close(host_f64(y[k].t), refs[k], False, "pair gelu")
        assert_close(host_f64(h[k].t), hs[k], False, "pair preact")
    w2 = [synth.normal_bf16((K, N), 570 + k, sigma=1.0 / np.sqrt(N)) for k in range(p)]
    dy = synth.normal_bf16((M, N), 580)
    hk = [synth.normal_bf16((M, K), 590 + k) for k in range(p)]
    dx = outs([(M, K)] * p, False)
    tp.tp_row_linear_bwd(None, [dev(b) for b in w2], dev(dy), [g.t for g in dx], None,
                         ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0), preact=[dev(a) for a in hk])
    for g, r in zip(dx, oracle.row_bwd_dx(w2, dy, preacts=hk)):
        assert_close(host_f64(g.t), r, False, "pair dgelu")


# ------------------------------------------------------------------ sequence-parallel backward

SP_BWD_CASES = [  # p, M, N, K, chunk_m
    (2, 256, 256, 128, 0), (4, 600, 264, 136, 0), (3, 300, 320, 192, 128), (2, 128, 136, 72, 32),
    (4, 192, 256, 64, 16), (8, 1024, 512, 256, 0)]


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K,chunk", SP_BWD_CASES)
def test_ag_matmul_bwd_exact(tp, tile_mode, split_k, p, M, N, K, chunk):
    Mp = M // p
    xs = [ints((Mp, K), 600 + s) for s in range(p)]
    ws = [ints((K, N), 610 + k) for k in range(p)]
    dys = [ints((M, N), 620 + k) for k in range(p)]
    dx = outs([(Mp, K)] * p, True)
    dw = outs([(K, N)] * p, True)
    tp.tp_ag_matmul_bwd([dev(a) for a in xs], [dev(b) for b in ws], [dev(d) for d in dys], [g.t for g in dx],
                        [g.t for g in dw], ws_for(tp, tp.TP_OP_AG_MM_BWD, p, M, N, K, chunk), chunk)
    for g, r in zip(dx, oracle.ag_matmul_bwd_dx(ws, dys)):
        check_exact(g, r, True)
    for g, r in zip(dw, oracle.ag_matmul_bwd_dw(xs, dys)):
        check_exact(g, r, True)


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K,chunk", SP_BWD_CASES)
def test_row_bwd_reducescatter_exact(tp, tile_mode, split_k, p, M, N, K, chunk):
    Mp = M // p
    xs = [ints((M, K), 630 + r) for r in range(p)]
    ws = [ints((K, N), 640 + r) for r in range(p)]
    dys = [ints((Mp, N), 650 + s) for s in range(p)]
    for f32 in (False, True):   # one output dtype per call
        dx = outs([(M, K)] * p, f32)
        dw = outs([(K, N)] * p, f32)
        tp.tp_row_linear_bwd_reducescatter([dev(a) for a in xs], [dev(b) for b in ws], [dev(d) for d in dys],
                                           [g.t for g in dx], [g.t for g in dw],
                                           ws_for(tp, tp.TP_OP_ROW_RS_BWD, p, M, N, K, chunk), chunk_m=chunk)
        for g, r in zip(dx, oracle.row_rs_bwd_dx(ws, dys)):
            check_exact(g, r, f32)
        for g, r in zip(dw, oracle.row_rs_bwd_dw(xs, dys)):
            check_exact(g, r, f32)


@pytest.mark.parametrize("p,M,N,K,chunk", [(4, 512, 256, 192, 0), (2, 128, 136, 64, 32)])
def test_row_bwd_reducescatter_dgelu(tp, split_k, p, M, N, K, chunk):
    Mp = M // p
    ws = [synth.normal_bf16((K, N), 660 + r, sigma=1.0 / np.sqrt(N)) for r in range(p)]
    dys = [synth.normal_bf16((Mp, N), 670 + s) for s in range(p)]
    hs = [synth.normal_bf16((M, K), 680 + r) for r in range(p)]
    dx = outs([(M, K)] * p, False)
    tp.tp_row_linear_bwd_reducescatter(None, [dev(b) for b in ws], [dev(d) for d in dys], [g.t for g in dx], None,
                                       ws_for(tp, tp.TP_OP_ROW_RS_BWD, p, M, N, K, chunk),
                                       preact=[dev(h) for h in hs], chunk_m=chunk)
    for g, r in zip(dx, oracle.row_rs_bwd_dx(ws, dys, preacts=hs)):
        g.check_bands()
        assert_close(host_f64(g.t), r, False, "SP bwd dgelu")


@pytest.mark.parametrize("tile_mode", [1, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K", [(2, 300, 520, 200), (4, 512, 264, 136), (3, 257, 136, 72)])
def test_store_paths_bitwise_identical(tp, tile_mode, p, M, N, K):
    """The staged epilogue leaves shared memory either by TMA store (the
    default wherever the groups' outputs allow it) or by plain 16-byte
    stores; both must write the same bits, including GeLU's H, ragged edges,
    replicas and the AllGather layout's row blocks."""
    import torch
    x = synth.normal_bf16((M, K), 560, 1.0 / np.sqrt(K))
    xs = [synth.normal_bf16((M, K), 561 + r, 1.0 / np.sqrt(K)) for r in range(p)]
    ws = [synth.normal_bf16((K, N), 570 + r) for r in range(p)]
    Mg = M // p * p
    X, XS, W = dev(x), [dev(a) for a in xs], [dev(b) for b in ws]
    XG = [dev(a[:Mg // p]) for a in xs]

    def run():
        bf = dict(dtype=torch.bfloat16, device="cuda")
        y = [torch.empty((M, N), **bf) for _ in range(p)]
        z = [torch.empty((M, N), **bf) for _ in range(p)]
        h = [torch.empty((M, N), **bf) for _ in range(p)]
        g = [torch.empty((Mg, N), **bf) for _ in range(p)]
        gh = [torch.empty((Mg, N), **bf) for _ in range(p)]
        f = torch.empty((M, N), dtype=torch.float32, device="cuda")
        wsp = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0)
        tp.tp_row_linear_fwd_allreduce(XS, W, y, wsp)                      # p replicas
        tp.tp_row_linear_fwd_allreduce(XS, W, [f], ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0))
        tp.tp_col_linear_fwd(X, W, z, ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, 0), epi=tp.TP_EPI_GELU, preact=h)
        tp.tp_ag_matmul(XG, W, g, ws_for(tp, tp.TP_OP_AG_MM, p, Mg, N, K, 0), epi=tp.TP_EPI_GELU, preact=gh)
        torch.cuda.synchronize()
        return [t.clone() for t in y + z + h + g + gh + [f]]

    a = run()
    assert tp.tp_debug_set(tp.TP_DEBUG_TMA_STORE, 0) == tp.TP_OK
    try:
        b = run()
    finally:
        tp.tp_debug_set(tp.TP_DEBUG_TMA_STORE, 1)
    for i, (u, v) in enumerate(zip(a, b)):
        iv = torch.int32 if u.dtype == torch.float32 else torch.int16
        assert torch.equal(u.view(iv), v.view(iv)), f"output {i} differs between the store paths"
    assert_close(host_f64(a[-1]), oracle.row_fwd_allreduce(xs, ws), True, "fp32 AllReduce")


@pytest.fixture
def no_fusion(tp):
    yield
    tp.tp_debug_set(tp.TP_DEBUG_NO_BWD_FUSION, 0)


@pytest.mark.parametrize("tile_mode", [0, 2], indirect=True)
@pytest.mark.parametrize("p,M,N,K", [(2, 2048, 2048, 2048), (3, 300, 264, 136), (4, 512, 256, 192)])
def test_backward_fused_launch_bitwise_and_exact(tp, tile_mode, no_fusion, p, M, N, K):
    """A backward call's dX and dW products may run as one CTA-pair launch
    (where the planner expects it to finish sooner than two); the results
    must equal those of the two separate launches bit for bit, and the
    oracle exactly on integer inputs, for the row backward (with GeLU'), the
    column backward and both sequence-parallel backward calls."""
    import torch
    x = ints((M, K), 600)
    xs = [ints((M, K), 601 + r) for r in range(p)]
    xsh = [ints((M // p, K), 611 + r) for r in range(p)]
    w = [ints((K, N), 621 + r) for r in range(p)]
    dy = ints((M, N), 631)
    dys = [ints((M, N), 641 + r) for r in range(p)]
    dysh = [ints((M // p, N), 651 + r) for r in range(p)]
    f32 = dict(dtype=torch.float32, device="cuda")
    W, DY, DYS, DYSH = [dev(a) for a in w], dev(dy), [dev(a) for a in dys], [dev(a) for a in dysh]
    X, XS, XSH = dev(x), [dev(a) for a in xs], [dev(a) for a in xsh]
    H = [dev(synth.normal_bf16((M, K), 661 + r)) for r in range(p)]

    def run():
        r = {}
        r["row_dx"] = [torch.empty((M, K), **f32) for _ in range(p)]
        r["row_dw"] = [torch.empty((K, N), **f32) for _ in range(p)]
        tp.tp_row_linear_bwd(XS, W, DY, r["row_dx"], r["row_dw"], ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0))
        r["row_dx_gelu"] = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        r["row_dw_bf16"] = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        tp.tp_row_linear_bwd(XS, W, DY, r["row_dx_gelu"], r["row_dw_bf16"],
                             ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0), preact=H)
        r["col_dx"] = [torch.empty((M, K), **f32)]
        r["col_dw"] = [torch.empty((K, N), **f32) for _ in range(p)]
        tp.tp_col_linear_bwd(X, W, DYS, r["col_dx"][0], r["col_dw"], ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0))
        r["ag_dx"] = [torch.empty((M // p, K), **f32) for _ in range(p)]
        r["ag_dw"] = [torch.empty((K, N), **f32) for _ in range(p)]
        tp.tp_ag_matmul_bwd(XSH, W, DYS, r["ag_dx"], r["ag_dw"], ws_for(tp, tp.TP_OP_AG_MM_BWD, p, M, N, K, 0))
        r["rs_dx"] = [torch.empty((M, K), **f32) for _ in range(p)]
        r["rs_dw"] = [torch.empty((K, N), **f32) for _ in range(p)]
        tp.tp_row_linear_bwd_reducescatter(XS, W, DYSH, r["rs_dx"], r["rs_dw"],
                                           ws_for(tp, tp.TP_OP_ROW_RS_BWD, p, M, N, K, 0))
        torch.cuda.synchronize()
        return r

    fused = run()
    assert tp.tp_debug_set(tp.TP_DEBUG_NO_BWD_FUSION, 1) == tp.TP_OK
    sep = run()
    for k in fused:
        for a, b in zip(fused[k], sep[k]):
            iv = torch.int32 if a.dtype == torch.float32 else torch.int16
            assert torch.equal(a.view(iv), b.view(iv)), f"{k}: fused and separate launches differ"
    refs = {"row_dx": oracle.row_bwd_dx(w, dy), "row_dw": oracle.row_bwd_dw(xs, dy),
            "col_dx": [oracle.col_bwd_dx(w, dys)], "col_dw": oracle.col_bwd_dw(x, dys),
            "ag_dx": oracle.ag_matmul_bwd_dx(w, dys), "ag_dw": oracle.ag_matmul_bwd_dw(xsh, dys),
            "rs_dx": oracle.row_rs_bwd_dx(w, dysh), "rs_dw": oracle.row_rs_bwd_dw(xs, dysh)}
    for k, ref in refs.items():
        for a, r in zip(fused[k], ref):
            assert np.array_equal(host_f64(a), r), f"{k}: not exact"


def test_cuda_graph_capture_replays_bitwise(tp):
    """Calls can be captured in a CUDA graph (after one eager call, which sets
    each kernel's attributes) and replayed: each replay reads the inputs'
    current contents, and gives the eager call's bits.  Covers the split-K
    second stage (the worked example), ReduceScatter, the CTA-pair kernel with
    last-wave slices, GeLU and the TMA-store epilogue."""
    import torch
    p, M, N, K = 2, 128, 2048, 1024
    p2, M2, N2, K2 = 2, 2048, 2560, 512
    x = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    w = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    x2 = [torch.empty((M2, K2), dtype=torch.bfloat16, device="cuda") for _ in range(p2)]
    w2 = [torch.empty((K2, N2), dtype=torch.bfloat16, device="cuda") for _ in range(p2)]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ys = [torch.empty((M // p, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    z = [torch.empty((M2, N2), dtype=torch.bfloat16, device="cuda") for _ in range(p2)]
    h = [torch.empty((M2, N2), dtype=torch.bfloat16, device="cuda") for _ in range(p2)]
    y2 = torch.empty((M2, N2), dtype=torch.float32, device="cuda")
    ws = max((ws_for(tp, op, pp, mm, nn, kk, c) for op, pp, mm, nn, kk, c in
              [(tp.TP_OP_ROW_AR, p, M, N, K, 32), (tp.TP_OP_ROW_RS, p, M, N, K, 32),
               (tp.TP_OP_COL_FWD, p2, M2, N2, K2, 0), (tp.TP_OP_ROW_AR, p2, M2, N2, K2, 0)]), key=lambda t: t.numel())

    def fill(seed):
        for i, t in enumerate(x + w):
            t.copy_(dev(synth.normal_bf16(tuple(t.shape), seed + i, 0.05)))
        for i, t in enumerate(x2 + w2):
            t.copy_(dev(ints(tuple(t.shape), seed + 50 + i)))

    def calls():
        tp.tp_row_linear_fwd_allreduce(x, w, [y], ws, 32)
        tp.tp_row_linear_fwd_reducescatter(x, w, ys, ws, 32)
        tp.tp_col_linear_fwd(x2[0], w2, z, ws, epi=tp.TP_EPI_GELU, preact=h)
        tp.tp_row_linear_fwd_allreduce(x2, w2, [y2], ws)

    def outputs():
        return [t.clone() for t in [y, *ys, *z, *h, y2]]

    fill(700)
    calls()                      # eager: kernel attributes set, caches filled
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            calls()
    torch.cuda.current_stream().wait_stream(s)
    for seed in (710, 720):
        fill(seed)
        calls()
        torch.cuda.synchronize()
        want = outputs()
        for t in [y, *ys, *z, *h, y2]:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(outputs(), want):
            iv = torch.int32 if a.dtype == torch.float32 else torch.int16
            assert torch.equal(a.view(iv), b.view(iv)), "graph replay differs from the eager calls"
    assert tp.tp_get_device_status(ws) == tp.TP_OK
    assert np.array_equal(host_f64(y2), oracle.row_fwd_allreduce([host_bits(t) for t in x2], [host_bits(t) for t in w2]))


def test_alternating_contraction_direction_exact(tp):
    """A contraction of 8192 or deeper on the CTA-pair kernel runs the whole
    tiles of every other wave last k-block first (rank p-1's segment first).
    Here 16 x 11 pair tiles are 2.3 waves over 4 x 2048: on integer inputs
    every partial sum stays exact, so the bf16 AllReduce and the column
    backward's fused dX must round exactly the oracle's sums, whichever order
    a tile took, and the ReduceScatter slices must equal the AllReduce rows."""
    import torch
    p, M, N, K = 4, 4096, 2816, 2048
    xs = [ints((M, K), 700 + r) for r in range(p)]
    ws = [ints((K, N), 710 + r) for r in range(p)]
    X, W = [dev(a) for a in xs], [dev(b) for b in ws]
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tp.tp_row_linear_fwd_allreduce(X, W, [y], ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0))
    assert np.array_equal(host_bits(y), oracle.round_bf16(oracle.row_fwd_allreduce(xs, ws)))
    ys = [torch.empty((M // p, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    tp.tp_row_linear_fwd_reducescatter(X, W, ys, ws_for(tp, tp.TP_OP_ROW_RS, p, M, N, K, 0))
    assert torch.equal(torch.cat(ys).view(torch.int16), y.view(torch.int16))
    # column backward: dX = sum_k dY_k . A_k^T over 4 x 2048 = 8192, 16 x 16
    # pair tiles (3.4 waves; waves 1 and 3 reversed, the last one in slices)
    N, K = 2048, 4096
    wc = [ints((K, N), 760 + k) for k in range(p)]
    dys = [ints((M, N), 720 + k) for k in range(p)]
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    tp.tp_col_linear_bwd(None, [dev(b) for b in wc], [dev(d) for d in dys], dx, None,
                         ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0))
    assert np.array_equal(host_bits(dx), oracle.round_bf16(oracle.col_bwd_dx(wc, dys)))


def test_single_band_weight_gradient_exact(tp):
    """dW_r = X_r^T . dY where the p X_r shards (4 x 2048 x 4608 bf16, 75 MB)
    exceed the L2 budget and the shared dY (38 MB) does not: the planner
    rasters all 16 N-tiles as one band instead of two bands of 8, so each
    X_r panel is streamed once.  The order of the tiles must not change the
    result: exact against the oracle on integer inputs (sums of 4608
    products stay below 2**24)."""
    import torch
    p, M, N, K = 4, 4608, 4096, 2048
    xs = [ints((M, K), 730 + r) for r in range(p)]
    w = [ints((K, N), 740 + r) for r in range(p)]
    dy = ints((M, N), 750)
    dw = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    tp.tp_row_linear_bwd([dev(a) for a in xs], [dev(b) for b in w], dev(dy), None, dw,
                         ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0))
    for g, r in zip(dw, oracle.row_bwd_dw(xs, dy)):
        assert np.array_equal(host_bits(g), oracle.round_bf16(r))


def test_long_backward_fused_launch_bitwise(tp, no_fusion):
    """FC2's backward at the MLP block's size (p = 4, M = K = N = 4096): dZ_k
    = dY . W_k^T * GeLU'(H_k) and dW_k = Z_k^T . dY are 1024 pair tiles each
    (13.5 waves), which the planner runs as one launch of 27 waves.  That
    launch must give the bits of the two separate launches, and sampled rows
    of both products must equal the oracle on integer inputs (sums of 4096
    products of values in [-4, 4] are exact).  GeLU' uses bf16 H."""
    import torch
    p, M, N, K = 4, 4096, 4096, 4096
    xs = [ints((M, K), 770 + r) for r in range(p)]
    w = [ints((K, N), 780 + r) for r in range(p)]
    dy = ints((M, N), 790)
    X, W, DY = [dev(a) for a in xs], [dev(b) for b in w], dev(dy)
    ws = ws_for(tp, tp.TP_OP_ROW_BWD, p, M, N, K, 0)

    def run(preact):
        dx = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        dw = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
        tp.tp_row_linear_bwd(X, W, DY, dx, dw, ws, preact=preact)
        torch.cuda.synchronize()
        assert tp.tp_get_device_status(ws) == tp.TP_OK
        return dx, dw

    H = [dev(synth.normal_bf16((M, K), 800 + r)) for r in range(p)]
    fused = [run(None), run(H)]
    assert tp.tp_debug_set(tp.TP_DEBUG_NO_BWD_FUSION, 1) == tp.TP_OK
    sep = [run(None), run(H)]
    for (fx, fw), (sx, sw) in zip(fused, sep):
        for a, b in zip(fx + fw, sx + sw):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "fused and separate launches differ"
    rows = np.array([0, 1, 255, 256, 1023, 2048, 3071, 4095])
    dx, dw = fused[0]
    ref_dx = oracle.row_bwd_dx(w, dy[rows])                          # dY . W_r^T on the sampled rows
    ref_dw = oracle.row_bwd_dw([x[:, rows] for x in xs], dy)          # X_r^T . dY on the sampled rows
    for r in range(p):
        assert np.array_equal(host_bits(dx[r])[rows], oracle.round_bf16(ref_dx[r]))
        assert np.array_equal(host_bits(dw[r])[rows], oracle.round_bf16(ref_dw[r]))


@pytest.fixture
def k_forward(tp):
    yield
    tp.tp_debug_set(tp.TP_DEBUG_K_ALTERNATE, 1)


def test_alternating_direction_is_taken_and_within_tolerance(tp, k_forward):
    """The reversed waves really run: on normal-valued inputs the planned
    AllReduce over 4 x 2048 (16 x 11 pair tiles, 2.3 waves) differs in its
    rounding from the same call with every tile forward
    (TP_DEBUG_K_ALTERNATE = 0), only in tiles of the second wave, while
    both stay within the bf16 tolerance of the oracle; each order is
    reproducible bit for bit."""
    import torch
    p, M, N, K = 4, 4096, 2816, 2048
    xs = [synth.normal_bf16((M, K), synth.seed_for(810, r), 1.0 / np.sqrt(p * K)) for r in range(p)]
    ws = [synth.normal_bf16((K, N), synth.seed_for(811, r)) for r in range(p)]
    X, W = [dev(a) for a in xs], [dev(b) for b in ws]
    wsp = ws_for(tp, tp.TP_OP_ROW_AR, p, M, N, K, 0)

    def run():
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        tp.tp_row_linear_fwd_allreduce(X, W, [y], wsp)
        return host_bits(y)

    planned = [run(), run()]
    assert tp.tp_debug_set(tp.TP_DEBUG_K_ALTERNATE, 0) == tp.TP_OK
    forward = [run(), run()]
    assert np.array_equal(planned[0], planned[1]) and np.array_equal(forward[0], forward[1])
    diff = planned[0] != forward[0]
    assert diff.any(), "no tile ran in the other order"
    # 256 x 256 tiles in which the two differ: only whole tiles of odd waves reverse
    tiles = {(int(i) // 256, int(j) // 256) for i, j in zip(*np.nonzero(diff))}
    assert len(tiles) <= 76
    ref = oracle.row_fwd_allreduce(xs, ws)
    for b in (planned[0], forward[0]):
        got = b.astype(np.uint32) << np.uint32(16)
        assert_close(got.view(np.float32).astype(np.float64), ref, False, "AllReduce")


def test_narrow_band_column_launches_exact(tp):
    """Where the shared operand X stays in L2 (column forward Y_k = X . A_k
    and dA_k = X^T . dY_k, p = 4 groups, 16 row tiles of 256), the planner
    rasters bands of 2 N-tiles instead of 8.  Only the tile order changes:
    bf16 outputs on integer inputs must round the oracle's exact sums."""
    import torch
    p, M, K, N = 4, 4096, 4096, 1024
    x = ints((M, K), 820)
    w = [ints((K, N), 821 + k) for k in range(p)]
    X, W = dev(x), [dev(b) for b in w]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    tp.tp_col_linear_fwd(X, W, ys, ws_for(tp, tp.TP_OP_COL_FWD, p, M, N, K, 0))
    for g, r in zip(ys, oracle.col_fwd(x, w)[0]):
        assert np.array_equal(host_bits(g), oracle.round_bf16(r))
    dys = [ints((M, N), 830 + k) for k in range(p)]
    dw = [torch.empty((K, N), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    tp.tp_col_linear_bwd(X, W, [dev(d) for d in dys], None, dw, ws_for(tp, tp.TP_OP_COL_BWD, p, M, N, K, 0))
    for g, r in zip(dw, oracle.col_bwd_dw(x, dys)):
        assert np.array_equal(host_bits(g), oracle.round_bf16(r))
