"""The autograd wrappers against the CPU oracle: forward outputs and every
gradient autograd hands back, for the column, row, MLP and sequence-parallel
layers.  The output gradients are seeded normals passed to
``torch.autograd.backward``; each gradient is compared with the oracle's
backward on the bf16 values the library saved or consumed.  Tolerance:
max|d|/max|ref| <= 5e-3 (bf16 results)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_close, dev, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ag():
    import gemm_reduce_fusion_gb300.autograd as ag
    return ag


def leaf(b16):
    return dev(b16).clone().requires_grad_(True)


def normals(shape, c, t, sigma=1.0):
    return synth.normal_bf16(shape, synth.seed_for(c, t), sigma)


@pytest.mark.parametrize("p,M,K,N", [(2, 300, 136, 264), (4, 256, 512, 128)])
def test_column_parallel_linear(ag, p, M, K, N):
    import torch
    x = normals((M, K), 70, 0)
    w = [normals((K, N), 70, 1 + k, 0.05) for k in range(p)]
    g = [normals((M, N), 70, 9 + k) for k in range(p)]
    X, W = leaf(x), [leaf(a) for a in w]
    Y = ag.column_parallel_linear(X, W)
    ref, _ = oracle.col_fwd(x, w)
    for k in range(p):
        assert_close(host_f64(Y[k]), ref[k], False, f"Y_{k}")
    torch.autograd.backward(Y, [dev(a) for a in g])
    assert_close(host_f64(X.grad), oracle.col_bwd_dx(w, g), False, "dX")
    for k, r in enumerate(oracle.col_bwd_dw(x, g)):
        assert_close(host_f64(W[k].grad), r, False, f"dA_{k}")


@pytest.mark.parametrize("p,M,K,N", [(2, 300, 136, 264), (4, 64, 512, 256)])
def test_row_parallel_linear(ag, p, M, K, N):
    import torch
    xs = [normals((M, K), 71, r) for r in range(p)]
    w = [normals((K, N), 71, 8 + r, 0.05) for r in range(p)]
    g = normals((M, N), 71, 20)
    X, W = [leaf(a) for a in xs], [leaf(a) for a in w]
    Y = ag.row_parallel_linear(X, W)
    assert_close(host_f64(Y), oracle.row_fwd_allreduce(xs, w), False, "Y")
    Y.backward(dev(g))
    for r, ref in enumerate(oracle.row_bwd_dx(w, g)):
        assert_close(host_f64(X[r].grad), ref, False, f"dX_{r}")
    for r, ref in enumerate(oracle.row_bwd_dw(xs, g)):
        assert_close(host_f64(W[r].grad), ref, False, f"dA_{r}")


def test_parallel_mlp_module(ag):
    """The MLP block as a module built from full weights: its shards are the
    contiguous column blocks of W1 and row blocks of W2."""
    import torch
    p, M, h, ffn = 4, 256, 256, 1024
    nk = ffn // p
    x = normals((M, h), 72, 0)
    w1 = normals((h, ffn), 72, 1, 0.05)
    w2 = normals((ffn, h), 72, 2, 0.05)
    g = normals((M, h), 72, 3)
    mlp = ag.ParallelMLP(dev(w1), dev(w2), p)
    X = leaf(x)
    Y = mlp(X)
    w1s = [np.ascontiguousarray(w1[:, k * nk:(k + 1) * nk]) for k in range(p)]
    w2s = [np.ascontiguousarray(w2[k * nk:(k + 1) * nk]) for k in range(p)]
    for k in range(p):
        assert np.array_equal(host_bits(mlp.w1[k]), w1s[k]) and np.array_equal(host_bits(mlp.w2[k]), w2s[k])
    # chained oracle: bf16 intermediates at the same boundaries as the library
    zr, hr = oracle.col_fwd(x, w1s, apply_gelu=True)
    zb = [oracle.round_bf16(a) for a in zr]
    hb = [oracle.round_bf16(a) for a in hr]
    assert_close(host_f64(Y), oracle.row_fwd_allreduce(zb, w2s), False, "Y")
    Y.backward(dev(g))
    dz = oracle.row_bwd_dx(w2s, g, preacts=hb)
    dzb = [oracle.round_bf16(a) for a in dz]
    for k, ref in enumerate(oracle.row_bwd_dw(zb, g)):
        assert_close(host_f64(mlp.w2[k].grad), ref, False, f"dW2_{k}")
    for k, ref in enumerate(oracle.col_bwd_dw(x, dzb)):
        assert_close(host_f64(mlp.w1[k].grad), ref, False, f"dW1_{k}")
    assert_close(host_f64(X.grad), oracle.col_bwd_dx(w1s, dzb), False, "dX")
    assert torch.cuda.is_available()


def test_row_module_and_column_module_chain(ag):
    """Column then row layer (no activation) chained through autograd equals
    the unsharded two-layer product and its gradients."""
    import torch
    p, M, h, f = 2, 128, 128, 256
    x = normals((M, h), 73, 0)
    w1 = normals((h, f), 73, 1, 0.05)
    w2 = normals((f, h), 73, 2, 0.05)
    g = normals((M, h), 73, 3)
    col = ag.ColumnParallelLinear(dev(w1), p)
    row = ag.RowParallelLinear(dev(w2), p)
    X = leaf(x)
    Y = row(list(col(X)))
    fs = f // p
    w1s = [np.ascontiguousarray(w1[:, k * fs:(k + 1) * fs]) for k in range(p)]
    w2s = [np.ascontiguousarray(w2[k * fs:(k + 1) * fs]) for k in range(p)]
    hb = [oracle.round_bf16(a) for a in oracle.col_fwd(x, w1s)[0]]
    assert_close(host_f64(Y), oracle.row_fwd_allreduce(hb, w2s), False, "Y")
    Y.backward(dev(g))
    dhb = [oracle.round_bf16(a) for a in oracle.row_bwd_dx(w2s, g)]
    assert_close(host_f64(X.grad), oracle.col_bwd_dx(w1s, dhb), False, "dX")
    for k, ref in enumerate(oracle.row_bwd_dw(hb, g)):
        assert_close(host_f64(row.weights[k].grad), ref, False, f"dW2_{k}")
    for k, ref in enumerate(oracle.col_bwd_dw(x, dhb)):
        assert_close(host_f64(col.weights[k].grad), ref, False, f"dW1_{k}")
    assert torch.is_tensor(Y)


def test_sequence_parallel_layers(ag):
    """AllGather+MatMul then MatMul+ReduceScatter as separate functions, and
    the fused sequence-parallel MLP module, against the oracle."""
    import torch
    p, Mp, h, nk = 4, 64, 128, 96
    M = Mp * p
    xs = [normals((Mp, h), 74, s) for s in range(p)]
    w1 = [normals((h, nk), 74, 4 + k, 0.05) for k in range(p)]
    w2 = [normals((nk, h), 74, 8 + k, 0.05) for k in range(p)]
    gs = [normals((Mp, h), 74, 12 + s) for s in range(p)]
    # separate layers, no activation
    X, W1, W2 = [leaf(a) for a in xs], [leaf(a) for a in w1], [leaf(a) for a in w2]
    H = ag.allgather_column_parallel_linear(X, W1)
    Y = ag.row_parallel_linear_reducescatter(list(H), W2)
    hr, _, _ = oracle.ag_matmul(xs, w1)
    hb = [oracle.round_bf16(a) for a in hr]
    for s, ref in enumerate(oracle.row_fwd_reducescatter(hb, w2)):
        assert_close(host_f64(Y[s]), ref, False, f"Y_{s}")
    torch.autograd.backward(Y, [dev(a) for a in gs])
    dhb = [oracle.round_bf16(a) for a in oracle.row_rs_bwd_dx(w2, gs)]
    for r, ref in enumerate(oracle.row_rs_bwd_dw(hb, gs)):
        assert_close(host_f64(W2[r].grad), ref, False, f"dW2_{r}")
    for s, ref in enumerate(oracle.ag_matmul_bwd_dx(w1, dhb)):
        assert_close(host_f64(X[s].grad), ref, False, f"dX_{s}")
    for k, ref in enumerate(oracle.ag_matmul_bwd_dw(xs, dhb)):
        assert_close(host_f64(W1[k].grad), ref, False, f"dW1_{k}")
    # the sequence-parallel MLP module (GeLU between the two layers)
    mlp = ag.ParallelMLP(dev(np.hstack(w1)), dev(np.vstack(w2)), p, sequence_parallel=True)
    X2 = [leaf(a) for a in xs]
    Y2 = mlp(X2)
    zr, hr2, _ = oracle.ag_matmul(xs, w1, apply_gelu=True)
    zb = [oracle.round_bf16(a) for a in zr]
    hb2 = [oracle.round_bf16(a) for a in hr2]
    for s, ref in enumerate(oracle.row_fwd_reducescatter(zb, w2)):
        assert_close(host_f64(Y2[s]), ref, False, f"MLP Y_{s}")
    torch.autograd.backward(Y2, [dev(a) for a in gs])
    dzb = [oracle.round_bf16(a) for a in oracle.row_rs_bwd_dx(w2, gs, preacts=hb2)]
    for s, ref in enumerate(oracle.ag_matmul_bwd_dx(w1, dzb)):
        assert_close(host_f64(X2[s].grad), ref, False, f"MLP dX_{s}")
    for k, ref in enumerate(oracle.ag_matmul_bwd_dw(xs, dzb)):
        assert_close(host_f64(mlp.w1[k].grad), ref, False, f"MLP dW1_{k}")
    for r, ref in enumerate(oracle.row_rs_bwd_dw(zb, gs)):
        assert_close(host_f64(mlp.w2[r].grad), ref, False, f"MLP dW2_{r}")


def test_mlp_with_biases_plain_and_sequence_parallel(ag):
    """The MLP block with b1 (split with FC1's columns, before the GeLU) and
    b2 (added once after the reduction), its bias gradients db1_k = row sums
    of dH_k and db2 = row sums of dY; then the sequence-parallel module."""
    import torch
    p, M, h, ffn = 2, 256, 128, 512
    nk = ffn // p
    x = normals((M, h), 75, 0)
    w1 = normals((h, ffn), 75, 1, 0.05)
    w2 = normals((ffn, h), 75, 2, 0.05)
    b1 = normals((ffn,), 75, 3)
    b2 = normals((h,), 75, 4)
    g = normals((M, h), 75, 5)
    w1s = [np.ascontiguousarray(w1[:, k * nk:(k + 1) * nk]) for k in range(p)]
    w2s = [np.ascontiguousarray(w2[k * nk:(k + 1) * nk]) for k in range(p)]
    b1s = [np.ascontiguousarray(b1[k * nk:(k + 1) * nk]) for k in range(p)]
    zr, hr = oracle.col_fwd(x, w1s, apply_gelu=True, biases=b1s)
    zb = [oracle.round_bf16(a) for a in zr]
    hb = [oracle.round_bf16(a) for a in hr]
    dzb = [oracle.round_bf16(a) for a in oracle.row_bwd_dx(w2s, g, preacts=hb)]
    for sp in (False, True):
        mlp = ag.ParallelMLP(dev(w1), dev(w2), p, b1=dev(b1), b2=dev(b2), sequence_parallel=sp)
        if not sp:
            X = leaf(x)
            Y = mlp(X)
            assert_close(host_f64(Y), oracle.row_fwd_allreduce(zb, w2s, bias=b2), False, "Y")
            Y.backward(dev(g))
            assert_close(host_f64(X.grad), oracle.col_bwd_dx(w1s, dzb), False, "dX")
        else:
            Mp = M // p
            X = [leaf(np.ascontiguousarray(x[s * Mp:(s + 1) * Mp])) for s in range(p)]
            Y = mlp(X)
            ref = oracle.row_fwd_allreduce(zb, w2s, bias=b2)
            for s in range(p):
                assert_close(host_f64(Y[s]), ref[s * Mp:(s + 1) * Mp], False, f"Y_{s}")
            torch.autograd.backward(Y, [dev(np.ascontiguousarray(g[s * Mp:(s + 1) * Mp])) for s in range(p)])
            dxr = oracle.col_bwd_dx(w1s, dzb)
            for s in range(p):
                assert_close(host_f64(X[s].grad), dxr[s * Mp:(s + 1) * Mp], False, f"dX_{s}")
        assert_close(host_f64(mlp.b2.grad), oracle.bias_grad(g), False, "db2")
        for k in range(p):
            assert_close(host_f64(mlp.b1[k].grad), oracle.bias_grad(dzb[k]), False, f"db1_{k}")
        for k, ref in enumerate(oracle.row_bwd_dw(zb, g)):
            assert_close(host_f64(mlp.w2[k].grad), ref, False, f"dW2_{k}")


def test_linear_modules_with_bias(ag):
    import torch
    p, M, h, f = 4, 128, 128, 256
    x = normals((M, h), 76, 0)
    w1 = normals((h, f), 76, 1, 0.05)
    b1 = normals((f,), 76, 2)
    w2 = normals((f, h), 76, 3, 0.05)
    b2 = normals((h,), 76, 4)
    g = normals((M, h), 76, 5)
    col = ag.ColumnParallelLinear(dev(w1), p, bias=dev(b1))
    row = ag.RowParallelLinear(dev(w2), p, bias=dev(b2))
    X = leaf(x)
    Y = row(list(col(X)))
    fs = f // p
    w1s = [np.ascontiguousarray(w1[:, k * fs:(k + 1) * fs]) for k in range(p)]
    b1s = [np.ascontiguousarray(b1[k * fs:(k + 1) * fs]) for k in range(p)]
    w2s = [np.ascontiguousarray(w2[k * fs:(k + 1) * fs]) for k in range(p)]
    hb = [oracle.round_bf16(a) for a in oracle.col_fwd(x, w1s, biases=b1s)[0]]
    assert_close(host_f64(Y), oracle.row_fwd_allreduce(hb, w2s, bias=b2), False, "Y")
    Y.backward(dev(g))
    dhb = [oracle.round_bf16(a) for a in oracle.row_bwd_dx(w2s, g)]
    assert_close(host_f64(row.bias.grad), oracle.bias_grad(g), False, "db2")
    for k in range(p):
        assert_close(host_f64(col.biases[k].grad), oracle.bias_grad(dhb[k]), False, f"db1_{k}")
    assert_close(host_f64(X.grad), oracle.col_bwd_dx(w1s, dhb), False, "dX")
    assert torch.is_tensor(Y)


def test_rejects_non_bf16(ag):
    import torch
    x = torch.zeros((16, 16), dtype=torch.float32, device="cuda")
    w = [torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")]
    with pytest.raises(TypeError):
        ag.column_parallel_linear(x, w)
