"""Host-side argument checks of the Python binding, on CPU.

The C ABI takes one M, N, K for all shards and cannot see buffer sizes, so
the binding checks every tensor's shape, dtype, layout and device before it
calls the library.  Here the library is replaced by a recorder and the
"current device" by the CPU tensors' device index (-1): every entry point
must pass the argument patterns the autograd layer and the tests use, and
must refuse a wrong shard, output, bias or dtype before anything reaches the
library."""
import pytest
import torch

import gemm_reduce_fusion_gb300 as tp

BF, F32 = torch.bfloat16, torch.float32


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("tp_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append(name)
            return tp.TP_OK
        setattr(self, name, fn)
        return fn


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(tp, "_lib", rec)
    monkeypatch.setattr(tp, "_current_device", lambda: -1)
    return rec


def z(*shape, dtype=BF):
    return torch.zeros(shape, dtype=dtype)


def zs(n, *shape, dtype=BF):
    return [z(*shape, dtype=dtype) for _ in range(n)]


WS = torch.zeros(256, dtype=torch.uint8)
p, M, N, K = 2, 8, 16, 24


def test_every_entry_point_accepts_its_documented_shapes(lib):
    tp.tp_row_linear_fwd_allreduce(zs(p, M, K), zs(p, K, N), [z(M, N)], WS, stream=0)
    tp.tp_row_linear_fwd_allreduce(zs(p, M, K), zs(p, K, N), zs(p, M, N, dtype=F32), WS, stream=0, bias=z(N))
    tp.tp_row_linear_fwd_reducescatter(zs(p, M, K), zs(p, K, N), zs(p, M // p, N), WS, stream=0, bias=z(N))
    tp.tp_col_linear_fwd(z(M, K), zs(p, K, N), zs(p, M, N), WS, stream=0)
    tp.tp_col_linear_fwd(z(M, K), zs(p, K, N), zs(p, M, N), WS, epi=tp.TP_EPI_GELU, preact=zs(p, M, N),
                         stream=0, bias=zs(p, N))
    tp.tp_col_linear_bwd(z(M, K), zs(p, K, N), zs(p, M, N), z(M, K), zs(p, K, N), WS, stream=0, db=zs(p, N))
    tp.tp_col_linear_bwd(None, zs(p, K, N), zs(p, M, N), z(M, K), None, WS, stream=0)
    tp.tp_col_linear_bwd(z(M, K), zs(p, K, N), zs(p, M, N), None, zs(p, K, N), WS, stream=0)
    tp.tp_row_linear_bwd(zs(p, M, K), zs(p, K, N), z(M, N), zs(p, M, K), zs(p, K, N), WS,
                         preact=zs(p, M, K), stream=0, db=z(N))
    tp.tp_row_linear_bwd(None, zs(p, K, N), z(M, N), zs(p, M, K), None, WS, stream=0)
    tp.tp_ag_matmul(zs(p, M // p, K), zs(p, K, N), zs(p, M, N), WS, x_gathered=z(M, K), epi=tp.TP_EPI_GELU,
                    preact=zs(p, M, N), stream=0, bias=zs(p, N))
    tp.tp_ag_matmul_bwd(zs(p, M // p, K), zs(p, K, N), zs(p, M, N), zs(p, M // p, K), zs(p, K, N), WS,
                        stream=0, db=zs(p, N))
    tp.tp_ag_matmul_bwd(None, zs(p, K, N), zs(p, M, N), zs(p, M // p, K), None, WS, stream=0)
    tp.tp_row_linear_bwd_reducescatter(zs(p, M, K), zs(p, K, N), zs(p, M // p, N), zs(p, M, K), zs(p, K, N),
                                       WS, preact=zs(p, M, K), stream=0, db=z(N))
    tp.tp_row_linear_fwd_unfused(zs(p, M, K), zs(p, K, N), z(M, N), WS, stream=0)
    tp.tp_row_linear_fwd_allreduce_noalloc(zs(p, M, K), zs(p, K, N), [z(M, N)], stream=0)
    # empty extents (M == 0, K == 0) are shapes like any other
    tp.tp_row_linear_fwd_allreduce(zs(p, 0, K), zs(p, K, N), [z(0, N)], WS, stream=0)
    tp.tp_row_linear_fwd_allreduce(zs(p, 5, 0), zs(p, 0, N), [z(5, N)], WS, stream=0)
    assert len(lib.calls) == 18


@pytest.mark.parametrize("case", [
    "short shard", "wide weight", "missing weight", "wrong output", "replica count", "bias length",
    "rs slice", "col preact", "col bias count", "bwd dw", "row bwd preact", "ag gathered", "unfused y"])
def test_wrong_shapes_are_refused_before_the_library(lib, case):
    x, w = zs(p, M, K), zs(p, K, N)
    calls = {
        "short shard": lambda: tp.tp_row_linear_fwd_allreduce([z(M, K), z(M - 1, K)], w, [z(M, N)], WS, stream=0),
        "wide weight": lambda: tp.tp_row_linear_fwd_allreduce(x, [z(K, N), z(K, N + 8)], [z(M, N)], WS, stream=0),
        "missing weight": lambda: tp.tp_row_linear_fwd_allreduce(x, w[:1], [z(M, N)], WS, stream=0),
        "wrong output": lambda: tp.tp_row_linear_fwd_allreduce(x, w, [z(M, N - 8)], WS, stream=0),
        "replica count": lambda: tp.tp_row_linear_fwd_allreduce(zs(3, M, K), zs(3, K, N), zs(2, M, N), WS,
                                                                stream=0),
        "bias length": lambda: tp.tp_row_linear_fwd_allreduce(x, w, [z(M, N)], WS, stream=0, bias=z(N + 8)),
        "rs slice": lambda: tp.tp_row_linear_fwd_reducescatter(x, w, zs(p, M, N), WS, stream=0),
        "col preact": lambda: tp.tp_col_linear_fwd(z(M, K), w, zs(p, M, N), WS, epi=tp.TP_EPI_GELU,
                                                   preact=zs(p, M, K), stream=0),
        "col bias count": lambda: tp.tp_col_linear_fwd(z(M, K), w, zs(p, M, N), WS, stream=0, bias=zs(1, N)),
        "bwd dw": lambda: tp.tp_col_linear_bwd(z(M, K), w, zs(p, M, N), None, zs(p, N, K), WS, stream=0),
        "row bwd preact": lambda: tp.tp_row_linear_bwd(None, w, z(M, N), zs(p, M, K), None, WS,
                                                       preact=zs(p, M, N), stream=0),
        "ag gathered": lambda: tp.tp_ag_matmul(zs(p, M // p, K), w, zs(p, M, N), WS, x_gathered=z(M // p, K),
                                               stream=0),
        "unfused y": lambda: tp.tp_row_linear_fwd_unfused(x, w, z(M // p, N), WS, stream=0),
    }
    with pytest.raises(ValueError):
        calls[case]()
    assert lib.calls == []


def test_wrong_dtype_layout_and_device_are_refused(lib, monkeypatch):
    x, w, y = zs(p, M, K), zs(p, K, N), [z(M, N)]
    with pytest.raises(TypeError, match="bfloat16"):
        tp.tp_row_linear_fwd_allreduce([z(M, K, dtype=F32), x[1]], w, y, WS, stream=0)
    with pytest.raises(TypeError, match="bfloat16"):
        tp.tp_row_linear_bwd(None, w, z(M, N), zs(p, M, K), None, WS, preact=zs(p, M, K, dtype=F32), stream=0)
    with pytest.raises(ValueError, match="contiguous"):
        tp.tp_row_linear_fwd_allreduce([z(K, M).t(), x[1]], w, y, WS, stream=0)
    # tensors on another device than the one the call runs on
    monkeypatch.setattr(tp, "_current_device", lambda: 0)
    with pytest.raises(TypeError, match="cuda:0"):
        tp.tp_row_linear_fwd_allreduce(x, w, y, WS, stream=0)
    assert lib.calls == []
