"""Pins of the CPU oracle against things other than itself (CPU only).

* brute force: pure-Python triple loops on tiny shapes (the 4 x 6, p = 2
  layer of the TP tutorial §5.3) and exact int64 products on larger
  integer-valued inputs, built from the *unsharded* layer and sliced the way
  the pages define the shards;
* closed forms: GeLU values from the normal CDF table, GeLU' against a
  central difference, the chunk-timeline formula and the page's printed
  timeline, the collective-volume factors and byte counts the pages print;
* planted mistakes: deliberately broken copies of oracle functions must fail
  the same pins, which shows the pins can see a dropped term, a wrong sign,
  a transposed operand or a misrouted slice.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _ints(shape, seed, bound=4):
    return synth.integer_bf16(shape, seed, bound)


def _as_int(b16):
    v = oracle.widen(b16)
    assert np.all(v == np.round(v))
    return v.astype(np.int64)


def _brute(a, b):
    """Textbook triple loop on Python ints."""
    m, k = len(a), len(a[0])
    n = len(b[0])
    assert len(b) == k
    return [[sum(int(a[i][t]) * int(b[t][j]) for t in range(k)) for j in range(n)] for i in range(m)]


def _shard_cols(full, p):
    n = full.shape[1] // p
    return [np.ascontiguousarray(full[:, k * n:(k + 1) * n]) for k in range(p)]


def _shard_rows(full, p):
    n = full.shape[0] // p
    return [np.ascontiguousarray(full[k * n:(k + 1) * n]) for k in range(p)]


# --------------------------------------------------------------- invariant checks
# Each returns True when the given implementation satisfies the pin; the
# planted-mistake test below feeds them broken implementations.

def check_row_fwd(row_fwd, p, m, k, n, seed):
    x = _ints((m, k * p), seed)
    a = _ints((k * p, n), seed + 1)
    xs = _shard_cols(x, p)            # X_k = X[:, k*in/p:(k+1)*in/p]
    ws = _shard_rows(a, p)            # A_k = A[k*in/p:(k+1)*in/p, :]
    want = _as_int(x) @ _as_int(a)    # unsharded layer, exact
    got = row_fwd(xs, ws)
    return got.shape == want.shape and np.array_equal(got, want.astype(np.float64))


def check_row_rs(row_rs, p, m, k, n, seed):
    x = _ints((m, k * p), seed)
    a = _ints((k * p, n), seed + 1)
    want = _as_int(x) @ _as_int(a)
    got = row_rs(_shard_cols(x, p), _shard_rows(a, p))
    mp = m // p
    return len(got) == p and all(
        np.array_equal(got[j], want[j * mp:(j + 1) * mp].astype(np.float64)) for j in range(p))


def check_col_fwd(col_fwd, p, m, k, n, seed):
    x = _ints((m, k), seed)
    a = _ints((k, n * p), seed + 1)
    want = _as_int(x) @ _as_int(a)
    ys, _ = col_fwd(x, _shard_cols(a, p))  # A_k = A[:, k*out/p:(k+1)*out/p]
    return np.array_equal(np.hstack(ys), want.astype(np.float64))


def check_col_bwd_dx(col_bwd_dx, p, m, k, n, seed):
    a = _ints((k, n * p), seed)
    dy = _ints((m, n * p), seed + 1)
    want = _as_int(dy) @ _as_int(a).T   # gradient of the unsharded layer
    got = col_bwd_dx(_shard_cols(a, p), _shard_cols(dy, p))
    return got.shape == want.shape and np.array_equal(got, want.astype(np.float64))


def check_col_bwd_dw(col_bwd_dw, p, m, k, n, seed):
    x = _ints((m, k), seed)
    dy = _ints((m, n * p), seed + 1)
    want = _as_int(x).T @ _as_int(dy)
    got = col_bwd_dw(x, _shard_cols(dy, p))
    return np.array_equal(np.hstack(got), want.astype(np.float64))


def check_row_bwd_dx(row_bwd_dx, p, m, k, n, seed):
    a = _ints((k * p, n), seed)
    dy = _ints((m, n), seed + 1)
    want = _as_int(dy) @ _as_int(a).T
    got = row_bwd_dx(_shard_rows(a, p), dy)
    return np.array_equal(np.hstack(got), want.astype(np.float64))


def check_row_bwd_dw(row_bwd_dw, p, m, k, n, seed):
    x = _ints((m, k * p), seed)
    dy = _ints((m, n), seed + 1)
    want = _as_int(x).T @ _as_int(dy)
    got = row_bwd_dw(_shard_cols(x, p), dy)
    return np.array_equal(np.vstack(got), want.astype(np.float64))


def check_ag(ag, p, m, k, n, seed):
    x = _ints((m, k), seed)
    a = _ints((k, n * p), seed + 1)
    want = _as_int(x) @ _as_int(a)
    ys, _, xg = ag(_shard_rows(x, p), _shard_cols(a, p))
    return np.array_equal(xg, _as_int(x).astype(np.float64)) and \
        np.array_equal(np.hstack(ys), want.astype(np.float64))


SHAPES = [(1, 8, 5, 7), (2, 6, 4, 6), (3, 9, 5, 4), (4, 8, 16, 8), (8, 16, 8, 3)]  # p, m, k, n


# --------------------------------------------------------------- brute force, tiny

def test_tp_tutorial_4x6_example_brute_force():
    """TP tutorial §5.3: in = 4, out = 6, p = 2; column shards 4x3, row shards 2x6."""
    m, inn, out, p = 3, 4, 6, 2
    x = _ints((m, inn), 11)
    a = _ints((inn, out), 12)
    xi, ai = _as_int(x), _as_int(a)
    full = _brute(xi.tolist(), ai.tolist())

    col_shards = _shard_cols(a, p)
    assert [s.shape for s in col_shards] == [(4, 3), (4, 3)]
    ys, _ = oracle.col_fwd(x, col_shards)
    for k in range(p):
        assert ys[k].tolist() == [row[3 * k:3 * k + 3] for row in full]

    row_shards = _shard_rows(a, p)
    assert [s.shape for s in row_shards] == [(2, 6), (2, 6)]
    xs = _shard_cols(x, p)
    parts = oracle.row_partials(xs, row_shards)
    for k in range(p):
        assert parts[k].tolist() == _brute(_as_int(xs[k]).tolist(), _as_int(row_shards[k]).tolist())
    assert oracle.row_fwd_allreduce(xs, row_shards).tolist() == full
    # summing, not concatenating, gives the layer output (M027 §07, first exercise)
    assert np.hstack(parts).shape != (m, out) or not np.array_equal(np.hstack(parts), full)


def test_p1_is_textbook_gemm():
    x = _ints((5, 7), 21)
    w = _ints((7, 3), 22)
    want = _brute(_as_int(x).tolist(), _as_int(w).tolist())
    assert oracle.row_fwd_allreduce([x], [w]).tolist() == want
    assert oracle.col_fwd(x, [w])[0][0].tolist() == want
    dy = _ints((5, 3), 23)
    want_dx = _brute(_as_int(dy).tolist(), _as_int(w).T.tolist())
    assert oracle.col_bwd_dx([w], [dy]).tolist() == want_dx
    assert oracle.row_bwd_dx([w], dy)[0].tolist() == want_dx
    want_dw = _brute(_as_int(x).T.tolist(), _as_int(dy).tolist())
    assert oracle.col_bwd_dw(x, [dy])[0].tolist() == want_dw
    assert oracle.row_bwd_dw([x], dy)[0].tolist() == want_dw


# --------------------------------------------------------------- invariants, exact

@pytest.mark.parametrize("p,m,k,n", SHAPES)
def test_invariants_exact(p, m, k, n):
    s = 1000 + 17 * p + m
    assert check_row_fwd(oracle.row_fwd_allreduce, p, m, k, n, s)
    assert check_row_rs(oracle.row_fwd_reducescatter, p, m, k, n, s)
    assert check_col_fwd(oracle.col_fwd, p, m, k, n, s)
    assert check_col_bwd_dx(oracle.col_bwd_dx, p, m, k, n, s)
    assert check_col_bwd_dw(oracle.col_bwd_dw, p, m, k, n, s)
    assert check_row_bwd_dx(oracle.row_bwd_dx, p, m, k, n, s)
    assert check_row_bwd_dw(oracle.row_bwd_dw, p, m, k, n, s)
    assert check_ag(oracle.ag_matmul, p, m, k, n, s)


def test_rs_slices_concatenate_to_allreduce():
    p, m = 4, 16
    xs = [synth.normal_bf16((m, 24), synth.seed_for(9, r)) for r in range(p)]
    ws = [synth.normal_bf16((24, 10), synth.seed_for(9, 8 + r)) for r in range(p)]
    ar = oracle.row_fwd_allreduce(xs, ws)
    rs = oracle.row_fwd_reducescatter(xs, ws)
    assert np.array_equal(np.vstack(rs), ar)


def test_rank_order_is_left_to_right():
    """The reduction sums partials r = 0, 1, ... in that order (fp64)."""
    # values chosen so that a different order rounds differently in fp64
    big, small = 2.0 ** 60, 1.0
    xs = [synth.f32_to_bf16_bits(np.array([[v]], np.float32)) for v in (big, small, -big)]
    ws = [synth.f32_to_bf16_bits(np.array([[1.0]], np.float32))] * 3
    y = oracle.row_fwd_allreduce(xs, ws)
    assert y[0, 0] == ((big + small) + -big)  # == 0.0 in fp64; another order gives 1.0
    assert y[0, 0] == 0.0


# --------------------------------------------------------------- GeLU closed forms

def test_gelu_closed_forms():
    # GeLU(x) = x * Phi(x); Phi(1) = 0.8413447460685429 (normal CDF table)
    assert oracle.gelu(np.array(0.0)) == 0.0
    assert abs(oracle.gelu(np.array(1.0)) - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu(np.array(-1.0)) + 0.15865525393145707) < 1e-15
    assert abs(oracle.gelu(np.array(2.0)) - 2 * 0.9772498680518208) < 1e-14
    x = np.linspace(-6, 6, 241)
    assert np.allclose(oracle.gelu(x) - oracle.gelu(-x), x, atol=1e-14, rtol=0)  # x*Phi(x) - (-x)Phi(-x)
    assert oracle.gelu(np.array(12.0)) == 12.0 and oracle.gelu(np.array(-12.0)) == 0.0


def test_gelu_prime_closed_forms():
    assert oracle.gelu_prime(np.array(0.0)) == 0.5
    # phi(1) = 0.24197072451914337: GeLU'(1) = Phi(1) + phi(1)
    assert abs(oracle.gelu_prime(np.array(1.0)) - (0.8413447460685429 + 0.24197072451914337)) < 1e-15
    x = np.linspace(-5, 5, 201)
    h = 1e-5
    fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
    assert np.max(np.abs(fd - oracle.gelu_prime(x))) < 1e-9
    assert oracle.gelu_prime(np.array(40.0)) == 1.0 and oracle.gelu_prime(np.array(-40.0)) == 0.0


def test_gelu_epilogues_special_cases():
    """Pins the epilogues wired into the layer functions, not only gelu()."""
    p, m, k, n = 2, 6, 8, 5
    a = _ints((k * p, n), 31)
    dy = _ints((m, n), 32)
    ws = _shard_rows(a, p)
    base = _as_int(dy) @ _as_int(a).T
    zero = [synth.f32_to_bf16_bits(np.zeros((m, k), np.float32))] * p
    got = oracle.row_bwd_dx(ws, dy, preacts=zero)          # GeLU'(0) = 1/2
    assert np.array_equal(np.hstack(got), base / 2.0)
    far = [synth.f32_to_bf16_bits(np.full((m, k), 64.0, np.float32))] * p
    assert np.array_equal(np.hstack(oracle.row_bwd_dx(ws, dy, preacts=far)), base.astype(np.float64))
    neg = [synth.f32_to_bf16_bits(np.full((m, k), -64.0, np.float32))] * p
    assert np.all(np.hstack(oracle.row_bwd_dx(ws, dy, preacts=neg)) == 0.0)

    x = synth.f32_to_bf16_bits(np.full((3, 4), 4.0, np.float32))
    w = synth.f32_to_bf16_bits(np.full((4, 2), 4.0, np.float32))   # H = 64 everywhere
    ys, hs = oracle.col_fwd(x, [w], apply_gelu=True)
    assert np.all(hs[0] == 64.0) and np.all(ys[0] == 64.0)
    ys, hs = oracle.col_fwd(x, [synth.f32_to_bf16_bits(-np.full((4, 2), 4.0, np.float32))], apply_gelu=True)
    assert np.all(hs[0] == -64.0) and np.all(ys[0] == 0.0)


# --------------------------------------------------------------- chunk timeline

def test_pipeline_timeline_golden():
    for c, m, n, t, serial in _read_rows("pipeline_timeline.txt"):
        assert oracle.pipeline_time(float(c), float(m), int(n)) == float(t)
        assert oracle.serial_time(float(c), float(m), int(n)) == float(serial)
    # -30 % as the page states
    assert abs(1 - oracle.pipeline_time(3, 2, 4) / oracle.serial_time(3, 2, 4) - 0.30) < 1e-12


def test_pipeline_timeline_exercise_and_edges():
    # M027 §07 exercise: compute 1 ms, communication 5 ms, 4 chunks.  By the
    # page's timeline rule: 1 + 3 x 5 + 5 = 21 ms against 4 x 6 = 24 ms serial.
    assert oracle.pipeline_time(1, 5, 4) == 21
    assert oracle.serial_time(1, 5, 4) == 24
    assert oracle.pipeline_time(2, 7, 1) == 9 == oracle.serial_time(2, 7, 1)  # one chunk: no overlap
    assert oracle.pipeline_time(3, 3, 5) == 18                                 # c = m: (n + 1) c
    assert oracle.pipeline_time(3, 2, 0) == 0


def test_worked_example_shapes_and_bytes():
    g = {r[0]: [int(v) for v in r[1:]] for r in _read_rows("worked_example.txt")}
    (m, n), (chunk_m,), (eb,) = g["y_r"], g["chunk_m"], g["elem_bytes"]
    assert oracle.n_chunks(m, chunk_m) == g["n_chunks"][0]
    assert m * n * eb == g["local_output_kib"][0] * 1024
    assert chunk_m * n * eb == g["chunk_kib"][0] * 1024
    assert g["x_r"][0] == m and g["x_r"][1] == g["w_r"][0] and g["w_r"][1] == n
    # the computation itself at these shapes: the sum of the two partials equals
    # the unsharded product (exact on integer inputs), chunk by chunk
    p = g["p"][0]
    k = g["x_r"][1]
    assert check_row_fwd(oracle.row_fwd_allreduce, p, m, k, 64, 77)


def test_n_chunks_rules():
    assert oracle.n_chunks(128, 32) == 4
    assert oracle.n_chunks(130, 32) == 5        # last chunk short
    assert oracle.n_chunks(16, 2048) == 1       # chunk_m > M is clamped to M
    assert [oracle.n_chunks(2048, c) for c in (16, 64, 256, 1024, 2048)] == [128, 32, 8, 2, 1]
    assert oracle.n_chunks(0, 32) == 0


def test_collective_volumes_golden():
    for p, f in _read_rows("allreduce_volume.txt"):
        assert oracle.allreduce_bytes(int(p), 1.0) == float(f)
        # AllGather + ReduceScatter carry the same volume as one AllReduce (TP §2.7)
        assert 2 * oracle.allgather_bytes(int(p), 1.0) == float(f)
    g = {r[0]: int(r[1]) for r in _read_rows("mlp_example.txt")}
    msg = g["b"] * g["s"] * g["h"] * g["elem_bytes"]
    assert oracle.allreduce_bytes(g["p"], msg) == g["allreduce_bytes"]
    assert g["h"] * g["ffn"] * g["elem_bytes"] == g["w1_mib"] << 20
    assert g["h"] * (g["ffn"] // g["p"]) * g["elem_bytes"] == g["w1_shard_mib"] << 20


# --------------------------------------------------------------- bf16 and the generator

def test_round_bf16_values():
    vals = np.array([1.0, 1.0 / 3.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.0, 0.0])
    assert oracle.round_bf16(vals).tolist() == [0x3F80, 0x3EAB, 0x3F80, 0x3F82, 0xC000, 0x0000]
    assert synth.f32_to_bf16_bits(vals.astype(np.float32)).tolist() == [0x3F80, 0x3EAB, 0x3F80, 0x3F82, 0xC000, 0]


def test_round_bf16_rounds_through_fp32():
    """The oracle rounds a float64 value to bf16 the way the library rounds
    its accumulator: first to fp32 (the accumulator's type), then to bf16,
    nearest even.  1 + 2^-8 + 2^-30 lies just above the bf16 midpoint
    between 1 and 1 + 2^-7, so rounding float64 -> bf16 directly would give
    1 + 2^-7 (0x3F81); through fp32 the 2^-30 is lost (below half an fp32
    ulp), the value becomes the exact midpoint and ties to even: 1.0."""
    x = np.array([1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8 + 2 ** -30), 3 * 2 ** -9 + 2 ** -40])
    assert oracle.round_bf16(x).tolist() == [0x3F80, 0xBF80, 0x3BC0]
    # a value that only the direct route rounds up, checked against exact
    # rational arithmetic: the direct nearest-bf16 is the upper neighbour
    from fractions import Fraction
    v = Fraction(1) + Fraction(1, 2 ** 8) + Fraction(1, 2 ** 30)
    lo, hi = Fraction(1), Fraction(1) + Fraction(1, 2 ** 7)
    assert v - lo > hi - v


def test_splitmix64_published_vectors():
    # Vigna's reference splitmix64 outputs for seeds 0 and 1234567
    assert [int(v) for v in synth.splitmix64(0, 0, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(v) for v in synth.splitmix64(1234567, 0, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_normal_generator_statistics_and_determinism():
    a = synth.normal_bf16((1 << 20,), 5, sigma=0.02)
    b = synth.normal_bf16((1 << 20,), 5, sigma=0.02)
    assert np.array_equal(a, b)
    v = oracle.widen(a)
    assert abs(v.mean()) < 1e-4 and abs(v.std() - 0.02) < 2e-4
    # chunked / threaded generation equals one long stream
    c = synth.normal_bf16((3, (1 << 21) + 7), 6)
    d = synth.normal_bf16(((1 << 21) * 3 + 21,), 6, threads=1)
    assert np.array_equal(c.reshape(-1), d)


# --------------------------------------------------------------- planted mistakes

def _drop_last(xs, ws):
    return oracle.row_fwd_allreduce(xs[:-1], ws[:-1]) if len(xs) > 1 else -oracle.row_fwd_allreduce(xs, ws)


def _wrong_sign(xs, ws):
    parts = oracle.row_partials(xs, ws)
    y = parts[0].copy()
    for q in parts[1:]:
        y = y - q
    return y if len(parts) > 1 else y + 1


def _misrouted_rs(xs, ws):
    s = oracle.row_fwd_reducescatter(xs, ws)
    return s[::-1] if len(s) > 1 else [s[0] * 2]


def _untransposed_dx(ws, dys):
    parts = [oracle.widen(d) @ oracle.widen(w).T[::-1] for d, w in zip(dys, ws)]
    return sum(parts[1:], parts[0])


def _col_shifted(x, ws):
    ys, hs = oracle.col_fwd(x, ws)
    return ys[1:] + ys[:1], hs


def _dw_no_transpose_fix(x, dys):
    return [oracle.widen(x).T @ oracle.widen(d)[::-1] for d in dys]


def _ag_wrong_order(xs, ws):
    return oracle.ag_matmul(xs[::-1], ws)


def test_planted_mistakes_are_caught():
    p, m, k, n = 2, 8, 6, 5
    assert not check_row_fwd(_drop_last, p, m, k, n, 3)
    assert not check_row_fwd(_wrong_sign, p, m, k, n, 3)
    assert not check_row_rs(_misrouted_rs, p, m, k, n, 3)
    assert not check_col_bwd_dx(_untransposed_dx, p, m, k, n, 3)
    assert not check_col_fwd(_col_shifted, p, m, k, n, 3)
    assert not check_col_bwd_dw(_dw_no_transpose_fix, p, m, k, n, 3)
    assert not check_ag(_ag_wrong_order, p, m, k, n, 3)
    bad_gelu = lambda h: 0.5 * h * (1.0 + np.tanh(h))  # noqa: E731 (wrong activation)
    assert abs(bad_gelu(1.0) - 0.8413447460685429) > 1e-3


# --------------------------------------------------------------- sequence-parallel backward

def check_ag_bwd(dx_fn, dw_fn, p, m, k, n, seed):
    """AllGather+MatMul backward against the unsharded layer Y = X A (A = [A_0 | ...]):
    dX = dY A^T scattered by rows, dA = X^T dY split by columns."""
    x = _ints((m, k), seed)
    a = _ints((k, n * p), seed + 1)
    dy = _ints((m, n * p), seed + 2)
    xs, ws, dys = _shard_rows(x, p), _shard_cols(a, p), _shard_cols(dy, p)
    want_dx = _as_int(dy) @ _as_int(a).T
    want_dw = _as_int(x).T @ _as_int(dy)
    got_dx = dx_fn(ws, dys)
    got_dw = dw_fn(xs, dys)
    return (len(got_dx) == p and np.array_equal(np.vstack(got_dx), want_dx.astype(np.float64)) and
            np.array_equal(np.hstack(got_dw), want_dw.astype(np.float64)))


def check_rs_bwd(dx_fn, dw_fn, p, m, k, n, seed):
    """MatMul+ReduceScatter backward against the unsharded layer Y = X A
    (X = [X_0 | ...], A = [A_0; ...]): dY gathered by rows, dX = dY A^T split by
    columns, dA = X^T dY split by rows."""
    x = _ints((m, k * p), seed)
    a = _ints((k * p, n), seed + 1)
    dy = _ints((m, n), seed + 2)
    xs, ws, dys = _shard_cols(x, p), _shard_rows(a, p), _shard_rows(dy, p)
    want_dx = _as_int(dy) @ _as_int(a).T
    want_dw = _as_int(x).T @ _as_int(dy)
    return (np.array_equal(np.hstack(dx_fn(ws, dys)), want_dx.astype(np.float64)) and
            np.array_equal(np.vstack(dw_fn(xs, dys)), want_dw.astype(np.float64)))


@pytest.mark.parametrize("p,m,k,n", [(1, 8, 5, 7), (2, 6, 4, 6), (4, 8, 16, 8), (8, 16, 8, 3)])
def test_sequence_parallel_backward_exact(p, m, k, n):
    assert check_ag_bwd(oracle.ag_matmul_bwd_dx, oracle.ag_matmul_bwd_dw, p, m, k, n, 2000 + p)
    assert check_rs_bwd(oracle.row_rs_bwd_dx, oracle.row_rs_bwd_dw, p, m, k, n, 2100 + p)


def test_sequence_parallel_backward_duality():
    """RS of the column-backward dX equals the column backward's row blocks, and
    the gathered-gradient row backward equals the row backward on the stacked dY."""
    p, m, k, n = 4, 8, 6, 5
    ws = [_ints((k, n), 2200 + i) for i in range(p)]
    dys = [_ints((m, n), 2210 + i) for i in range(p)]
    assert np.array_equal(np.vstack(oracle.ag_matmul_bwd_dx(ws, dys)), oracle.col_bwd_dx(ws, dys))
    shards = [_ints((m // p, n), 2220 + i) for i in range(p)]
    assert all(np.array_equal(a, b) for a, b in
               zip(oracle.row_rs_bwd_dx(ws, shards), oracle.row_bwd_dx(ws, np.vstack(shards))))


def test_sequence_parallel_backward_planted_mistakes():
    p, m, k, n = 2, 8, 6, 5
    wrong_order_dx = lambda ws, dys: oracle.ag_matmul_bwd_dx(ws, dys)[::-1]          # noqa: E731
    assert not check_ag_bwd(wrong_order_dx, oracle.ag_matmul_bwd_dw, p, m, k, n, 5)
    wrong_gather_dw = lambda xs, dys: oracle.ag_matmul_bwd_dw(xs[::-1], dys)          # noqa: E731
    assert not check_ag_bwd(oracle.ag_matmul_bwd_dx, wrong_gather_dw, p, m, k, n, 5)
    wrong_gather_dx = lambda ws, dys: oracle.row_rs_bwd_dx(ws, dys[::-1])             # noqa: E731
    assert not check_rs_bwd(wrong_gather_dx, oracle.row_rs_bwd_dw, p, m, k, n, 6)


# --------------------------------------------------------------- bf16-collective emulation

def _scalar_ranks(vals):
    """Rank r contributes the 1x1 partial vals[r] (X_r = [[v]], W_r = [[1]])."""
    one = synth.f32_to_bf16_bits(np.array([[1.0]], np.float32))
    xs = [synth.f32_to_bf16_bits(np.array([[v]], np.float32)) for v in vals]
    return xs, [one] * len(vals)


def test_bf16_collective_hand_values():
    """bf16 keeps 8 significant bits: between 256 and 512 its step is 2, and a
    tie goes to the even significand (256, not 258)."""
    coll = oracle.row_fwd_allreduce_bf16_collective
    # running sum rounded: 256 + 1 = 257 -> 256 (exact sum 257)
    assert coll(*_scalar_ranks([256.0, 1.0]))[0, 0] == 256.0
    assert oracle.row_fwd_allreduce(*_scalar_ranks([256.0, 1.0]))[0, 0] == 257.0
    assert coll(*_scalar_ranks([255.0, 2.0]))[0, 0] == 256.0
    # rank order: (1 + 1) + 256 = 258 exactly, (256 + 1) + 1 = 256
    assert coll(*_scalar_ranks([1.0, 1.0, 256.0]))[0, 0] == 258.0
    assert coll(*_scalar_ranks([256.0, 1.0, 1.0]))[0, 0] == 256.0
    # each partial is rounded before it enters the sum: p = 1, P_0 = 256 + 1
    x = synth.f32_to_bf16_bits(np.array([[1.0, 1.0]], np.float32))
    w = synth.f32_to_bf16_bits(np.array([[256.0], [1.0]], np.float32))
    assert coll([x], [w])[0, 0] == 256.0
    assert oracle.row_fwd_allreduce([x], [w])[0, 0] == 257.0


def test_bf16_collective_small_integers_are_exact():
    """Partials and running sums within [-256, 256] are bf16 integers: no
    rounding happens and the emulation equals the exact sum."""
    p = 4
    xs = [_ints((6, 4), 3000 + r, 2) for r in range(p)]
    ws = [_ints((4, 5), 3010 + r, 2) for r in range(p)]
    assert np.array_equal(oracle.row_fwd_allreduce_bf16_collective(xs, ws), oracle.row_fwd_allreduce(xs, ws))


def test_bf16_collective_error_bound_and_representable():
    """Every output is a bf16 value, and it differs from the exact sum by at
    most the p partial roundings plus the p - 1 sum roundings, each at most
    half a bf16 step (2^-8 relative) of the value it rounds."""
    p, m, k, n = 8, 16, 64, 12
    xs = [synth.normal_bf16((m, k), synth.seed_for(60, r)) for r in range(p)]
    ws = [synth.normal_bf16((k, n), synth.seed_for(60, 8 + r)) for r in range(p)]
    got = oracle.row_fwd_allreduce_bf16_collective(xs, ws)
    assert np.array_equal(oracle.widen(oracle.round_bf16(got)), got)
    parts = oracle.row_partials(xs, ws)
    exact = oracle.row_fwd_allreduce(xs, ws)
    u = 2.0 ** -8
    bound = sum(np.abs(pr) for pr in parts) * u * (1 + u) ** (2 * p)
    for r in range(1, p):
        bound = bound + np.abs(sum(parts[:r + 1])) * u * (1 + u) ** (2 * p)
    bound = bound + sum(np.abs(pr) for pr in parts) * (2 * p * u) ** 2 * 4
    assert np.all(np.abs(got - exact) <= bound)
    assert not np.array_equal(got, exact)


def test_bf16_collective_planted_mistakes():
    """Dropping the partial rounding, the running-sum rounding or the rank
    order each changes a hand value above."""
    def no_partial_rounding(xs, ws):
        parts = oracle.row_partials(xs, ws)
        acc = parts[0]
        for pr in parts[1:]:
            acc = oracle.widen(oracle.round_bf16(acc + pr))
        return oracle.widen(oracle.round_bf16(acc))

    def no_sum_rounding(xs, ws):
        parts = oracle.row_partials(xs, ws)
        return sum(oracle.widen(oracle.round_bf16(pr)) for pr in parts)

    def reversed_order(xs, ws):
        return oracle.row_fwd_allreduce_bf16_collective(xs[::-1], ws[::-1])

    x = synth.f32_to_bf16_bits(np.array([[1.0, 1.0]], np.float32))
    w = synth.f32_to_bf16_bits(np.array([[256.0], [1.0]], np.float32))
    # P_0 = 257 and P_1 = 1: rounded first, 256 + 1 -> 256; unrounded, 258
    one = synth.f32_to_bf16_bits(np.array([[1.0]], np.float32))
    assert oracle.row_fwd_allreduce_bf16_collective([x, one], [w, one])[0, 0] == 256.0
    assert no_partial_rounding([x, one], [w, one])[0, 0] == 258.0
    assert no_sum_rounding(*_scalar_ranks([256.0, 1.0]))[0, 0] == 257.0
    assert reversed_order(*_scalar_ranks([256.0, 1.0, 1.0]))[0, 0] == 258.0


# --------------------------------------------------------------- bias

def test_bias_forward_matches_the_unsharded_layer():
    """Y = X A + b of the unsharded layer, with b added once on the row
    layer and b split into the column blocks b_k on the column layer."""
    p, m, k, n = 4, 8, 6, 12
    x = _ints((m, k * p), 4000)
    a = _ints((k * p, n), 4001)
    b = _ints((1, n), 4002)[0]
    want = _as_int(x) @ _as_int(a) + _as_int(b)[None, :]
    got = oracle.row_fwd_allreduce(_shard_cols(x, p), _shard_rows(a, p), bias=b)
    assert np.array_equal(got, want.astype(np.float64))
    rs = oracle.row_fwd_reducescatter(_shard_cols(x, p), _shard_rows(a, p), bias=b)
    assert np.array_equal(np.vstack(rs), want.astype(np.float64))
    xc = _ints((m, k), 4003)
    ac = _ints((k, n * p), 4004)
    bc = _ints((1, n * p), 4005)[0]
    wantc = _as_int(xc) @ _as_int(ac) + _as_int(bc)[None, :]
    bks = [bc[j * n:(j + 1) * n] for j in range(p)]
    ys, _ = oracle.col_fwd(xc, _shard_cols(ac, p), biases=bks)
    assert np.array_equal(np.hstack(ys), wantc.astype(np.float64))
    yg, _, _ = oracle.ag_matmul(_shard_rows(xc, p), _shard_cols(ac, p), biases=bks)
    assert np.array_equal(np.hstack(yg), wantc.astype(np.float64))
    # GeLU sees the biased pre-activation
    z, h = oracle.col_fwd(xc, _shard_cols(ac, p), apply_gelu=True, biases=bks)
    assert np.array_equal(np.hstack(h), wantc.astype(np.float64))
    assert np.allclose(np.hstack(z), oracle.gelu(wantc.astype(np.float64)))


def test_bias_grad_is_the_forward_difference():
    """For L = sum(G * Y), raising b_j by one raises L by exactly sum_i G[i, j]
    (integer inputs: every value exact), which is what bias_grad returns; the
    row-shard form sums the shards' rows."""
    p, m, k, n = 2, 6, 4, 5
    x = _ints((m, k * p), 4100)
    a = _ints((k * p, n), 4101)
    b = _ints((1, n), 4102)[0]
    g = _ints((m, n), 4103)
    xs, ws = _shard_cols(x, p), _shard_rows(a, p)
    base = float(np.sum(oracle.widen(g) * oracle.row_fwd_allreduce(xs, ws, bias=b)))
    db = oracle.bias_grad(g)
    for j in range(n):
        bj = oracle.widen(b).copy()
        bj[j] += 1.0
        up = float(np.sum(oracle.widen(g) * oracle.row_fwd_allreduce(xs, ws, bias=oracle.round_bf16(bj))))
        assert up - base == db[j]
    assert np.array_equal(oracle.bias_grad(_shard_rows(g, 3)), db)


def test_bias_planted_mistakes():
    p, m, k, n = 2, 4, 3, 4
    x = _ints((m, k * p), 4200)
    a = _ints((k * p, n), 4201)
    b = _ints((1, n), 4202, 3)[0]
    want = _as_int(x) @ _as_int(a) + _as_int(b)[None, :]
    # a bias added by every rank (p times) is caught
    twice = oracle.row_fwd_allreduce(_shard_cols(x, p), _shard_rows(a, p)) + p * oracle.widen(b)[None, :]
    assert np.any(_as_int(b) != 0)
    assert not np.array_equal(twice, want.astype(np.float64))
    # a bias gradient over the wrong axis is caught
    g = _ints((m, n), 4203)
    assert not np.array_equal(oracle.widen(g).sum(axis=1)[:n], oracle.bias_grad(g))
