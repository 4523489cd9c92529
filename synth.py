"""Seeded synthetic inputs for the sharded-Linear tests and benchmark.

This module is shared by the CPU oracle's tests and by the CUDA path's
tests and benchmark.  It only *draws* numbers; it holds none of the
sharded-Linear arithmetic.  Every tensor is returned as a numpy ``uint16``
array of bfloat16 bit patterns, so both sides consume bit-identical inputs.

Generator (counter based, platform independent):

* splitmix64 (Vigna's published mixer): the i-th 64-bit word of stream
  ``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)``;
* two consecutive words give two uniforms ``u = (w >> 11) * 2**-53``;
* Box-Muller turns ``(1 - u0, u1)`` into two standard normals (float64);
* the normal is scaled by sigma in float64, rounded to float32, then to
  bfloat16 with round-to-nearest-even.

Seeds follow ``0x5EED0000 + 16 * config_index + tensor_index``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
MIX1 = np.uint64(0xBF58476D1CE4E5B9)
MIX2 = np.uint64(0x94D049BB133111EB)
SEED_BASE = 0x5EED0000

_CHUNK = 1 << 22  # elements per worker chunk


def seed_for(config_index: int, tensor_index: int) -> int:
    """Seed of tensor ``tensor_index`` of workload ``config_index``."""
    return SEED_BASE + 16 * config_index + tensor_index


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of the splitmix64 stream of ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * MIX1
        z = (z ^ (z >> np.uint64(27))) * MIX2
        return z ^ (z >> np.uint64(31))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_chunk(seed: int, first_pair: int, n_pairs: int) -> np.ndarray:
    w = splitmix64(seed, 2 * first_pair, 2 * n_pairs).reshape(n_pairs, 2)
    scale = 2.0 ** -53
    u0 = 1.0 - (w[:, 0] >> np.uint64(11)).astype(np.float64) * scale  # (0, 1]
    u1 = (w[:, 1] >> np.uint64(11)).astype(np.float64) * scale        # [0, 1)
    r = np.sqrt(-2.0 * np.log(u0))
    t = 2.0 * np.pi * u1
    out = np.empty((n_pairs, 2), dtype=np.float64)
    out[:, 0] = r * np.cos(t)
    out[:, 1] = r * np.sin(t)
    return out.reshape(-1)


def normal_bf16(shape, seed: int, sigma: float = 1.0, threads: int | None = None) -> np.ndarray:
    """bfloat16 bits of N(0, sigma**2) draws, element ``i`` from pair ``i // 2``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=np.uint16)
    if n == 0:
        return out.reshape(shape)
    n_pairs = (n + 1) // 2
    pairs_per_chunk = _CHUNK // 2

    def work(first_pair):
        cnt = min(pairs_per_chunk, n_pairs - first_pair)
        vals = _normal_chunk(seed, first_pair, cnt) * sigma
        lo = 2 * first_pair
        hi = min(n, lo + 2 * cnt)
        out[lo:hi] = f32_to_bf16_bits(vals[: hi - lo].astype(np.float32))

    starts = list(range(0, n_pairs, pairs_per_chunk))
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    if len(starts) == 1 or threads <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


def integer_bf16(shape, seed: int, bound: int = 4) -> np.ndarray:
    """bfloat16 bits of integers drawn uniformly from ``[-bound, bound]``.

    Products and sums of such values stay exact in float32 as long as every
    partial sum stays below 2**24, which makes GPU output comparable bit for
    bit with an exact reference.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    w = splitmix64(seed, 0, n)
    v = (w % np.uint64(2 * bound + 1)).astype(np.int64) - bound
    return f32_to_bf16_bits(v.astype(np.float32)).reshape(shape)


def onehot_bf16(rows: int, cols: int, seed: int) -> np.ndarray:
    """A matrix with exactly one 1.0 per row at a seeded column (others 0).

    Used as a coordinate encoding: multiplying by it routes whole rows or
    columns, so any transposed or misrouted tile shows up as a wrong value.
    """
    w = splitmix64(seed, 0, rows)
    col = (w % np.uint64(max(cols, 1))).astype(np.int64)
    m = np.zeros((rows, cols), dtype=np.float32)
    m[np.arange(rows), col] = 1.0
    return f32_to_bf16_bits(m)


def ramp_bf16(rows: int, cols: int, scale: float = 1.0) -> np.ndarray:
    """Distinct small integers ``((i * cols + j) % 251 - 125) * scale`` as bf16."""
    i = np.arange(rows, dtype=np.int64)[:, None]
    j = np.arange(cols, dtype=np.int64)[None, :]
    v = ((i * cols + j) % 251 - 125).astype(np.float32) * np.float32(scale)
    return f32_to_bf16_bits(v)


# --------------------------------------------------------------- workload recipes
# Shapes, value distributions and seeds of the five sharded-Linear workloads.
# Each recipe only names tensors and draws them; what is computed from them
# lives in the library (GPU) and in the oracle (CPU).  Each recipe has its
# own seed namespace c (1 to 5, in the order below): tensor group g draws
# from seed_for(10 * c + g, shard).

def _sd(c, g, k=0):
    return seed_for(10 * c + g, k)


def worked_example_inputs():
    """Row-parallel Linear, p = 2: X_r [128, 1024], W_r [1024, 2048], N(0,1)/sqrt(2048)."""
    s = 1.0 / np.sqrt(2048.0)
    return {"x": [normal_bf16((128, 1024), _sd(1, 0, r), s) for r in range(2)],
            "w": [normal_bf16((1024, 2048), _sd(1, 1, r), s) for r in range(2)]}


def mlp_block_inputs():
    """MLP block, p = 4, 4096 tokens, h = 4096, ffn = 16384: X, dY N(0,1); W N(0, 0.02)."""
    p, m, h, nk = 4, 4096, 4096, 4096
    return {"x": normal_bf16((m, h), _sd(2, 0)),
            "w1": [normal_bf16((h, nk), _sd(2, 1, k), 0.02) for k in range(p)],
            "w2": [normal_bf16((nk, h), _sd(2, 2, k), 0.02) for k in range(p)],
            "dy": normal_bf16((m, h), _sd(2, 3))}


def mha_projection_inputs():
    """MHA projections, p = 4, 2 x 2048 tokens, h = 4096, 8 heads x 128 per shard:
    X, attention output O_k, dY, dQKV_k N(0,1); W_qkv_k [4096, 3072], W_O_k [1024, 4096] N(0, 0.02)."""
    p, m, h = 4, 4096, 4096
    return {"x": normal_bf16((m, h), _sd(3, 0)),
            "wqkv": [normal_bf16((h, 3 * 1024), _sd(3, 1, k), 0.02) for k in range(p)],
            "o": [normal_bf16((m, 1024), _sd(3, 2, k)) for k in range(p)],
            "wo": [normal_bf16((1024, h), _sd(3, 3, k), 0.02) for k in range(p)],
            "dy": normal_bf16((m, h), _sd(3, 4)),
            "dqkv": [normal_bf16((m, 3 * 1024), _sd(3, 5, k)) for k in range(p)]}


def sequence_parallel_pair_inputs():
    """Sequence-parallel pair, p = 8: X_r [1024, 8192] N(0,1); W1_k [8192, 3584], W2_k [3584, 8192] N(0, 0.02)."""
    p = 8
    return {"x": [normal_bf16((1024, 8192), _sd(4, 0, r)) for r in range(p)],
            "w1": [normal_bf16((8192, 3584), _sd(4, 1, k), 0.02) for k in range(p)],
            "w2": [normal_bf16((3584, 8192), _sd(4, 2, k), 0.02) for k in range(p)]}


def gpt3_mlp_activations(m: int):
    """GPT-3-scale MLP input X [m, 12288] N(0,1)."""
    return normal_bf16((m, 12288), _sd(5, 0, 0 if m == 2048 else 1))


def gpt3_mlp_weights():
    """GPT-3-scale MLP weights, p = 8: W1_k [12288, 6144], W2_k [6144, 12288] N(0, 0.02)."""
    p = 8
    return {"w1": [normal_bf16((12288, 6144), _sd(5, 1, k), 0.02) for k in range(p)],
            "w2": [normal_bf16((6144, 12288), _sd(5, 2, k), 0.02) for k in range(p)]}


def gpt3_mlp_inputs(m: int):
    """GPT-3-scale MLP, p = 8, h = 12288, ffn = 49152: X [m, 12288] N(0,1); W N(0, 0.02)."""
    return dict(gpt3_mlp_weights(), x=gpt3_mlp_activations(m))
