"""Seeded synthetic inputs for the attention forward workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can be fed
from it without sharing any of the method's code.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; constants as in Vigna's public splitmix64.c)
used as a counter-based generator -- uniform ``n`` of stream ``s`` is the
splitmix64 output function applied to ``key(seed, s) + n * gamma`` (gamma the
golden-ratio increment) -- then the Box-Muller transform in float64 (uniforms
2i and 2i+1 give normal i), then round-to-nearest-even to bfloat16.  The output is therefore a
pure function of (seed, stream, index) and does not depend on torch's or
numpy's own random number state.

Workload recipes (FlashAttention-3 deep-reading report, §4.1 and §4.3):
  * plain:    Q, K, V iid N(0, 1);
  * outliers: N(0, 1) with 0.1 % of the entries replaced by N(0, 10^2)
              (standard deviation 10), the outlier-heavy distribution the
              report's §4.3 (Table 3) uses to compare FP8 schemes.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one independent counter stream per (tensor, purpose).
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
_OUTLIER_SELECT = 16   # added to the tensor stream for the outlier mask
_OUTLIER_VALUE = 32    # added to the tensor stream for the outlier values


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed & 0xFFFFFFFF) << 20 | (stream & 0xFFFFF)], dtype=np.uint64)
    return _mix(s + _GOLDEN)[0]


def _uniform53(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in (0, 1]: 53 high bits of splitmix64 outputs."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start, start + count, dtype=np.uint64)
        z = _mix(ctr * _GOLDEN + _key(seed, stream))
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def standard_normal(n: int, seed: int, stream: int) -> np.ndarray:
    """n iid N(0,1) float64 values (Box-Muller, cosine branch)."""
    out = np.empty(n, dtype=np.float64)
    chunk = 1 << 20

    def fill(s: int) -> None:
        c = min(chunk, n - s)
        u = _uniform53(seed, stream, 2 * s, 2 * c)
        out[s:s + c] = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * np.pi * u[1::2])

    starts = range(0, n, chunk)
    if n > chunk:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, starts))
    else:
        for s in starts:
            fill(s)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (nearest, ties to even); uint16 bits.

    The value is first rounded to float32, then to bfloat16; that is part of
    the recipe's definition.  Inputs are finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def tensor_bf16(shape, seed: int, stream: int, outliers: bool = False,
                outlier_frac: float = 1e-3, outlier_std: float = 10.0) -> np.ndarray:
    """A bf16 tensor (as uint16 bits) of the given shape."""
    n = int(np.prod(shape))
    x = standard_normal(n, seed, stream)
    if outliers:
        sel = np.empty(n, dtype=bool)
        chunk = 1 << 23
        for s in range(0, n, chunk):
            c = min(chunk, n - s)
            sel[s:s + c] = _uniform53(seed, stream + _OUTLIER_SELECT, s, c) <= outlier_frac
        idx = np.nonzero(sel)[0]
        if idx.size:
            x[idx] = outlier_std * _normal_at(idx, seed, stream + _OUTLIER_VALUE)
    return to_bf16_bits(x).reshape(shape)


def _normal_at(idx: np.ndarray, seed: int, stream: int) -> np.ndarray:
    """standard_normal(...)[idx] without drawing the whole stream."""
    with np.errstate(over="ignore"):
        key = _key(seed, stream)
        c1 = (2 * idx).astype(np.uint64)
        u1 = ((_mix(c1 * _GOLDEN + key) >> np.uint64(11)).astype(np.float64) + 1.0) / 9007199254740992.0
        u2 = ((_mix((c1 + np.uint64(1)) * _GOLDEN + key) >> np.uint64(11)).astype(np.float64) + 1.0) / 9007199254740992.0
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def qkv_bf16(B: int, N: int, H: int, d: int, seed: int = 0, outliers: bool = False):
    """Q, K, V as bf16 bit arrays in (batch, seqlen, heads, head_dim) layout."""
    shape = (B, N, H, d)
    return tuple(tensor_bf16(shape, seed, s, outliers) for s in (STREAM_Q, STREAM_K, STREAM_V))


def sample_rows(N: int, count: int, seed: int, must=()) -> np.ndarray:
    """Sorted distinct query rows: the first/last rows, tile-boundary rows,
    the rows in ``must`` and seeded uniform picks, ``count`` in total
    (or all rows when N <= count)."""
    if N <= count:
        return np.arange(N, dtype=np.int32)
    fixed = {0, 1, N - 1, N - 2}
    for t in (63, 64, 127, 128, 129, 255, 256, 257):
        if t < N:
            fixed.add(t)
    fixed.update(int(r) for r in must if 0 <= r < N)
    rows = set(fixed)
    k = 0
    while len(rows) < count:
        u = _uniform53(seed, 77, k, 4 * count)
        for x in (u * N).astype(np.int64):
            if len(rows) >= count:
                break
            rows.add(int(min(x, N - 1)))
        k += 4 * count
    return np.array(sorted(rows), dtype=np.int32)


def rope_tables(N: int, d: int, base: float = 10000.0):
    """Rotary-embedding tables for token positions 0..N-1: cos and sin of the
    angle n * base^(-2i/d) for pair index i < d/2, evaluated in float64 and
    rounded to binary32; shape (N, d/2) each.  (The frequencies of Su et al.,
    "RoFormer", 2021.)  These are inputs of the RoPE prep, like Q and K."""
    i = np.arange(d // 2, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / d)
    ang = np.arange(N, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
