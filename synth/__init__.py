"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module holds no arithmetic of the ConvRot method: it only draws numbers.
Every tensor is a pure function of (seed, stream id, element index), so any
row slab of a large tensor can be regenerated on its own.

Generator (one counter-based stream per (seed, stream id)):
  * splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014; the constants of Vigna's public-domain C version):
    state advances by the golden gamma 0x9E3779B97F4A7C15 and each state is
    passed through the two-multiply finaliser.
  * stream base  = mix(mix(seed) + stream_id); word i = mix(base + (i + 1) * gamma).
  * uniform in (0, 1): ((word >> 11) + 0.5) * 2^-53.
  * normal: Box-Muller on the pair (u[2j], u[2j+1]):
      z[2j] = sqrt(-2 ln u1) cos(2 pi u2),  z[2j+1] = sqrt(-2 ln u1) sin(2 pi u2).
  * bf16 inputs: the fp64 sample rounded to nearest-even bf16.

Stream ids: x = 0, W = 1, lora A = 2, lora B = 3, dY = 4, token ids = 5,
outlier-channel pick = 6, embedding table = 7.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_X, STREAM_W, STREAM_A, STREAM_B, STREAM_DY, STREAM_IDS, STREAM_OUTLIER, STREAM_TABLE = range(8)

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(v: int) -> int:
    with np.errstate(over="ignore"):
        return int(_mix(np.array([v & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def stream_base(seed: int, stream: int) -> int:
    return _mix_scalar((_mix_scalar(seed) + stream) & 0xFFFFFFFFFFFFFFFF)


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Words start .. start+count-1 of the stream, as uint64."""
    base = np.uint64(stream_base(seed, stream))
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GAMMA)


def uniform(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    w = words(seed, stream, start, count)
    return ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, start: int, count: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """Elements start .. start+count-1 of the stream's N(mu, sigma) sequence (fp64)."""
    out = np.empty(count, dtype=np.float64)
    pos = 0
    while pos < count:
        n = min(_CHUNK, count - pos)
        i0 = start + pos
        p0 = i0 // 2
        p1 = (i0 + n - 1) // 2 + 1
        u = uniform(seed, stream, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
        r = np.sqrt(-2.0 * np.log(u[:, 0]))
        t = 2.0 * np.pi * u[:, 1]
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        off = i0 - 2 * p0
        out[pos:pos + n] = z[off:off + n]
        pos += n
    return out * sigma + mu


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)  # first rounding
    b = f.view(np.uint32).astype(np.uint64)
    # Second rounding from fp32 to bf16 must not double-round: redo it from fp64.
    # Exactly: take the two bf16 neighbours of the fp32 value and pick the nearer
    # to the fp64 value, ties to even mantissa.
    lo = (b & np.uint64(0xFFFF0000)).astype(np.uint32)
    hi = (lo.astype(np.uint64) + np.uint64(0x10000)).astype(np.uint32)
    flo = lo.view(np.float32).astype(np.float64)
    fhi = hi.view(np.float32).astype(np.float64)
    # the neighbour above the largest finite bf16 is 2^128 (it rounds to infinity)
    at_inf = (hi & np.uint32(0x7FFFFFFF)) == np.uint32(0x7F800000)
    fhi = np.where(at_inf, np.copysign(2.0 ** 128, flo), fhi)
    v64 = np.asarray(v, dtype=np.float64)
    dlo = np.abs(v64 - flo)
    dhi = np.abs(v64 - fhi)
    even_lo = ((lo >> 16) & 1) == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ~even_lo)
    res = np.where(pick_hi, hi, lo) >> 16
    return res.astype(np.uint16)


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_bf16(seed: int, stream: int, rows: int, cols: int, sigma: float, row0: int = 0) -> np.ndarray:
    """bf16 bits [rows, cols] of N(0, sigma); row0 selects a slab of a taller tensor."""
    v = normal(seed, stream, row0 * cols, rows * cols, 0.0, sigma)
    return f64_to_bf16_bits(v).reshape(rows, cols)


def outlier_columns(seed: int, K: int, count: int) -> np.ndarray:
    """`count` distinct column indices of [0, K), by a seeded permutation (sort of uniform keys)."""
    keys = words(seed, STREAM_OUTLIER, 0, K)
    return np.sort(np.argsort(keys, kind="stable")[:count])


def activations_bf16(seed: int, rows: int, K: int, n_outliers: int, factor: float, row0: int = 0,
                     stream: int = STREAM_X) -> np.ndarray:
    """x ~ N(0, 1) with `n_outliers` channels (same columns in every row) multiplied by `factor`."""
    v = normal(seed, stream, row0 * K, rows * K, 0.0, 1.0).reshape(rows, K)
    if n_outliers:
        v[:, outlier_columns(seed, K, n_outliers)] *= factor
    return f64_to_bf16_bits(v)


def token_ids(seed: int, n: int, V: int, set_index: int = 0) -> np.ndarray:
    """n ids uniform in [0, V) (int64); set_index selects one of several disjoint id sets."""
    u = uniform(seed, STREAM_IDS, set_index * n, n)
    return np.minimum((u * V).astype(np.int64), V - 1)


def lora_pair(seed: int, N: int, K: int, rank: int, sigma: float):
    """LoRA A fp32 [rank, K] and B fp32 [N, rank], ~N(0, sigma)."""
    A = normal(seed, STREAM_A, 0, rank * K, 0.0, sigma).astype(np.float32).reshape(rank, K)
    B = normal(seed, STREAM_B, 0, N * rank, 0.0, sigma).astype(np.float32).reshape(N, rank)
    return A, B


# Workloads (sizes, distributions and structure of the pages' use of the layer).
WORKLOADS = {
    "tiny": dict(M=64, K=256, N=128, block=32, x_outliers=4, x_factor=20.0, w_sigma=0.02),
    "img1024": dict(M=4096, K=4096, N=4096, block=128, x_outliers=41, x_factor=30.0, w_sigma=0.02),
    "qkv_lora": dict(M=4096, K=4096, N=12288, block=128, x_outliers=41, x_factor=30.0, w_sigma=0.02,
                     lora_rank=16, lora_alpha=16.0, lora_scale=1.0, lora_sigma=0.01),
    "train20k": dict(M=20480, K=4096, N=16384, block=128, x_outliers=41, x_factor=30.0, w_sigma=0.02,
                     dy_sigma=1e-3),
    "embed": dict(V=248000, D=4096, block=128, table_sigma=0.02, n_ids=8192, id_sets=8),
}
