"""The generator of `synth`, evaluated with torch on a CUDA device.

Same definition, same stream layout, same results as the numpy version (a GPU
test checks bit equality on samples); it exists so that multi-GB inputs of the
large workloads can be drawn in milliseconds.  Holds no arithmetic of the
ConvRot method.
"""
from __future__ import annotations

import math

import torch

from . import GAMMA, STREAM_OUTLIER, STREAM_X, _M1, _M2, outlier_columns, stream_base

_CHUNK = 1 << 26


def _signed(u: int) -> int:
    u &= 0xFFFFFFFFFFFFFFFF
    return u - (1 << 64) if u >= 1 << 63 else u


_G = _signed(int(GAMMA))
_K1 = _signed(int(_M1))
_K2 = _signed(int(_M2))


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _lsr(z, 30)) * _K1
    z = (z ^ _lsr(z, 27)) * _K2
    return z ^ _lsr(z, 31)


def words(seed: int, stream: int, start: int, count: int, device) -> torch.Tensor:
    base = _signed(stream_base(seed, stream))
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    return _mix(idx * _G + base)


def uniform(seed: int, stream: int, start: int, count: int, device) -> torch.Tensor:
    return (_lsr(words(seed, stream, start, count, device), 11).double() + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, start: int, count: int, device, mu: float = 0.0, sigma: float = 1.0):
    out = torch.empty(count, dtype=torch.float64, device=device)
    pos = 0
    while pos < count:
        n = min(_CHUNK, count - pos)
        i0 = start + pos
        p0 = i0 // 2
        p1 = (i0 + n - 1) // 2 + 1
        u = uniform(seed, stream, 2 * p0, 2 * (p1 - p0), device).view(-1, 2)
        r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
        t = 2.0 * math.pi * u[:, 1]
        z = torch.stack([r * torch.cos(t), r * torch.sin(t)], dim=1).reshape(-1)
        off = i0 - 2 * p0
        out[pos:pos + n] = z[off:off + n]
        pos += n
    return out * sigma + mu


def f64_to_bf16(v: torch.Tensor) -> torch.Tensor:
    """Round fp64 to bf16 (nearest, ties to even) in one rounding; returns torch.bfloat16."""
    f = v.float()
    b = f.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    lo = b & 0xFFFF0000
    hi = lo + 0x10000
    flo = _u32_to_f32(lo).double()
    fhi = _u32_to_f32(hi & 0xFFFFFFFF).double()
    at_inf = (hi & 0x7FFFFFFF) == 0x7F800000
    fhi = torch.where(at_inf, torch.copysign(torch.full_like(flo, 2.0 ** 128), flo), fhi)
    dlo = (v - flo).abs()
    dhi = (v - fhi).abs()
    even_lo = ((lo >> 16) & 1) == 0
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ~even_lo)
    res = torch.where(pick_hi, hi, lo) >> 16
    res = torch.where(res >= 1 << 15, res - (1 << 16), res)
    return res.to(torch.int16).view(torch.bfloat16)


def _u32_to_f32(u: torch.Tensor) -> torch.Tensor:
    s = torch.where(u >= 1 << 31, u - (1 << 32), u).to(torch.int32)
    return s.view(torch.float32)


def normal_bf16(seed: int, stream: int, rows: int, cols: int, sigma: float, device, row0: int = 0):
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    total = rows * cols
    pos = 0
    while pos < total:
        n = min(_CHUNK, total - pos)
        flat[pos:pos + n] = f64_to_bf16(normal(seed, stream, row0 * cols + pos, n, device, 0.0, sigma))
        pos += n
    return out


def activations_bf16(seed: int, rows: int, K: int, n_outliers: int, factor: float, device, row0: int = 0,
                     stream: int = STREAM_X):
    out = torch.empty((rows, K), dtype=torch.bfloat16, device=device)
    cols = torch.from_numpy(outlier_columns(seed, K, n_outliers)).to(device) if n_outliers else None
    step = max(1, _CHUNK // K)
    for r in range(0, rows, step):
        nr = min(step, rows - r)
        v = normal(seed, stream, (row0 + r) * K, nr * K, device).view(nr, K)
        if cols is not None:
            v[:, cols] *= factor
        out[r:r + nr] = f64_to_bf16(v)
    return out


def token_ids(seed: int, n: int, V: int, device, set_index: int = 0) -> torch.Tensor:
    from . import STREAM_IDS
    u = uniform(seed, STREAM_IDS, set_index * n, n, device)
    return torch.clamp((u * V).to(torch.int64), max=V - 1)


def lora_pair(seed: int, N: int, K: int, rank: int, sigma: float, device):
    from . import STREAM_A, STREAM_B
    A = normal(seed, STREAM_A, 0, rank * K, device, 0.0, sigma).float().view(rank, K)
    B = normal(seed, STREAM_B, 0, N * rank, device, 0.0, sigma).float().view(N, rank)
    return A, B


__all__ = ["words", "uniform", "normal", "f64_to_bf16", "normal_bf16", "activations_bf16", "token_ids", "lora_pair",
           "STREAM_OUTLIER"]
