"""Shared helpers of the GPU parity tests (marshalling and comparison rules)."""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth

# Tolerances (the layer's stated acceptance rules):
#   int8 codes: differ by at most 1, on at most 1e-5 of the elements, and only at
#               rounding near-ties (|frac(v/s) - 1/2| < 1e-4);
#   int32 accumulators: bit-exact;
#   bf16 outputs: relative Frobenius error <= 1e-2 against the oracle and
#               <= 5e-2 against the unquantized bf16 matmul.
CODE_MISMATCH_FRAC = 1e-5
NEAR_TIE = 1e-4
REL_FRO_ORACLE = 1e-2
REL_FRO_BF16 = 5e-2
SCALE_RTOL = 2.0 ** -21   # a few fp32 ulps: the scale is one fp32 rounding of the same max


def torch_bf16(bits, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bits_of(t):
    """bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def codes_of(t):
    """int8 or fp16-held code tensor -> numpy int8."""
    import torch
    a = t.detach().cpu()
    if a.dtype == torch.float16:
        f = a.float().numpy()
        assert np.all(f == np.rint(f)) and np.abs(f).max(initial=0) <= 127
        return f.astype(np.int8)
    return a.numpy().astype(np.int8)


def f64(bits):
    return synth.bf16_bits_to_f64(bits)


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def exact_ratio(x_f64, b):
    """v / s in fp64 for every element (the quantity whose rounding gives the code)."""
    v = oracle.rotate_rows(x_f64, b)
    amax = np.abs(v).max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(amax > 0, v * 127.0 / amax, 0.0)


def check_codes(q_gpu, q_ref, x_f64, b, what="codes"):
    """Apply the code tolerance; x_f64 are the (pre-rotation) rows in fp64."""
    q_gpu = np.asarray(q_gpu, dtype=np.int16)
    q_ref = np.asarray(q_ref, dtype=np.int16)
    assert q_gpu.shape == q_ref.shape
    diff = q_gpu != q_ref
    n = int(diff.sum())
    if n == 0:
        return 0
    assert np.abs(q_gpu - q_ref).max() <= 1, f"{what}: a code differs by more than 1"
    assert n <= max(1, math.ceil(CODE_MISMATCH_FRAC * q_gpu.size)), f"{what}: {n} of {q_gpu.size} codes differ"
    rows = np.unique(np.nonzero(diff)[0])
    ratio = exact_ratio(x_f64[rows], b)
    sub = diff[rows]
    f = np.abs(ratio[sub])
    assert np.all(np.abs(f - np.floor(f) - 0.5) < NEAR_TIE), f"{what}: a differing code is not at a near-tie"
    return n


def check_scales(s_gpu, s_ref, what="scales"):
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    s_ref = np.asarray(s_ref, dtype=np.float64)
    np.testing.assert_allclose(s_gpu, s_ref, rtol=SCALE_RTOL, atol=0, err_msg=what)
