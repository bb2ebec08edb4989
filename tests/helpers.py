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


# ------------------------------------------------------------ exact ties
#
# Rows whose rotated values land exactly on rounding ties.  With x = H_b w on
# every block (H_b the Sylvester Hadamard matrix, w integer), the block
# transform is u = H_b x = b w exactly (H_b H_b = b I), so the code of element
# j is rne(127 u_j / max|u|).  Each row holds one block w = +-254 e_i (its x is
# +-254 everywhere, the row maximum) and sparse integer blocks with |w| <= 127,
# so the codes are rne(w / 2): every odd w is an exact tie (k + 1/2), which
# round-half-to-even sends to the even neighbour (1.5 -> 2, 2.5 -> 2,
# -0.5 -> 0).  |x| <= 254, so every x is an integer exact in bf16, and all the
# fp32 arithmetic of the transform and of the scaling by 127 / (254 b) = 1 / (2b)
# is exact: no rounding order can move a value off its tie.


def sylvester(b):
    from scipy.linalg import hadamard  # Sylvester order: H[i][j] = (-1)^popcount(i & j)
    return hadamard(b).astype(np.int64)


def tie_coefficients(seed, rows, K, b, small=15, nnz=7):
    """Integer block coefficients w [rows, K] (see above); the row maximum |w| = 254."""
    rng = np.random.default_rng(seed)
    nblk = K // b
    w = np.zeros((rows, nblk, b), dtype=np.int64)
    k = min(b, nnz)
    for r in range(rows):
        for j in range(nblk):
            idx = rng.choice(b, size=k, replace=False)
            vals = rng.integers(-small, small + 1, size=k)
            vals[0] = rng.integers(-127, 128)
            w[r, j, idx] = vals
        jb = int(rng.integers(nblk))
        w[r, jb, :] = 0
        w[r, jb, int(rng.integers(b))] = 254 if rng.integers(2) else -254
    return w.reshape(rows, K)


def blocks_times_h(w, b):
    """w H_b on every block of b along the rows (H_b symmetric: equals H_b w per block)."""
    rows, K = w.shape
    return (w.reshape(rows, K // b, b) @ sylvester(b)).reshape(rows, K)


def int_to_bf16_bits(v):
    """Integers of magnitude <= 256 (exact in bf16) -> bf16 bit patterns."""
    v = np.asarray(v)
    assert np.abs(v).max(initial=0) <= 256
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def tie_rows(seed, rows, K, b):
    """(x bf16 bits [rows, K], expected codes [rows, K], count of exact ties)."""
    w = tie_coefficients(seed, rows, K, b)
    x = blocks_times_h(w, b)
    codes = np.rint(w / 2.0).astype(np.int8)  # numpy rounds half to even
    return int_to_bf16_bits(x), codes, int(np.sum(w % 2 != 0))


def ordered_bf16(bits):
    """bf16 bit patterns -> integers in value order (+0 and -0 both map to 0)."""
    b = np.asarray(bits).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_dequant_elementwise(got_bits, ref_bits, bias_bits=None, mask=None, what="outputs"):
    """Dequantized bf16 outputs against the oracle's, element by element, on outputs
    whose code rows agree (mask): the GPU evaluates acc * (s_x * s_w) + bias in fp32
    (each scale within a few fp32 ulps of the oracle's) and rounds once to bf16, the
    oracle evaluates it in fp64, so the two are at most one bf16 step apart, plus an
    allowance of 2^-19 (|y - bias| + |bias|) for the fp32 roundings where a bias
    cancels the product."""
    g = f64(got_bits)
    r = f64(ref_bits)
    bias = np.zeros(r.shape[-1]) if bias_bits is None else f64(bias_bits)
    if mask is None:
        mask = np.ones(r.shape, dtype=bool)
    step = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(g), np.abs(r)), 2.0 ** -126))) - 7)
    tol = step + 2.0 ** -19 * (np.abs(r - bias) + np.abs(bias))
    bad = mask & (np.abs(g - r) > tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond one bf16 step, e.g. {np.argwhere(bad)[:3]}"
    if bias_bits is None:
        d = np.abs(ordered_bf16(got_bits) - ordered_bf16(ref_bits))
        assert int(d[mask].max(initial=0)) <= 1, f"{what}: more than one bf16 step apart"
    return int(mask.sum())


def tie_bwd_weight(seed, N, K, b, p=16):
    """Inputs of the backward-weight preparation whose transform along N lands on
    exact ties, for b a perfect square (1/sqrt(b) exact).  Every weight row has one
    code sigma_j = +-1 per block of K, at the same position e_j for all rows, so
    (Wq R)[n, k] = tau_k / sqrt(b) with tau_k = sigma_j H[e_j, k mod b]; the row
    scales are s = (H_b w) 2^-p on every block of N with w_0 the largest entry, so
    they are positive and exact.  Then W_eff[n, k] = s_n tau_k / sqrt(b), the
    transform of each row of W_eff^T along N is tau_k sqrt(b) w 2^-p, the row
    maximum comes from the block with w_0 = 254, and the codes are
    tau_k rne(w / 2).  Returns (Wq [N, K], s_w [N], expected WtQ [K, N])."""
    rng = np.random.default_rng(seed)
    H = sylvester(b)
    nb, kb = N // b, K // b
    w = np.zeros((nb, b), dtype=np.int64)
    big = int(rng.integers(nb))
    for i in range(nb):
        idx = rng.choice(np.arange(1, b), size=min(b - 1, 6), replace=False)
        w[i, idx] = rng.integers(-15, 16, size=len(idx))
        w[i, 0] = 254 if i == big else int(rng.integers(120, 254))
    s = (w @ H).reshape(N).astype(np.float64) * 2.0 ** -p
    assert np.all(s > 0)
    Wq = np.zeros((N, K), dtype=np.int8)
    tau = np.empty(K, dtype=np.int64)
    for j in range(kb):
        e = int(rng.integers(b))
        sig = 1 if rng.integers(2) else -1
        Wq[:, j * b + e] = sig
        tau[j * b:(j + 1) * b] = sig * H[e]
    codes = (tau[:, None] * np.rint(w.reshape(N) / 2.0)[None, :]).astype(np.int8)
    return Wq, s.astype(np.float32), codes
