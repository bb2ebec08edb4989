"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or mathematics fix:
hand-worked fixtures under tests/golden/, library routines that compute the
same textbook objects (scipy's Sylvester Hadamard, numpy matmul), closed
forms, invariants of an orthogonal rotation, and brute force on tiny inputs.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
import synth
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(v):
    return synth.f64_to_bf16_bits(np.asarray(v, dtype=np.float64))


def _f64(h):
    return synth.bf16_bits_to_f64(h)


def _kron_rotation(K, b):
    """Dense R = I (x) H_b / sqrt(b) from scipy's (Sylvester-order) Hadamard."""
    return np.kron(np.eye(K // b), scipy.linalg.hadamard(b).astype(np.float64) / math.sqrt(b))


def _near_tie(v_over_s, tol=1e-4):
    f = np.abs(v_over_s) - np.floor(np.abs(v_over_s))
    return np.abs(f - 0.5) < tol


# ------------------------------------------------------------------ Hadamard


def test_hadamard_h2_literal():
    assert oracle.hadamard(2).tolist() == [[1.0, 1.0], [1.0, -1.0]]


def test_hadamard_golden_h4_h8():
    lines = read_golden("hadamard_sylvester_4_8.txt")
    i = 0
    while i < len(lines):
        b = int(lines[i])
        rows = [list(map(float, lines[i + 1 + r].split())) for r in range(b)]
        assert oracle.hadamard(b).tolist() == rows
        i += 1 + b


@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_matches_scipy_and_is_orthogonal(b):
    H = oracle.hadamard(b)
    assert np.array_equal(H, scipy.linalg.hadamard(b).astype(np.float64))
    assert np.array_equal(H @ H.T, b * np.eye(b))
    assert np.array_equal(H, H.T)


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(RuntimeError):
        oracle.hadamard(12)


# ------------------------------------------------------------------ rotation


@pytest.mark.parametrize("b", [32, 64, 128, 256])
def test_rotation_equals_dense_block_diagonal_product(b):
    K = 2 * b
    x = synth.normal(3, 0, 0, 5 * K).reshape(5, K)
    got = oracle.rotate_rows(x, b)
    want = x @ _kron_rotation(K, b)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("b", [32, 128])
def test_rotation_preserves_norms_and_products(b):
    K = 4 * b
    x = synth.normal(4, 0, 0, 8 * K).reshape(8, K)
    w = synth.normal(4, 1, 0, 6 * K).reshape(6, K)
    xr = oracle.rotate_rows(x, b)
    wr = oracle.rotate_rows(w, b)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    prod = x @ w.T
    np.testing.assert_allclose(xr @ wr.T, prod, rtol=0, atol=1e-12 * np.abs(prod).max())
    # R is an involution (symmetric and orthogonal): rotating twice is the identity.
    np.testing.assert_allclose(oracle.rotate_rows(xr, b), x, rtol=0, atol=1e-12)


def test_rotation_of_one_hot_spreads_evenly():
    b = 128
    x = np.zeros((1, b))
    x[0, 37] = 3.0
    v = oracle.rotate_rows(x, b)[0]
    np.testing.assert_allclose(np.abs(v), 3.0 / math.sqrt(b), rtol=1e-15)
    np.testing.assert_array_equal(np.sign(v), scipy.linalg.hadamard(b)[37])


# ------------------------------------------------------------------ bf16


def test_bf16_rounding_golden():
    for line in read_golden("bf16_rounding.txt"):
        val, bits = (t.strip() for t in line.split("|"))
        v = float.fromhex(val) if "0x" in val else float(val)
        assert oracle.f64_to_bf16(v) == int(bits, 16), val
        assert int(synth.f64_to_bf16_bits(np.array([v]))[0]) == int(bits, 16), val


def test_bf16_roundtrip_exact():
    h = np.arange(0, 0x7F80, 7, dtype=np.uint16)
    for bits in h[::97]:
        assert oracle.f64_to_bf16(oracle.bf16_to_f64(int(bits))) == int(bits)


# ------------------------------------------------------------------ quantizer


def test_quantizer_golden_hand_cases():
    for line in read_golden("quant_hand_cases.txt"):
        name, b, xs, snum, codes = (t.strip() for t in line.split("|"))
        b = int(b)
        x = np.array([list(map(float, xs.split()))])
        q, s = oracle.quantize_rows_bf16(_bf16(x), b)
        assert q[0].tolist() == list(map(int, codes.split())), name
        assert s[0] == np.float32(float(snum) / 127.0), name


@pytest.mark.parametrize("b", [32, 64, 128, 256])
def test_quantizer_invariants(b):
    K = 4 * b
    x = synth.activations_bf16(11, 16, K, 4, 20.0)
    q, s = oracle.quantize_rows_bf16(x, b)
    v = oracle.rotate_rows(_f64(x), b)
    amax = np.abs(v).max(axis=1)
    np.testing.assert_allclose(s, (amax / 127.0).astype(np.float32), rtol=0, atol=0)
    # the amax element maps to +-127 and no code leaves [-127, 127]
    arg = np.abs(v).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(16), arg]) == 127)
    assert q.min() >= -127 and q.max() <= 127
    # reconstruction error at most half a step per element (plus fp32 slack)
    err = np.abs(s[:, None].astype(np.float64) * q - v)
    assert np.all(err <= s[:, None] * (0.5 + 1e-5))


def test_quantizer_b1_is_textbook_absmax_int8():
    K = 96
    x = synth.activations_bf16(12, 20, K, 3, 25.0)
    q, s = oracle.quantize_rows_bf16(x, 1)
    xf = _f64(x)
    sd = np.abs(xf).max(axis=1, keepdims=True) / 127.0
    want = np.clip(np.rint(xf / sd), -127, 127)
    ratio = xf / sd
    diff = q != want
    assert diff.sum() == 0 or np.all(_near_tie(ratio[diff]))
    np.testing.assert_array_equal(s, (sd[:, 0]).astype(np.float32))


@pytest.mark.parametrize("b", [32, 128])
def test_quantizer_brute_force_fp64_definition(b):
    """Against round(v/s) of the dense fp64 definition: equal except at near-ties."""
    K = 2 * b
    x = synth.activations_bf16(13, 64, K, 2, 30.0)
    q, s = oracle.quantize_rows_bf16(x, b)
    v = _f64(x) @ _kron_rotation(K, b)
    sd = np.abs(v).max(axis=1, keepdims=True) / 127.0
    ratio = v / sd
    want = np.clip(np.rint(ratio), -127, 127)
    diff = q != want
    assert np.all(np.abs(q - want) <= 1)
    assert diff.sum() == 0 or np.all(_near_tie(ratio[diff]))


@pytest.mark.parametrize("b", [8, 16, 32, 64, 128, 256])
def test_quantizer_exact_ties_round_half_to_even_in_bulk(b):
    """Rows built as x = H_b w per block (integer w, one block +-254 e_i per row) rotate
    exactly to u = b w, so the codes are rne(127 w / 254) = rne(w / 2): every odd w is an
    exact tie and must go to the even neighbour (1.5 -> 2, 2.5 -> 2, -0.5 -> 0), and the
    scale is 254 sqrt(b) / 127 = 2 sqrt(b).  A quantizer that rounded ties away from zero
    or truncated would fail on hundreds of elements here."""
    from helpers import tie_rows
    x, want, nties = tie_rows(b, 12, 2048, b)
    assert nties > 100
    q, s = oracle.quantize_rows_bf16(x, b)
    np.testing.assert_array_equal(q, want)
    np.testing.assert_array_equal(s, np.float32(2.0 * math.sqrt(b)))


@pytest.mark.parametrize("b", [16, 64, 256])
def test_bwd_weight_exact_ties_round_half_to_even(b):
    """The backward weight of a constructed base (one +-1 code per block of K, row scales
    (H_b w) 2^-16 along N) transforms along N to exact ties; its codes are tau_k rne(w / 2)."""
    from helpers import tie_bwd_weight
    Wq, s, want = tie_bwd_weight(b, 2 * b, 2 * b, b)
    q, _ = oracle.prepare_bwd_weight(Wq, s, b)
    np.testing.assert_array_equal(q, want)


def test_quantizer_zero_row_and_ldx():
    x = np.zeros((3, 64), dtype=np.uint16)
    x[1] = _bf16(synth.normal(1, 0, 0, 64))
    q, s = oracle.quantize_rows_bf16(x, 32)
    assert s[0] == 0 and s[2] == 0 and np.all(q[0] == 0) and np.all(q[2] == 0)
    assert s[1] > 0


def test_rotation_reduces_outlier_quantization_error():
    """The rotation smooths activation outliers (guide section 7.1): with outlier
    channels the int8 GEMM error must drop when b grows from 1 to 128."""
    M, K, N = 32, 512, 48
    x = synth.activations_bf16(21, M, K, 5, 30.0)
    w = synth.normal_bf16(21, synth.STREAM_W, N, K, 0.02)
    ref = _f64(x) @ _f64(w).T
    errs = {}
    for b in (1, 128):
        wq, sw = oracle.quantize_weight(w, b)
        y, _, _ = oracle.linear_fwd(x, wq, sw, b)
        errs[b] = np.linalg.norm(_f64(y) - ref) / np.linalg.norm(ref)
    assert errs[128] < 0.5 * errs[1]
    assert errs[128] < 5e-2


# ------------------------------------------------------------------ GEMM / epilogue


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (17, 9, 64), (64, 128, 256)])
def test_gemm_s32_brute_force(shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    B = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    C = oracle.gemm_s32(A, B)
    want = A.astype(np.int64) @ B.astype(np.int64).T
    np.testing.assert_array_equal(C, want.astype(np.int32))
    # not transposed the other way round
    if M != N and M > 1:
        assert not np.array_equal(C.shape, (N, M))


def test_gemm_s32_extreme_values_and_overflow():
    K = 4096
    A = np.full((2, K), 127, dtype=np.int8)
    B = np.full((3, K), -127, dtype=np.int8)
    B[1] = 127
    C = oracle.gemm_s32(A, B)
    assert C[0, 0] == -127 * 127 * K and C[0, 1] == 127 * 127 * K
    big = np.full((1, 140000), 127, dtype=np.int8)
    with pytest.raises(RuntimeError):
        oracle.gemm_s32(big, big)


def test_dequant_hand_values():
    acc = np.array([[100, -7], [0, 3]], dtype=np.int32)
    sa = np.array([0.5, 2.0], dtype=np.float32)
    sb = np.array([0.25, 1.0], dtype=np.float32)
    bias = _bf16([1.0, -0.5])
    y = _f64(oracle.dequant(acc, sa, sb))
    np.testing.assert_array_equal(y, [[12.5, -3.5], [0.0, 6.0]])
    yb = _f64(oracle.dequant(acc, sa, sb, bias))
    np.testing.assert_array_equal(yb, [[13.5, -4.0], [1.0, 5.5]])


def test_linear_fwd_close_to_unquantized_matmul():
    M, K, N, b = 64, 256, 128, 32
    x = synth.activations_bf16(0, M, K, 4, 20.0)
    w = synth.normal_bf16(0, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(w, b)
    y, xq, sx = oracle.linear_fwd(x, wq, sw, b)
    ref = _f64(x) @ _f64(w).T
    rel = np.linalg.norm(_f64(y) - ref) / np.linalg.norm(ref)
    assert rel < 5e-2
    # the pieces compose: y == dequant(gemm(xq, wq))
    np.testing.assert_array_equal(y, oracle.dequant(oracle.gemm_s32(xq, wq), sx, sw))


# ------------------------------------------------------------------ LoRA


def test_lora_merge_identities_and_value():
    N, K, r = 24, 64, 4
    w = synth.normal_bf16(5, synth.STREAM_W, N, K, 0.02)
    A, B = synth.lora_pair(5, N, K, r, 0.01)
    assert np.array_equal(oracle.lora_merge(w, A, B, 16.0, 0.0), w)
    assert np.array_equal(oracle.lora_merge(w, A, np.zeros_like(B), 16.0, 1.0), w)
    merged = oracle.lora_merge(w, A, B, 8.0, 1.0)
    want = _f64(w) + (8.0 / r) * (B.astype(np.float64) @ A.astype(np.float64))
    got = _f64(merged)
    # within half a bf16 step of the exact merge (plus fp32 evaluation slack)
    step = 2.0 ** (np.floor(np.log2(np.abs(want))) - 7)
    assert np.all(np.abs(got - want) <= 0.5 * step * (1 + 1e-3))
    qm, sm = oracle.quantize_weight(w, 32, A, B, 8.0, 1.0)
    qr, sr = oracle.quantize_rows_bf16(merged, 32)
    assert np.array_equal(qm, qr) and np.array_equal(sm, sr)
    q0, s0 = oracle.quantize_weight(w, 32, A, B, 8.0, 0.0)
    qp, sp = oracle.quantize_weight(w, 32)
    assert np.array_equal(q0, qp) and np.array_equal(s0, sp)


def test_lora_bypass_forward():
    M, K, N, b, r = 24, 256, 64, 32, 8
    x = synth.activations_bf16(20, M, K, 4, 20.0)
    w = synth.normal_bf16(20, synth.STREAM_W, N, K, 0.02)
    A, B = synth.lora_pair(20, N, K, r, 0.05)
    wq, sw = oracle.quantize_weight(w, b)
    # scale 0 is the plain forward, bit for bit
    y0, _, _ = oracle.linear_fwd(x, wq, sw, b)
    np.testing.assert_array_equal(oracle.linear_fwd_lora(x, wq, sw, b, A, B, 16.0, 0.0), y0)
    # zero weight codes leave only the branch: the closed form c * x A^T B^T (numpy), one bf16 rounding
    c = float(np.float32(1.0 * 16.0 / r))
    yz = oracle.linear_fwd_lora(x, np.zeros_like(wq), sw, b, A, B, 16.0, 1.0)
    ref = _bf16(c * ((_f64(x) @ A.astype(np.float64).T) @ B.astype(np.float64).T))
    assert np.all(np.abs(yz.astype(np.int32) - ref.astype(np.int32)) <= 1)
    # the bypass and the merged weight compute the same layer up to quantization
    y = oracle.linear_fwd_lora(x, wq, sw, b, A, B, 16.0, 1.0)
    merged = _f64(w) + c * (B.astype(np.float64) @ A.astype(np.float64))
    full = _f64(x) @ merged.T
    assert np.linalg.norm(_f64(y) - full) / np.linalg.norm(full) < 5e-2
    lora_only = c * (_f64(x) @ A.astype(np.float64).T) @ B.astype(np.float64).T
    assert np.linalg.norm(lora_only) > 0.1 * np.linalg.norm(full)   # the branch is not negligible here


# ------------------------------------------------------------------ backward


def test_bwd_weight_prep_recovers_base_and_bwd_close_to_bf16():
    M, K, N, b = 48, 128, 256, 32
    w = synth.normal_bf16(7, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(w, b)
    wtq, swt = oracle.prepare_bwd_weight(wq, sw, b)
    assert wtq.shape == (K, N) and swt.shape == (K,)
    w_eff = (sw[:, None].astype(np.float64) * wq) @ _kron_rotation(K, b)   # [N, K]
    back = (swt[:, None].astype(np.float64) * wtq) @ _kron_rotation(N, b)  # [K, N] in original basis
    err = np.abs(back - w_eff.T)
    assert np.all(err <= math.sqrt(b) * swt[:, None] * 0.5 * (1 + 1e-6))
    dy = synth.normal_bf16(7, synth.STREAM_DY, M, N, 1e-3)
    dx, dyq, sdy = oracle.linear_bwd_x(dy, wtq, swt, b)
    ref = _f64(dy) @ _f64(w)
    rel = np.linalg.norm(_f64(dx) - ref) / np.linalg.norm(ref)
    assert rel < 5e-2
    np.testing.assert_array_equal(dx, oracle.dequant(oracle.gemm_s32(dyq, wtq), sdy, swt))


def test_bf16_gemm_brute_force_and_numpy():
    rng = np.random.default_rng(11)
    A = _bf16(rng.normal(size=(3, 7)))
    B = _bf16(rng.normal(size=(4, 7)))
    C = oracle.gemm_bf16(A, B)
    for m in range(3):          # pure-Python loops: the fp64 sum in k order, then one rounding
        for n in range(4):
            acc = 0.0
            for k in range(7):
                acc += float(_f64(A[m, k])) * float(_f64(B[n, k]))
            assert C[m, n] == oracle.f64_to_bf16(acc)
    A = synth.normal_bf16(12, 4, 33, 300, 1.0)
    B = synth.normal_bf16(12, 1, 17, 300, 0.5)
    ref = _bf16(_f64(A) @ _f64(B).T)
    C = oracle.gemm_bf16(A, B)
    ulps = np.abs(C.astype(np.int32) - ref.astype(np.int32))
    assert np.all(ulps <= 1) and np.mean(ulps) < 1e-2   # summation order differs from numpy's


def test_bf16_mode_dequant_weight():
    K, N, b = 256, 96, 32
    w = synth.normal_bf16(13, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(w, b)
    t = oracle.dequant_weight_t(wq, sw, b)
    assert t.shape == (K, N) and t.dtype == np.uint16
    # b = 1 (no rotation) is the plain dequantization s * q, rounded to bf16
    wq1, sw1 = oracle.quantize_weight(w, 1)
    np.testing.assert_array_equal(oracle.dequant_weight_t(wq1, sw1, 1),
                                  _bf16(sw1[:, None].astype(np.float64) * wq1).T)
    # the rotated-back weight recovers the base within half a step per element in the
    # rotated basis (orthogonal R), plus one bf16 rounding
    got = _f64(t).T                                              # [N, K]
    per_row = np.linalg.norm(got - _f64(w), axis=1)
    bound = np.sqrt(K) * sw * 0.5 + np.linalg.norm(got, axis=1) * 2.0 ** -8
    assert np.all(per_row <= bound * (1 + 1e-6))
    assert np.linalg.norm(got - _f64(w)) / np.linalg.norm(_f64(w)) < 2e-2
    # it is one bf16 rounding of the W_eff that the int8 mode quantizes along N (a dense
    # product with scipy's Hadamard; where the exact value is 0 the dense product leaves
    # a rounding residue of ~1e-13)
    w_eff = (sw[:, None].astype(np.float64) * wq) @ _kron_rotation(K, b)
    assert np.all(np.abs(_f64(t).T - w_eff) <= np.abs(w_eff) * 2.0 ** -8 + 1e-12)


def test_bf16_mode_grad_x_close_to_bf16_matmul():
    M, K, N, b = 40, 128, 256, 32
    w = synth.normal_bf16(14, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(w, b)
    dy = synth.normal_bf16(14, synth.STREAM_DY, M, N, 1e-3)
    dx = oracle.linear_bwd_x_bf16(dy, wq, sw, b)
    assert dx.shape == (M, K)
    ref = _f64(dy) @ _f64(w)
    rel = np.linalg.norm(_f64(dx) - ref) / np.linalg.norm(ref)
    assert rel < 2e-2
    # the int8 mode is further from the bf16 product than the bf16 mode
    wtq, swt = oracle.prepare_bwd_weight(wq, sw, b)
    dx8, _, _ = oracle.linear_bwd_x(dy, wtq, swt, b)
    assert np.linalg.norm(_f64(dx8) - ref) > np.linalg.norm(_f64(dx) - ref)


def test_int8_backward_second_reading():
    M, K, N = 40, 128, 256
    w = synth.normal_bf16(22, synth.STREAM_W, N, K, 0.02)
    dy = synth.normal_bf16(22, synth.STREAM_DY, M, N, 1e-3)
    for b in (1, 32):
        wq, sw = oracle.quantize_weight(w, b)
        dx, dq, sd = oracle.linear_bwd_x_r2(dy, wq, sw, b)
        # the codes are the per-row absmax codes of the fp32 product dY * s_w, without rotation
        d32 = (_f64(dy).astype(np.float32) * sw[None, :]).astype(np.float64)
        q1, s1 = oracle.quantize_rows_f64(d32, 1)
        np.testing.assert_array_equal(dq, q1)
        np.testing.assert_array_equal(sd, s1)
        acc = dq.astype(np.int64) @ wq.astype(np.int64)            # numpy integer product over N
        if b == 1:   # no rotation: one rounding of s_d * acc
            np.testing.assert_array_equal(dx, _bf16(sd[:, None].astype(np.float64) * acc))
        else:        # the rotation preserves row norms (up to the bf16 rounding)
            base = sd[:, None].astype(np.float64) * acc
            np.testing.assert_allclose(np.linalg.norm(_f64(dx), axis=1), np.linalg.norm(base, axis=1), rtol=4e-3)
        ref = _f64(dy) @ _f64(w)
        assert np.linalg.norm(_f64(dx) - ref) / np.linalg.norm(ref) < 5e-2


# ------------------------------------------------------------------ embedding


def test_embedding_lookup_inverse_rotation_recovers_rows():
    V, D, b = 300, 256, 128
    table = synth.normal_bf16(9, synth.STREAM_TABLE, V, D, 0.02)
    eq, se = oracle.quantize_rows_bf16(table, b)
    ids = synth.token_ids(9, 50, V)
    ids[3] = V          # out of range
    ids[7] = -1         # out of range
    out, bad = oracle.embedding_lookup(ids, eq, se, b)
    assert bad == 2
    assert np.all(out[3] == 0) and np.all(out[7] == 0)
    good = np.array([i for i in range(50) if i not in (3, 7)])
    orig = _f64(table[ids[good]])
    got = _f64(out[good])
    bound = math.sqrt(b) * se[ids[good]][:, None] * 0.5 + np.abs(got) * 2.0 ** -8
    assert np.all(np.abs(got - orig) <= bound * (1 + 1e-6))
    rel = np.linalg.norm(got - orig) / np.linalg.norm(orig)
    assert rel < 2e-2
    # without the inverse rotation the rows do not match (the claim of the PR summary)
    raw = se[ids[good]][:, None].astype(np.float64) * eq[ids[good]]
    assert np.linalg.norm(raw - orig) / np.linalg.norm(orig) > 0.5
