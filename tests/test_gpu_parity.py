"""GPU parity: the CUDA library (called through its C ABI binding) against the
CPU oracle on the same seeded inputs.  Sizes span several 128x256 GEMM tiles,
K chunks of 1024 and ragged tails in M, N and K."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import (REL_FRO_BF16, REL_FRO_ORACLE, bits_of, check_codes, check_dequant_elementwise, check_scales,
                     codes_of, f64, rel_fro, torch_bf16)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    cr.lib()
    assert cr.convrot_get_error() == cr.OK


def _i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _rand_codes(rng, shape):
    return rng.integers(-127, 128, size=shape, dtype=np.int8)


def _agreeing_codes(x_t, xq_ref, Wq_t, wq_ref, b):
    """Masks [M, N] of the outputs whose activation row (first mask), and also whose
    weight row (second mask), have the same codes on the GPU (the forward's own
    quantizer kernel) as in the oracle."""
    xq, _ = cr.convrot_quantize_activation(x_t, b)
    rows = np.all(codes_of(xq) == xq_ref, axis=1)
    cols = np.all(codes_of(Wq_t) == wq_ref, axis=1)
    return rows[:, None] & np.ones(len(cols), dtype=bool)[None, :], rows[:, None] & cols[None, :]


# ------------------------------------------------------------------ GEMM (int32)


@pytest.mark.parametrize("M,N,K", [(1, 16, 16), (128, 256, 64), (129, 272, 1040), (300, 528, 2064), (64, 128, 256),
                                   (17, 48, 4096)])
def test_gemm_s32_bit_exact(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = _rand_codes(rng, (M, K))
    B = _rand_codes(rng, (N, K))
    C = cr.convrot_gemm_s32(_i8(A), _i8(B))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(C.cpu().numpy(), oracle.gemm_s32(A, B))
    assert cr.convrot_get_error() == cr.OK


@pytest.mark.parametrize("K", [1024, 4096, 16384])
def test_gemm_s32_extremes_cross_the_fp32_exact_range(K):
    """All-127 operands drive every partial sum past 2^24 for K > 1040."""
    M, N = 130, 272
    A = np.full((M, K), 127, dtype=np.int8)
    B = np.full((N, K), 127, dtype=np.int8)
    A[1::2] = -127
    B[:, ::3] *= -1
    C = cr.convrot_gemm_s32(_i8(A), _i8(B)).cpu().numpy()
    np.testing.assert_array_equal(C, oracle.gemm_s32(A, B))
    assert abs(int(C[0, 1])) > 1 << 24 or K <= 1040


def test_gemm_at_the_contraction_limit():
    """K = 2^17, the longest contraction the integer GEMM entries accept: all-+-127 operands put sums at
    127 * 127 * 2^17 = 2,114,060,288 in magnitude, still exact in int32. Checked on the int32 path and on the
    widened-weight GEMM of the training step (2048 K blocks, 128 exact fp32 chunks per tile)."""
    K = 1 << 17
    M, N = 3, 32
    A = np.full((M, K), 127, dtype=np.int8)
    A[1] = -127
    A[2, ::2] = -127
    B = np.full((N, K), 127, dtype=np.int8)
    B[1::2] = -127
    B[2, 1::3] = -127
    ref = oracle.gemm_s32(A, B)
    assert int(np.abs(ref).max()) == 127 * 127 * K
    np.testing.assert_array_equal(cr.convrot_gemm_s32(_i8(A), _i8(B)).cpu().numpy(), ref)
    sx = np.full(M, 2.0 ** -24, dtype=np.float32)
    sw = np.linspace(0.5, 2.0, N).astype(np.float32) * np.float32(2.0 ** -8)
    y_ref = oracle.dequant(ref, sx, sw, None)
    w16 = cr.convrot_widen_codes(_i8(B))
    y = bits_of(cr.convrot_gemm_dequant_w16(torch.from_numpy(A.astype(np.float16)).cuda(), _f32(sx), w16, _f32(sw)))
    ulps = np.abs(y.astype(np.int32) - y_ref.astype(np.int32))
    assert np.all(ulps[(y >> 15) == (y_ref >> 15)] <= 1) and np.mean(y == y_ref) > 0.9
    assert cr.convrot_get_error() == cr.OK


def test_gemm_s32_random_signs_long_k():
    rng = np.random.default_rng(5)
    M, N, K = 140, 260 - 4, 16384 + 64
    A = (rng.integers(0, 2, size=(M, K)) * 254 - 127).astype(np.int8)
    B = (rng.integers(0, 2, size=(N, K)) * 254 - 127).astype(np.int8)
    C = cr.convrot_gemm_s32(_i8(A), _i8(B)).cpu().numpy()
    np.testing.assert_array_equal(C, oracle.gemm_s32(A, B))


# ------------------------------------------------------------------ quantizers


@pytest.mark.parametrize("block", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("K", [512, 4096])
def test_quantize_weight_parity(block, K):
    N = 70
    W = synth.normal_bf16(1, synth.STREAM_W, N, K, 0.02)
    W[5] = 0  # an all-zero row
    q_ref, s_ref = oracle.quantize_weight(W, block)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), block)
    check_codes(codes_of(Wq), q_ref, f64(W), block)
    check_scales(sw.cpu().numpy(), s_ref)
    assert float(sw[5]) == 0.0 and int(Wq[5].abs().max()) == 0


@pytest.mark.parametrize("K,block", [(12288, 128), (16384, 128), (32768, 128), (8192, 64), (12288, 256), (8256, 64)])
def test_quantize_long_rows_parity(K, block):
    """Long rows: the TMA-staged kernel (multiples of 64 from 8192 to 16384 elements, including a
    row group narrower than the CTA) and rows longer than one CTA pass; fp16-held and int8 codes."""
    M = 9
    x = synth.activations_bf16(2, M, K, 41, 30.0)
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    check_codes(codes_of(xq), q_ref, f64(x), block)
    check_scales(sx.cpu().numpy(), s_ref)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(x), block)
    check_codes(codes_of(Wq), q_ref, f64(x), block)
    check_scales(sw.cpu().numpy(), s_ref)
    assert cr.convrot_get_error() == cr.OK


@pytest.mark.parametrize("block", [32, 128])
def test_quantize_activation_parity(block):
    M, K = 333, 1024
    x = synth.activations_bf16(3, M, K, 10, 30.0)
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    assert xq.dtype == torch.float16
    check_codes(codes_of(xq), q_ref, f64(x), block)
    check_scales(sx.cpu().numpy(), s_ref)


@pytest.mark.parametrize("N,K,ld,block", [(40, 256, 384, 32), (7, 8192, 8320, 128)])
def test_quantize_weight_with_row_stride(N, K, ld, block):
    """Rows with a stride larger than their length (the second case goes through the
    TMA-staged kernel, whose tensor map carries the stride)."""
    Wfull = synth.normal_bf16(4, synth.STREAM_W, N, ld, 0.02)
    q_ref, s_ref = oracle.quantize_weight(np.ascontiguousarray(Wfull[:, :K]), block)
    t = torch_bf16(Wfull)
    Wq = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    rc = cr.lib().convrot_quantize_weight(cr._ptr(t), N, K, ld, block, None, None, 0, 1.0, 1.0, cr._ptr(Wq),
                                          cr._ptr(sw), cr._stream(None))
    assert rc == cr.OK
    check_codes(codes_of(Wq), q_ref, f64(Wfull[:, :K]), block)
    check_scales(sw.cpu().numpy(), s_ref)
    assert cr.convrot_get_error() == cr.OK


# Cases of the cluster kernel (rank <= 16 padded to 4, 8 or 16; K split into
# power-of-two slices over 1 to 8 CTAs: 512x1, 512x8, 512x2, 512x6, 512x5,
# 2048x6 with 512 threads, 128x3 with one warp; ragged row tiles) and of the
# row kernel it falls back to (rank 24; K = 96).
@pytest.mark.parametrize("N,K,rank,block", [(96, 512, 16, 128), (50, 4096, 16, 128), (33, 1024, 3, 128),
                                            (41, 3072, 16, 128), (23, 2560, 7, 64), (9, 12288, 16, 256),
                                            (20, 384, 5, 128), (30, 256, 24, 32), (17, 96, 4, 32),
                                            (20, 32768, 16, 128)])
def test_quantize_weight_lora_merge_parity(N, K, rank, block):
    W = synth.normal_bf16(6, synth.STREAM_W, N, K, 0.02)
    A, B = synth.lora_pair(6, N, K, rank, 0.01)
    q_ref, s_ref = oracle.quantize_weight(W, block, A, B, 16.0, 1.0)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), block, _f32(A), _f32(B), 16.0, 1.0)
    merged = oracle.lora_merge(W, A, B, 16.0, 1.0)
    check_codes(codes_of(Wq), q_ref, f64(merged), block)
    check_scales(sw.cpu().numpy(), s_ref)
    # scale = 0 reproduces the unmerged path bit for bit
    Wq0, sw0 = cr.convrot_quantize_weight(torch_bf16(W), block, _f32(A), _f32(B), 16.0, 0.0)
    Wqp, swp = cr.convrot_quantize_weight(torch_bf16(W), block)
    assert torch.equal(Wq0, Wqp) and torch.equal(sw0, swp)


def test_quantize_weight_lora_with_row_stride():
    N, K, ld, rank, b = 37, 2048, 2560, 16, 128
    Wfull = synth.normal_bf16(8, synth.STREAM_W, N, ld, 0.02)
    W = np.ascontiguousarray(Wfull[:, :K])
    A, B = synth.lora_pair(8, N, K, rank, 0.01)
    q_ref, s_ref = oracle.quantize_weight(W, b, A, B, 16.0, 1.0)
    t, At, Bt = torch_bf16(Wfull), _f32(A), _f32(B)
    Wq = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    rc = cr.lib().convrot_quantize_weight(cr._ptr(t), N, K, ld, b, cr._ptr(At), cr._ptr(Bt), rank, 16.0, 1.0,
                                          cr._ptr(Wq), cr._ptr(sw), cr._stream(None))
    assert rc == cr.OK and cr.convrot_get_error() == cr.OK
    check_codes(codes_of(Wq), q_ref, f64(oracle.lora_merge(W, A, B, 16.0, 1.0)), b)
    check_scales(sw.cpu().numpy(), s_ref)


def test_fused_qkv_slabs_equal_separate_projections():
    """A fused q/k/v weight is three row slabs: quantization is per row, so each
    slab (with its own LoRA pair, or with its rows of a shared one) quantizes
    through a slab view into the fused buffers, and the fused forward's column
    blocks equal the per-slab forwards bit for bit.  Pre-quantized slabs (codes
    and scales produced elsewhere) are used through the same views."""
    D, K, b, r = 256, 512, 128, 8
    W = synth.normal_bf16(18, synth.STREAM_W, 3 * D, K, 0.02)
    pairs = [synth.lora_pair(18 + s, D, K, r, 0.01) for s in range(3)]
    Wt = torch_bf16(W)
    Wq = torch.empty((3 * D, K), dtype=torch.int8, device="cuda")
    sw = torch.empty((3 * D,), dtype=torch.float32, device="cuda")
    for s, (A, B) in enumerate(pairs):
        rows = slice(s * D, (s + 1) * D)
        cr.convrot_quantize_weight(Wt[rows], b, _f32(A), _f32(B), 16.0, 1.0, Wq=Wq[rows], scale_w=sw[rows])
        q_ref, s_ref = oracle.quantize_weight(np.ascontiguousarray(W[rows]), b, A, B, 16.0, 1.0)
        merged = oracle.lora_merge(np.ascontiguousarray(W[rows]), A, B, 16.0, 1.0)
        check_codes(codes_of(Wq[rows]), q_ref, f64(merged), b, f"slab {s} codes")
        check_scales(sw[rows].cpu().numpy(), s_ref, f"slab {s} scales")
    x = torch_bf16(synth.activations_bf16(18, 200, K, 5, 30.0))
    y = cr.convrot_linear_fwd(x, Wq, sw, b)
    for s in range(3):
        rows = slice(s * D, (s + 1) * D)
        assert torch.equal(cr.convrot_linear_fwd(x, Wq[rows], sw[rows], b), y[:, rows])
    # one LoRA pair over the stacked weight = the same pair's rows per slab
    A, B = synth.lora_pair(21, 3 * D, K, r, 0.01)
    Wq_f, sw_f = cr.convrot_quantize_weight(Wt, b, _f32(A), _f32(B), 16.0, 1.0)
    for s in range(3):
        rows = slice(s * D, (s + 1) * D)
        Wq_s, sw_s = cr.convrot_quantize_weight(Wt[rows], b, _f32(A), _f32(np.ascontiguousarray(B[rows])), 16.0, 1.0)
        assert torch.equal(Wq_s, Wq_f[rows]) and torch.equal(sw_s, sw_f[rows])
    # pre-quantized ingest: oracle codes and scales, split by views, give the fused result per slab
    wq_o, sw_o = oracle.quantize_weight(W, b)
    Wq_o, sw_o_t = _i8(wq_o), _f32(sw_o)
    y_o = cr.convrot_linear_fwd(x, Wq_o, sw_o_t, b)
    for s in range(3):
        rows = slice(s * D, (s + 1) * D)
        assert torch.equal(cr.convrot_linear_fwd(x, Wq_o[rows], sw_o_t[rows], b), y_o[:, rows])


# ------------------------------------------------------------------ fused GEMM + epilogue


@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_dequant_on_oracle_codes(with_bias):
    M, K, N, b = 300, 2048, 528, 128
    x = synth.activations_bf16(7, M, K, 20, 30.0)
    W = synth.normal_bf16(7, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, b)
    xq, sx = oracle.quantize_rows_bf16(x, b)
    bias = synth.normal_bf16(7, 9, 1, N, 0.5)[0] if with_bias else None
    y_ref = oracle.dequant(oracle.gemm_s32(xq, wq), sx, sw, bias)
    y = cr.convrot_gemm_dequant(torch.from_numpy(xq.astype(np.float16)).cuda(), _f32(sx), _i8(wq), _f32(sw),
                                None if bias is None else torch_bf16(bias))
    yb = bits_of(y)
    assert rel_fro(f64(yb), f64(y_ref)) <= REL_FRO_ORACLE
    # the epilogue differs from the fp64 oracle by at most one bf16 rounding step
    ulps = np.abs(yb.astype(np.int32) - y_ref.astype(np.int32))
    same_sign = (yb >> 15) == (y_ref >> 15)
    assert np.all(ulps[same_sign] <= 1)
    assert np.mean(yb == y_ref) > 0.99


@pytest.mark.parametrize("M,K,N", [(300, 1024, 400), (64, 256, 128), (513, 4096, 272), (129, 1088, 272)])
def test_widened_weight_path_is_bit_identical(M, K, N):
    """The widened-weight path (fp16 copy of the codes in the workspace, GEMM without
    in-loop widening) and the fused path give the same bits; both match the oracle."""
    b = 128 if K % 128 == 0 else 32
    x = synth.activations_bf16(19, M, K, 8, 30.0)
    W = synth.normal_bf16(19, synth.STREAM_W, N, K, 0.02)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    wq_ref, sw_ref = oracle.quantize_weight(W, b)
    check_codes(codes_of(Wq), wq_ref, f64(W), b)
    w16 = cr.convrot_widen_codes(Wq)
    assert torch.equal(w16.float(), Wq.float())
    fast = cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b)
    small = torch.empty(cr.convrot_act_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    fused = cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b, workspace=small)
    assert torch.equal(fast, fused)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), b)
    assert torch.equal(cr.convrot_gemm_dequant_w16(xq, sx, w16, sw), cr.convrot_gemm_dequant(xq, sx, Wq, sw))
    # against the oracle, every oracle input from the oracle: the GPU runs on the oracle's codes
    y_ref, _, _ = oracle.linear_fwd(x, wq_ref, sw_ref, b)
    y_o = cr.convrot_linear_fwd(torch_bf16(x), _i8(wq_ref), _f32(sw_ref), b)
    assert rel_fro(f64(bits_of(y_o)), f64(y_ref)) <= REL_FRO_ORACLE
    assert rel_fro(f64(bits_of(fast)), f64(y_ref)) <= REL_FRO_ORACLE
    # int32 path of the widened operand: exact integer sums
    A = np.random.default_rng(19).integers(-127, 128, size=(M, K), dtype=np.int8)
    acc = cr.convrot_gemm_s32(_i8(A), _i8(wq_ref))
    np.testing.assert_array_equal(acc.cpu().numpy(), oracle.gemm_s32(A, wq_ref))


def test_widened_gemm_row_slices_agree():
    """Every output row of the widened-weight GEMM depends only on its own token row, so a large call (80
    token tiles, a ragged last one, the raster of its shape) and calls on row slices of it (other tile
    boundaries, other rasters, ragged first and last tiles) give the same rows bit for bit, and the fused
    single-CTA kernel agrees."""
    M, K, N, b = 20000, 256, 16384, 128
    x = synth.activations_bf16(23, M, K, 8, 30.0)
    W = synth.normal_bf16(23, synth.STREAM_W, N, K, 0.02)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    w16 = cr.convrot_widen_codes(Wq)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), b)
    bias = torch_bf16(synth.normal_bf16(23, 9, 1, N, 0.5)[0])
    y = cr.convrot_gemm_dequant_w16(xq, sx, w16, sw, bias=bias)
    for r0, r1 in [(0, 4096), (M - 300, M), (7777, 7777 + 513)]:
        ys = cr.convrot_gemm_dequant_w16(xq[r0:r1].clone(), sx[r0:r1].clone(), w16, sw, bias=bias)  # fresh, aligned
        assert torch.equal(ys, y[r0:r1]), (r0, r1)
    yf = cr.convrot_gemm_dequant(xq[:4096].clone(), sx[:4096].clone(), Wq, sw, bias=bias)
    assert torch.equal(yf, y[:4096])


@pytest.mark.parametrize("M,K,N,rank,with_bias", [(300, 1024, 272, 16, False), (65, 512, 128, 5, True),
                                                   (513, 4096, 400, 16, True), (65, 256, 128, 8, False),
                                                   (40, 1056, 96, 16, True), (5, 256, 4096, 16, True),
                                                   (1, 512, 2064, 3, False), (33, 32, 48, 1, True),
                                                   (70, 96, 272, 7, False), (17, 32768, 272, 16, True)])
def test_linear_fwd_lora_bypass_parity(M, K, N, rank, with_bias):
    """Shapes cover one column span (K = 256), 2, 4 and 8 spans (the clusters of the
    down-projection), spans that do not divide K (K = 1056: the last span is empty),
    few rows with many weight rows (the row tiles past M that only write B's
    parts), K = 32 and 96 (a K block only half filled: zeros from the copies of x
    and A), rank 1 and 7, and K = 32768, the longest row (spans of 4096, 32 integer
    chunks per tile before the bypass block)."""
    b = 128 if K % 128 == 0 else 32
    x = synth.activations_bf16(21, M, K, 8, 30.0)
    W = synth.normal_bf16(21, synth.STREAM_W, N, K, 0.02)
    A, B = synth.lora_pair(21, N, K, rank, 0.05)
    bias = synth.normal_bf16(21, 9, 1, N, 0.5)[0] if with_bias else None
    wq, sw = oracle.quantize_weight(W, b)
    y = cr.convrot_linear_fwd_lora(torch_bf16(x), _i8(wq), _f32(sw), b, _f32(A), _f32(B), 16.0, 1.0,
                                   bias=None if bias is None else torch_bf16(bias))
    assert cr.convrot_get_error() == cr.OK
    ref = oracle.linear_fwd_lora(x, wq, sw, b, A, B, 16.0, 1.0, bias)
    yb = bits_of(y)
    assert rel_fro(f64(yb), f64(ref)) <= REL_FRO_ORACLE
    assert np.mean(yb == ref) > 0.9
    # Every output within one bf16 step of the oracle's, plus what fp32 arithmetic leaves where the terms of
    # y = acc * s_x * s_w + bias + L cancel: 2^-19 of the plain terms (as for the plain forward) and 2^-12 of the
    # branch L, whose down-projection the GPU accumulates in fp32 over K (up to 32768 terms).
    g, r = f64(yb), f64(ref)
    step = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(g), np.abs(r)), 2.0 ** -126))) - 7)
    plain = f64(oracle.linear_fwd(x, wq, sw, b)[0])
    branch = (16.0 / rank) * ((f64(x) @ A.T.astype(np.float64)) @ B.T.astype(np.float64))
    cb = np.zeros(N) if bias is None else np.abs(f64(bias))
    tol = step + 2.0 ** -19 * (np.abs(plain) + cb) + 2.0 ** -12 * np.abs(branch)
    # on the token rows whose codes the GPU and the oracle agree on (they may differ by one at near-ties)
    xq_gpu, _ = cr.convrot_quantize_activation(torch_bf16(x), b)
    rows = np.all(xq_gpu.cpu().numpy().astype(np.int64) == oracle.quantize_rows_bf16(x, b)[0].astype(np.int64),
                  axis=1)
    assert rows.mean() > 0.9
    bad = (np.abs(g - r) > tol) & rows[:, None]
    assert not bad.any(), np.argwhere(bad)[:4]
    # scale 0: exactly the plain forward
    y0 = cr.convrot_linear_fwd_lora(torch_bf16(x), _i8(wq), _f32(sw), b, _f32(A), _f32(B), 16.0, 0.0,
                                    bias=None if bias is None else torch_bf16(bias))
    yp = cr.convrot_linear_fwd(torch_bf16(x), _i8(wq), _f32(sw), b, bias=None if bias is None else torch_bf16(bias))
    assert torch.equal(y0, yp)
    # the bypass and the merged-then-quantized weight compute the same layer up to quantization
    c = np.float32(16.0 / rank)
    full = f64(x) @ (f64(W) + float(c) * (B.astype(np.float64) @ A.astype(np.float64))).T
    if bias is not None:
        full = full + f64(bias)
    assert rel_fro(f64(yb), full) <= REL_FRO_BF16


def test_linear_fwd_lora_zero_adapter_is_the_plain_forward():
    """A zero B with a nonzero coefficient runs the bypass kernels with a zero
    branch: the result equals the plain forward bit for bit (the integer sums
    here stay below 2^24, where the fp32 addition of the last chunk is exact)."""
    M, K, N, rank, b = 300, 1024, 400, 16, 128
    x = synth.activations_bf16(25, M, K, 8, 30.0)
    W = synth.normal_bf16(25, synth.STREAM_W, N, K, 0.02)
    A, _ = synth.lora_pair(25, N, K, rank, 0.05)
    B = np.zeros((N, rank), dtype=np.float32)
    bias = torch_bf16(synth.normal_bf16(25, 9, 1, N, 0.5)[0])
    wq, sw = oracle.quantize_weight(W, b)
    y = cr.convrot_linear_fwd_lora(torch_bf16(x), _i8(wq), _f32(sw), b, _f32(A), _f32(B), 16.0, 1.0, bias=bias)
    assert cr.convrot_get_error() == cr.OK
    assert torch.equal(y, cr.convrot_linear_fwd(torch_bf16(x), _i8(wq), _f32(sw), b, bias=bias))


@pytest.mark.parametrize("lora_sigma", [0.05, 2.0])
def test_linear_fwd_lora_bypass_zero_rows_and_large_branch(lora_sigma):
    """All-zero rows of x and of W (scale 0, codes 0): those outputs are bias +
    the branch alone.  lora_sigma = 2 makes the branch larger than the base
    product, so the branch carries most of each output.  scale = 0 still gives
    the plain forward bit for bit, zero rows included."""
    M, K, N, rank, b = 300, 1024, 400, 16, 128
    x = synth.activations_bf16(23, M, K, 8, 30.0)
    x[[3, 100, 299]] = 0
    W = synth.normal_bf16(23, synth.STREAM_W, N, K, 0.02)
    W[[5, 130, 399]] = 0
    A, B = synth.lora_pair(23, N, K, rank, lora_sigma)
    bias = synth.normal_bf16(23, 9, 1, N, 0.5)[0]
    wq, sw = oracle.quantize_weight(W, b)
    assert sw[5] == 0 and not wq[5].any()
    args = (torch_bf16(x), _i8(wq), _f32(sw), b, _f32(A), _f32(B), 16.0)
    y = cr.convrot_linear_fwd_lora(*args, 1.0, bias=torch_bf16(bias))
    assert cr.convrot_get_error() == cr.OK
    ref = oracle.linear_fwd_lora(x, wq, sw, b, A, B, 16.0, 1.0, bias)
    yb = bits_of(y)
    ulps = np.abs(yb.astype(np.int32) - ref.astype(np.int32))
    same_sign = (yb >> 15) == (ref >> 15)
    assert np.mean(ulps[same_sign] <= 1) > 0.999 and np.mean(yb == ref) > 0.9
    zr = np.ix_([3, 100, 299], np.arange(N))
    zc = np.ix_(np.arange(M), [5, 130, 399])
    for sel in (zr, zc):
        d = np.abs(yb[sel].astype(np.int32) - ref[sel].astype(np.int32))
        assert np.all(d[(yb[sel] >> 15) == (ref[sel] >> 15)] <= 1)
    y0 = cr.convrot_linear_fwd_lora(*args, 0.0, bias=torch_bf16(bias))
    assert torch.equal(y0, cr.convrot_linear_fwd(torch_bf16(x), _i8(wq), _f32(sw), b, bias=torch_bf16(bias)))


@pytest.mark.parametrize("case", range(8))
def test_randomized_small_shapes(case):
    """Seeded random shapes: M not a multiple of the tile, N a multiple of 16, every block size,
    an all-zero activation row and an all-zero weight row."""
    rng = np.random.default_rng(1000 + case)
    b = int(rng.choice([32, 64, 128, 256]))
    K = b * int(rng.integers(1, 1024 // b + 1))
    if K % 16:
        K = b * 2
    M = int(rng.integers(1, 700))
    N = 16 * int(rng.integers(1, 40))
    x = synth.activations_bf16(2000 + case, M, K, int(rng.integers(0, 8)), 25.0)
    W = synth.normal_bf16(2000 + case, synth.STREAM_W, N, K, 0.02)
    x[rng.integers(0, M)] = 0
    W[rng.integers(0, N)] = 0
    wq_ref, sw_ref = oracle.quantize_weight(W, b)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    check_codes(codes_of(Wq), wq_ref, f64(W), b)
    check_scales(sw.cpu().numpy(), sw_ref)
    y = cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b)
    small = torch.empty(cr.convrot_act_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    assert torch.equal(y, cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b, workspace=small))
    y_ref, xq_ref, _ = oracle.linear_fwd(x, wq_ref, sw_ref, b)
    assert rel_fro(f64(bits_of(y)), f64(y_ref)) <= REL_FRO_ORACLE
    y_o = cr.convrot_linear_fwd(torch_bf16(x), _i8(wq_ref), _f32(sw_ref), b)
    assert rel_fro(f64(bits_of(y_o)), f64(y_ref)) <= REL_FRO_ORACLE
    # element by element wherever the code rows agree (all but near-tie rows)
    xrows, mask = _agreeing_codes(torch_bf16(x), xq_ref, Wq, wq_ref, b)
    assert mask.mean() > 0.9
    check_dequant_elementwise(bits_of(y), y_ref, mask=mask, what="forward on the GPU's codes")
    check_dequant_elementwise(bits_of(y_o), y_ref, mask=xrows, what="forward on the oracle's weight codes")
    assert cr.convrot_get_error() == cr.OK


def test_linear_fwd_tiny_workload():
    wl = synth.WORKLOADS["tiny"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    x = synth.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"])
    W = synth.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"])
    wq_ref, sw_ref = oracle.quantize_weight(W, b)
    y_ref, xq_ref, sx_ref = oracle.linear_fwd(x, wq_ref, sw_ref, b)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    check_codes(codes_of(Wq), wq_ref, f64(W), b)
    y = cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b)
    yb = f64(bits_of(y))
    assert rel_fro(yb, f64(y_ref)) <= REL_FRO_ORACLE
    assert rel_fro(yb, f64(x) @ f64(W).T) <= REL_FRO_BF16
    xrows, mask = _agreeing_codes(torch_bf16(x), xq_ref, Wq, wq_ref, b)
    assert mask.mean() > 0.9
    check_dequant_elementwise(bits_of(y), y_ref, mask=mask, what="tiny forward")
    y_o = cr.convrot_linear_fwd(torch_bf16(x), _i8(wq_ref), _f32(sw_ref), b)
    check_dequant_elementwise(bits_of(y_o), y_ref, mask=xrows, what="tiny forward on the oracle's weight codes")
    assert cr.convrot_get_error() == cr.OK


def test_linear_fwd_ragged_multi_tile():
    M, K, N, b = 259, 1152, 400, 64
    x = synth.activations_bf16(8, M, K, 12, 30.0)
    W = synth.normal_bf16(8, synth.STREAM_W, N, K, 0.02)
    bias = synth.normal_bf16(8, 9, 1, N, 0.1)[0]
    wq_ref, sw_ref = oracle.quantize_weight(W, b)
    y_ref, _, _ = oracle.linear_fwd(x, wq_ref, sw_ref, b, bias)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    y = cr.convrot_linear_fwd(torch_bf16(x), Wq, sw, b, bias=torch_bf16(bias))
    yb = f64(bits_of(y))
    assert rel_fro(yb, f64(y_ref)) <= REL_FRO_ORACLE
    assert rel_fro(yb, f64(x) @ f64(W).T + f64(bias)) <= REL_FRO_BF16
    _, xq_ref, _ = oracle.linear_fwd(x, wq_ref, sw_ref, b, bias)
    _, mask = _agreeing_codes(torch_bf16(x), xq_ref, Wq, wq_ref, b)
    assert mask.mean() > 0.9
    check_dequant_elementwise(bits_of(y), y_ref, bias_bits=bias, mask=mask, what="ragged forward with bias")


# ------------------------------------------------------------------ backward


@pytest.mark.parametrize("block,K,N", [(32, 256, 768), (128, 256, 768), (16, 48, 400), (8, 80, 272), (64, 192, 320),
                                       (256, 512, 512), (128, 256, 32768)])
def test_bwd_prep_and_grad_x_parity(block, K, N):
    """Tiles of 128 (or b) weight rows and columns, ragged in both, every block size, and N = 32768 (the longest
    row of the backward weight and the longest contraction of grad_x)."""
    M = 150
    W = synth.normal_bf16(9, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    wtq_ref, swt_ref = oracle.prepare_bwd_weight(wq, sw, block)
    WtQ, swt = cr.convrot_prepare_bwd_weight(_i8(wq), _f32(sw), block)
    w_eff_t = ((sw[:, None].astype(np.float64) * wq) @ np.kron(np.eye(K // block), oracle.hadamard(block) /
                                                               math.sqrt(block))).T
    check_codes(codes_of(WtQ), wtq_ref, w_eff_t, block, "bwd weight codes")
    check_scales(swt.cpu().numpy(), swt_ref, "bwd weight scales")
    dY = synth.normal_bf16(9, synth.STREAM_DY, M, N, 1e-3)
    dX_ref, _, _ = oracle.linear_bwd_x(dY, wtq_ref, swt_ref, block)
    dX = cr.convrot_linear_bwd_x(torch_bf16(dY), WtQ, swt, block)
    d = f64(bits_of(dX))
    assert rel_fro(d, f64(dX_ref)) <= REL_FRO_ORACLE
    assert rel_fro(d, f64(dY) @ f64(W)) <= REL_FRO_BF16


# ------------------------------------------------------------------ bf16 backward


def _check_bf16_sums(got_bits, ref_bits, K):
    """bf16 results of fp32-accumulated sums of K terms against the fp64-summed
    oracle: one bf16 rounding step apart (relative), plus an absolute allowance
    for the fp32 accumulation (a random walk of K roundings of about 2^-24 of the
    running sum, with a margin of 64) near zero; almost always identical."""
    g, r = f64(got_bits), f64(ref_bits)
    tol = np.abs(r) * 2.0 ** -7 + 64 * 2.0 ** -24 * math.sqrt(K) * np.sqrt(np.mean(r * r))
    assert np.all(np.abs(g - r) <= tol)
    assert np.mean(got_bits == ref_bits) > 0.98
    assert rel_fro(g, r) <= REL_FRO_ORACLE


@pytest.mark.parametrize("N,K,block", [(80, 256, 32), (192, 1024, 128), (16, 512, 256), (64, 64, 8), (48, 48, 16),
                                       (64, 32768, 128)])
def test_dequant_weight_t_parity(N, K, block):
    W = synth.normal_bf16(15, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    ref = oracle.dequant_weight_t(wq, sw, block)
    got = bits_of(cr.convrot_dequant_weight_t(_i8(wq), _f32(sw), block))
    assert got.shape == (K, N)
    # both sides round a value accurate to >= 44 bits once to bf16: identical
    np.testing.assert_array_equal(got, ref)


def test_dequant_weight_t_rounding_midpoints():
    """Values on and beside bf16 rounding midpoints.  With b = 64 (1/sqrt(b) = 1/8 exact)
    and one code q per row, W_eff = s q H[j, k] / 8 = +-s q / 8; the scales are chosen so
    that s q / 8 lands exactly on a midpoint between two bf16 values (ties go to even), or
    one and a few fp32 steps beside it, across binades; q in {1, 3, 5, 7, 127} makes the
    product inexact in fp32 for most rows.  Every value must be the correctly rounded one."""
    b, K = 64, 128
    rng = np.random.default_rng(41)
    qs, ss = [], []
    for e in range(-12, 3):
        for mant in (0, 37, 101, 127):
            mid = (1.0 + (2 * mant + 1) / 256.0) * 2.0 ** e  # halfway between two bf16 neighbours
            for q in (1, 3, 5, 7, 127):
                for off in (0, 1, -1, 2, -2, 5):
                    s = np.float32(8.0 * mid / q)
                    s = np.nextafter(s, np.float32(np.inf)) if off > 0 else s
                    for _ in range(max(0, abs(off) - 1)):
                        s = np.nextafter(s, np.float32(np.inf) if off > 0 else np.float32(-np.inf))
                    if off < 0:
                        s = np.nextafter(s, np.float32(-np.inf))
                    qs.append(q if rng.integers(2) else -q)
                    ss.append(s)
    N = (len(qs) + 15) // 16 * 16
    wq = np.zeros((N, K), dtype=np.int8)
    sw = np.zeros(N, dtype=np.float32)
    for n, (q, s) in enumerate(zip(qs, ss)):
        wq[n, rng.integers(b)] = q
        wq[n, b + rng.integers(b)] = -q
        sw[n] = s
    ref = oracle.dequant_weight_t(wq, sw, b)
    got = bits_of(cr.convrot_dequant_weight_t(_i8(wq), _f32(sw), b))
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(300, 272, 1008), (64, 128, 64), (513, 400, 4096), (129, 272, 1040)])
def test_gemm_bf16_parity(M, N, K):
    A = synth.normal_bf16(16, synth.STREAM_DY, M, K, 1.0)
    B = synth.normal_bf16(16, synth.STREAM_W, N, K, 0.05)
    got = bits_of(cr.convrot_gemm_bf16(torch_bf16(A), torch_bf16(B)))
    _check_bf16_sums(got, oracle.gemm_bf16(A, B), K)


@pytest.mark.parametrize("block", [32, 128])
def test_linear_bwd_x_bf16_parity(block):
    M, K, N = 300, 384, 528
    W = synth.normal_bf16(17, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    dY = synth.normal_bf16(17, synth.STREAM_DY, M, N, 1e-3)
    ws = torch.empty(cr.convrot_bwd_x_bf16_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    dX = cr.convrot_linear_bwd_x_bf16(torch_bf16(dY), _i8(wq), _f32(sw), block, workspace=ws)
    assert cr.convrot_get_error() == cr.OK
    # the workspace holds the transient W_eff^T
    weff_t = ws[:K * N * 2].view(torch.int16).view(K, N).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(weff_t, oracle.dequant_weight_t(wq, sw, block))
    got = bits_of(dX)
    _check_bf16_sums(got, oracle.linear_bwd_x_bf16(dY, wq, sw, block), N)
    assert rel_fro(f64(got), f64(dY) @ f64(W)) <= REL_FRO_BF16


@pytest.mark.parametrize("M,N,K,block", [(150, 768, 256, 32), (300, 512, 384, 128), (37, 1024, 256, 256), (40, 32768, 256, 128)])
def test_linear_bwd_x_second_reading_parity(M, N, K, block):
    W = synth.normal_bf16(23, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    dY = synth.normal_bf16(23, synth.STREAM_DY, M, N, 1e-3)
    ws = torch.empty(cr.convrot_bwd_x_r2_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    dX = cr.convrot_linear_bwd_x_r2(torch_bf16(dY), _i8(wq), _f32(sw), block, workspace=ws)
    assert cr.convrot_get_error() == cr.OK
    ref, dq_ref, sd_ref = oracle.linear_bwd_x_r2(dY, wq, sw, block)
    # the unrotated codes and scales are decided in the same fp32 arithmetic: identical
    dq = ws[:M * N * 2].view(torch.float16).view(M, N)
    np.testing.assert_array_equal(codes_of(dq), dq_ref)
    off = (M * N * 2 + 255) // 256 * 256
    np.testing.assert_array_equal(ws[off:off + 4 * M].view(torch.float32).cpu().numpy(), sd_ref)
    got = bits_of(dX)
    _check_bf16_sums(got, ref, K)
    assert rel_fro(f64(got), f64(dY) @ f64(W)) <= REL_FRO_BF16


# ------------------------------------------------------------------ embedding


def test_embedding_lookup_parity_and_bad_ids():
    V, D, b = 1000, 512, 128
    table = synth.normal_bf16(10, synth.STREAM_TABLE, V, D, 0.02)
    eq_ref, se_ref = oracle.quantize_rows_bf16(table, b)
    Eq, se = cr.convrot_quantize_weight(torch_bf16(table), b)
    check_codes(codes_of(Eq), eq_ref, f64(table), b)
    ids = synth.token_ids(10, 300, V)
    out = cr.convrot_embedding_lookup(torch.from_numpy(ids).cuda(), _i8(eq_ref), _f32(se_ref), b)
    out_ref, bad = oracle.embedding_lookup(ids, eq_ref, se_ref, b)
    assert bad == 0
    ob = bits_of(out)
    assert rel_fro(f64(ob), f64(out_ref)) <= REL_FRO_ORACLE
    assert np.mean(ob == out_ref) > 0.99
    assert rel_fro(f64(ob), f64(table[ids])) < 2e-2
    assert cr.convrot_get_error() == cr.OK
    ids[[4, 9]] = [V, -3]
    out = cr.convrot_embedding_lookup(torch.from_numpy(ids).cuda(), _i8(eq_ref), _f32(se_ref), b)
    assert cr.convrot_get_error() == cr.ERR_INDEX
    assert cr.convrot_get_error() == cr.OK  # cleared
    ob = bits_of(out)
    assert np.all(ob[4] == 0) and np.all(ob[9] == 0)
    good = [i for i in range(300) if i not in (4, 9)]
    assert rel_fro(f64(ob[good]), f64(out_ref[good])) <= REL_FRO_ORACLE


# ------------------------------------------------------------------ edge cases


def test_empty_problems_are_no_ops():
    W = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    Wq, sw = cr.convrot_quantize_weight(W, 32)
    assert Wq.shape == (0, 256)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    Wq2, sw2 = cr.convrot_quantize_weight(torch.ones((32, 256), dtype=torch.bfloat16, device="cuda"), 32)
    y = cr.convrot_linear_fwd(x, Wq2, sw2, 32)
    assert y.shape == (0, 32)
    out = cr.convrot_embedding_lookup(torch.zeros((0,), dtype=torch.int64, device="cuda"), Wq2, sw2, 32)
    assert out.shape == (0, 256)
    assert cr.convrot_get_error() == cr.OK


def test_argument_errors_raise():
    x = torch.ones((4, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cr.ConvRotError):
        cr.convrot_quantize_activation(x, 64)  # 96 is not a multiple of 64
    with pytest.raises(TypeError):
        cr.convrot_quantize_activation(x.float(), 32)


# ------------------------------------------------------------------ both kernel layouts


@pytest.mark.parametrize("K,block", [(48, 16), (80, 8), (272, 16)])
def test_quantize_rows_not_multiple_of_32(K, block):
    """Row lengths that are not a multiple of 32 take the 8-elements-per-thread kernel."""
    M = 37
    x = synth.activations_bf16(31, M, K, 3, 30.0)
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    check_codes(codes_of(xq), q_ref, f64(x), block)
    check_scales(sx.cpu().numpy(), s_ref)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(x), block)
    check_codes(codes_of(Wq), q_ref, f64(x), block)


def test_quantize_16_byte_aligned_input_takes_the_narrow_path():
    """An input that is 16- but not 32-byte aligned (row stride 264) must give the same codes."""
    N, K, ld, b = 21, 256, 264, 64
    full = synth.normal_bf16(32, synth.STREAM_W, N, ld + 8, 0.02)
    t = torch_bf16(full)
    q_ref, s_ref = oracle.quantize_weight(np.ascontiguousarray(full[:, 8:8 + K]), b)
    Wq = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    base = t.data_ptr() + 16  # column 8: 16-byte aligned, not 32
    # rows of the view: stride ld + 8 elements
    rc = cr.lib().convrot_quantize_weight(cr.ctypes.c_void_p(base), N, K, ld + 8, b, None, None, 0, 1.0, 1.0,
                                          cr._ptr(Wq), cr._ptr(sw), cr._stream(None))
    assert rc == cr.OK
    check_codes(codes_of(Wq), q_ref, f64(full[:, 8:8 + K]), b)
    check_scales(sw.cpu().numpy(), s_ref)


@pytest.mark.parametrize("D,block", [(48, 16), (4096, 128), (512, 256), (32768, 128)])
def test_embedding_lookup_layouts(D, block):
    V = 300
    table = synth.normal_bf16(33, synth.STREAM_TABLE, V, D, 0.02)
    eq, se = oracle.quantize_rows_bf16(table, block)
    ids = synth.token_ids(33, 77, V)
    ref, bad = oracle.embedding_lookup(ids, eq, se, block)
    out = cr.convrot_embedding_lookup(torch.from_numpy(ids).cuda(), _i8(eq), _f32(se), block)
    ob = bits_of(out)
    assert rel_fro(f64(ob), f64(ref)) <= REL_FRO_ORACLE
    assert np.mean(ob == ref) > 0.99
    assert cr.convrot_get_error() == cr.OK
