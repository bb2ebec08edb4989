"""Exact rounding ties on every quantizer path of the GPU library.

Codes are round-half-to-even of v / s (the pages attribute their only code
differences to rounding ties: sd-scripts PR #2461 "ConvRot INT8",
Verification; MOSS-Image LoRA training guide, section 7.1).  The general
parity tests allow a one-code difference at near-ties, where fp32 summation
order decides; at an EXACT tie only the even neighbour is right.  The rows
here are built so that every rotated value is exact in fp32 and many land
exactly on k + 1/2 (see helpers.tie_rows): each path must give the even
neighbour on every one of them, equal to the closed form rne(w / 2) and to
the oracle, with no allowance.
"""
import numpy as np
import pytest

import oracle
from helpers import check_scales, codes_of, int_to_bf16_bits, tie_bwd_weight, tie_rows, torch_bf16

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


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).cuda()


def _exact(got, want, ref, what):
    got = np.asarray(got, dtype=np.int8)
    assert np.array_equal(ref, want), f"{what}: the oracle is off the closed form"
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ at exact ties, first at {bad[:4].tolist()}"


# Row lengths: rows of 32-element chunks with one (K <= 16384) or two slots per
# thread (K = 32768), and the TMA-staged kernel (multiples of 64 from 8192 to 16384).
@pytest.mark.parametrize("block", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("K", [512, 4096])
def test_exact_ties_row_kernels(block, K):
    x, want, nties = tie_rows(100 + block + K, 37, K, block)
    assert nties > 0
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(x), block)
    _exact(codes_of(Wq), want, q_ref, f"int8 codes b={block} K={K}")
    check_scales(sw.cpu().numpy(), s_ref)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    _exact(codes_of(xq), want, q_ref, f"fp16-held codes b={block} K={K}")
    check_scales(sx.cpu().numpy(), s_ref)
    assert cr.convrot_get_error() == cr.OK


@pytest.mark.parametrize("K,block", [(8192, 128), (16384, 128), (12288, 256), (8256, 64), (32768, 128)])
def test_exact_ties_long_rows(K, block):
    """8192..16384: the TMA-staged kernel (dY rows of the backward); 32768: two slots per thread."""
    x, want, _ = tie_rows(200 + K + block, 9, K, block)
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    _exact(codes_of(xq), want, q_ref, f"fp16-held codes K={K}")
    check_scales(sx.cpu().numpy(), s_ref)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(x), block)
    _exact(codes_of(Wq), want, q_ref, f"int8 codes K={K}")
    check_scales(sw.cpu().numpy(), s_ref)
    assert cr.convrot_get_error() == cr.OK


@pytest.mark.parametrize("K,block", [(48, 16), (80, 8), (272, 16), (80, 16)])
def test_exact_ties_narrow_kernel(K, block):
    """Row lengths that are not a multiple of 32 take the 8-elements-per-thread kernel."""
    x, want, _ = tie_rows(300 + K + block, 41, K, block)
    q_ref, s_ref = oracle.quantize_rows_bf16(x, block)
    xq, sx = cr.convrot_quantize_activation(torch_bf16(x), block)
    _exact(codes_of(xq), want, q_ref, "fp16-held codes (narrow)")
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(x), block)
    _exact(codes_of(Wq), want, q_ref, "int8 codes (narrow)")
    check_scales(sw.cpu().numpy(), s_ref)


def test_exact_ties_narrow_kernel_16_byte_aligned():
    """A 16- but not 32-byte aligned input takes the 8-element kernel at K = 256."""
    N, K, b = 21, 256, 64
    x, want, _ = tie_rows(400, N, K, b)
    ld = K + 8
    full = np.zeros((N, ld + 8), dtype=np.uint16)
    full[:, 8:8 + K] = x
    t = torch_bf16(full)
    Wq = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sw = torch.empty((N,), dtype=torch.float32, device="cuda")
    rc = cr.lib().convrot_quantize_weight(cr.ctypes.c_void_p(t.data_ptr() + 16), N, K, ld + 8, b, None, None, 0,
                                          1.0, 1.0, cr._ptr(Wq), cr._ptr(sw), cr._stream(None))
    assert rc == cr.OK
    q_ref, s_ref = oracle.quantize_rows_bf16(x, b)
    _exact(codes_of(Wq), want, q_ref, "int8 codes (16-byte aligned input)")
    check_scales(sw.cpu().numpy(), s_ref)


def _integer_lora(seed, N, K, rank):
    """A, B with entries in {-1, 0, 1} and at most one nonzero of A per column, so
    every merge term d = sum_j B[n, j] A[j, k] is in {-1, 0, 1} and exact."""
    rng = np.random.default_rng(seed)
    A = np.zeros((rank, K), dtype=np.float32)
    rows = rng.integers(rank, size=K)
    on = rng.random(K) < 0.5
    A[rows[on], np.nonzero(on)[0]] = rng.choice([-1.0, 1.0], size=int(on.sum()))
    B = rng.choice([-1.0, 0.0, 1.0], size=(N, rank)).astype(np.float32)
    d = (B.astype(np.float64) @ A.astype(np.float64))
    assert np.abs(d).max() <= 1
    return A, B, d


# (N, K, rank, block): the cluster kernel (rank <= 16; K split over 8, 2 and 1 CTAs)
# and the row kernel it falls back to (rank 24).
@pytest.mark.parametrize("N,K,rank,block", [(40, 4096, 16, 128), (33, 1024, 5, 64), (20, 512, 8, 256),
                                            (30, 256, 24, 32)])
def test_exact_ties_lora_merge(N, K, rank, block):
    """The merge W' = bf16(W + c B@A) lands exactly on tie rows: an integer adapter with
    c = scale * alpha / rank = 1 and W = x_tie - B@A (integers, exact in bf16), and a
    random adapter with scale 0 (W' = W)."""
    x, want, _ = tie_rows(500 + N + K, N, K, block)
    A, B, d = _integer_lora(600 + rank, N, K, rank)
    xt = np.asarray((x.astype(np.uint32) << 16).view(np.float32), dtype=np.float64)
    W = int_to_bf16_bits((xt - d).astype(np.int64))
    merged = oracle.lora_merge(W, A, B, float(rank), 1.0)
    assert np.array_equal(merged, x), "the integer merge must reproduce the tie rows"
    q_ref, s_ref = oracle.quantize_weight(W, block, A, B, float(rank), 1.0)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), block, _f32(A), _f32(B), float(rank), 1.0)
    _exact(codes_of(Wq), want, q_ref, f"merged codes rank={rank}")
    check_scales(sw.cpu().numpy(), s_ref)
    rng = np.random.default_rng(700 + rank)
    A2 = rng.normal(0, 0.01, size=(rank, K)).astype(np.float32)
    B2 = rng.normal(0, 0.01, size=(N, rank)).astype(np.float32)
    q0, s0 = oracle.quantize_weight(x, block, A2, B2, 16.0, 0.0)
    Wq0, sw0 = cr.convrot_quantize_weight(torch_bf16(x), block, _f32(A2), _f32(B2), 16.0, 0.0)
    _exact(codes_of(Wq0), want, q0, f"scale-0 merge codes rank={rank}")
    check_scales(sw0.cpu().numpy(), s0)
    assert cr.convrot_get_error() == cr.OK


@pytest.mark.parametrize("N,K,block", [(64, 32, 16), (256, 128, 64), (192, 64, 64), (512, 512, 256)])
def test_exact_ties_backward_weight(N, K, block):
    """The one-off int8 backward weight: the double-float transform along N lands on
    exact ties (helpers.tie_bwd_weight); the codes of W_eff^T must be the even neighbours."""
    Wq, s, want = tie_bwd_weight(800 + N + K, N, K, block)
    q_ref, s_ref = oracle.prepare_bwd_weight(Wq, s, block)
    WtQ, swt = cr.convrot_prepare_bwd_weight(_i8(Wq), _f32(s), block)
    _exact(codes_of(WtQ), want, q_ref, f"backward weight codes b={block}")
    check_scales(swt.cpu().numpy(), s_ref)
    assert cr.convrot_get_error() == cr.OK
