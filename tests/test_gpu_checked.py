"""The checked variant of the library (libconvrot_checked: the same kernels
compiled with -DCONVROT_CHECKED, every instrumented global-memory access tested
against its tensor's extent) on the parity shapes: no access may leave its
tensor (convrot_get_error stays CONVROT_OK, never CONVROT_ERR_BOUNDS), and every
output must be bit-identical to the release library's, which the parity tests
hold against the oracle.  The shapes take each kernel family through its ragged
edges: rows and columns off the tile sizes, K chunks of 16 past a multiple of
32, the narrow (8-element) and wide (32-element) quantizer paths, the
TMA-staged rows, the cluster LoRA merge and its row-kernel fallback, every
block size of the backward weight, and embedding tables of both layouts."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import torch_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    for variant in ("release", "checked"):
        prev = cr.select_library(variant)
        try:
            assert cr.convrot_get_error() == cr.OK
        finally:
            cr.select_library(prev)
    yield
    cr.select_library("release")


def _i8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int8)).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _raw(t):
    """The bytes of a tensor (or of each tensor of a tuple), on the host."""
    if isinstance(t, (tuple, list)):
        return [_raw(u) for u in t]
    return t.contiguous().view(torch.uint8).cpu().numpy()


def _both(fn):
    """fn() under the release library, then under the checked one; the checked
    run must record no out-of-extent access and match the release bytes."""
    prev = cr.select_library("release")
    try:
        ref = _raw(fn())
        assert cr.convrot_get_error() == cr.OK
        cr.select_library("checked")
        got = _raw(fn())
        status = cr.convrot_get_error()
        assert status == cr.OK, cr.status_string(status)
    finally:
        cr.select_library(prev)
    if isinstance(ref, list):
        for r, g in zip(ref, got):
            np.testing.assert_array_equal(g, r)
    else:
        np.testing.assert_array_equal(got, ref)


def test_bounds_flag_reporting_path():
    """A failed check (one that accesses nothing) reaches convrot_get_error as
    CONVROT_ERR_BOUNDS in the checked library, once; the release library has no
    checks and says so."""
    prev = cr.select_library("checked")
    try:
        assert cr.convrot_get_error() == cr.OK
        assert cr.lib().convrot_selftest_bounds_flag(None) == cr.OK
        assert cr.convrot_get_error() == cr.ERR_BOUNDS
        assert cr.convrot_get_error() == cr.OK  # cleared
    finally:
        cr.select_library(prev)
    assert cr.lib().convrot_selftest_bounds_flag(None) == cr.ERR_UNSUPPORTED
    assert cr.convrot_get_error() == cr.OK


def test_checked_library_is_a_separate_build():
    prev = cr.select_library("checked")
    try:
        L = cr.lib()
        assert L._name == cr.library_path("checked")
        assert cr.status_string(cr.ERR_BOUNDS) == "CONVROT_ERR_BOUNDS"
    finally:
        cr.select_library(prev)
    assert cr.lib()._name == cr.library_path("release")


@pytest.mark.parametrize("M,K,block", [(300, 1040, 16), (129, 4096, 128), (7, 12288, 128), (33, 32768, 128),
                                       (65, 48, 16), (40, 80, 8), (17, 8192, 256), (5, 272, 16)])
def test_checked_quantize_activation(M, K, block):
    x = torch_bf16(synth.activations_bf16(31, M, K, 4, 20.0))
    _both(lambda: cr.convrot_quantize_activation(x, block))


@pytest.mark.parametrize("N,K,ld,block", [(40, 256, 384, 32), (7, 8192, 8320, 128)])
def test_checked_quantize_weight_row_stride(N, K, ld, block):
    Wfull = torch_bf16(synth.normal_bf16(4, synth.STREAM_W, N, ld, 0.02))

    def run():
        Wq = torch.empty((N, K), dtype=torch.int8, device="cuda")
        sw = torch.empty((N,), dtype=torch.float32, device="cuda")
        rc = cr.lib().convrot_quantize_weight(cr._ptr(Wfull), N, K, ld, block, None, None, 0, 1.0, 1.0, cr._ptr(Wq),
                                              cr._ptr(sw), cr._stream(None))
        assert rc == cr.OK
        return Wq, sw

    _both(run)


@pytest.mark.parametrize("N,K,rank,block", [(50, 4096, 16, 128), (33, 1024, 3, 128), (23, 2560, 7, 64),
                                            (30, 256, 24, 32), (17, 96, 4, 32), (20, 32768, 16, 128)])
def test_checked_quantize_weight_lora_merge(N, K, rank, block):
    W = torch_bf16(synth.normal_bf16(6, synth.STREAM_W, N, K, 0.02))
    A, B = synth.lora_pair(6, N, K, rank, 0.01)
    A, B = _f32(A), _f32(B)
    _both(lambda: cr.convrot_quantize_weight(W, block, A, B, 16.0, 1.0))


@pytest.mark.parametrize("M,K,N,block,bias", [(300, 1024, 400, 128, True), (513, 4096, 272, 128, False),
                                              (1, 48, 16, 16, True), (129, 1040, 272, 16, False),
                                              (17, 32768, 272, 128, True)])
def test_checked_linear_fwd(M, K, N, block, bias):
    W = synth.normal_bf16(8, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    x = torch_bf16(synth.activations_bf16(8, M, K, 4, 20.0))
    b = torch_bf16(synth.normal_bf16(8, synth.STREAM_B, 1, N, 0.1)[0]) if bias else None
    Wq, s = _i8(wq), _f32(sw)
    _both(lambda: cr.convrot_linear_fwd(x, Wq, s, block, bias=b))
    _both(lambda: cr.convrot_linear_fwd_noalloc(x, Wq, s, block, bias=b))


@pytest.mark.parametrize("M,K,N,rank", [(300, 1024, 272, 16), (65, 512, 128, 5), (5, 256, 4096, 16),
                                        (17, 32768, 272, 16)])
def test_checked_linear_fwd_lora(M, K, N, rank):
    block = 128
    W = synth.normal_bf16(12, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    A, B = synth.lora_pair(12, N, K, rank, 0.01)
    x = torch_bf16(synth.activations_bf16(12, M, K, 4, 20.0))
    Wq, s, At, Bt = _i8(wq), _f32(sw), _f32(A), _f32(B)
    _both(lambda: cr.convrot_linear_fwd_lora(x, Wq, s, block, At, Bt, 16.0, 1.0))


@pytest.mark.parametrize("block,K,N", [(32, 256, 768), (128, 256, 768), (16, 48, 400), (8, 80, 272),
                                       (64, 192, 320), (256, 512, 512), (128, 256, 32768)])
def test_checked_bwd_weight_and_grad_x(block, K, N):
    M = 150
    W = synth.normal_bf16(9, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    Wq, s = _i8(wq), _f32(sw)
    dY = torch_bf16(synth.normal_bf16(9, synth.STREAM_DY, M, N, 1e-3))
    _both(lambda: cr.convrot_prepare_bwd_weight(Wq, s, block))
    WtQ, swt = cr.convrot_prepare_bwd_weight(Wq, s, block)
    _both(lambda: cr.convrot_linear_bwd_x(dY, WtQ, swt, block))


@pytest.mark.parametrize("N,K,block", [(80, 256, 32), (192, 1024, 128), (16, 512, 256), (64, 64, 8), (48, 48, 16),
                                       (64, 32768, 128)])
def test_checked_dequant_weight_t(N, K, block):
    W = synth.normal_bf16(14, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    Wq, s = _i8(wq), _f32(sw)
    _both(lambda: cr.convrot_dequant_weight_t(Wq, s, block))


@pytest.mark.parametrize("M,N,K,block", [(300, 544, 384, 32), (37, 1024, 256, 256), (40, 32768, 256, 128)])
def test_checked_grad_x_bf16_and_second_reading(M, N, K, block):
    W = synth.normal_bf16(17, synth.STREAM_W, N, K, 0.02)
    wq, sw = oracle.quantize_weight(W, block)
    Wq, s = _i8(wq), _f32(sw)
    dY = torch_bf16(synth.normal_bf16(17, synth.STREAM_DY, M, N, 1e-3))
    _both(lambda: cr.convrot_linear_bwd_x_bf16(dY, Wq, s, block))
    _both(lambda: cr.convrot_linear_bwd_x_r2(dY, Wq, s, block))


@pytest.mark.parametrize("V,D,block,n", [(1000, 512, 128, 300), (97, 48, 16, 130), (64, 4096, 128, 33),
                                         (64, 32768, 128, 40)])
def test_checked_embedding_lookup(V, D, block, n):
    table = synth.normal_bf16(10, synth.STREAM_TABLE, V, D, 0.02)
    eq, se = oracle.quantize_rows_bf16(table, block)
    ids = torch.from_numpy(synth.token_ids(10, n, V)).cuda()
    Eq, s = _i8(eq), _f32(se)
    _both(lambda: cr.convrot_embedding_lookup(ids, Eq, s, block))


@pytest.mark.parametrize("M,N,K", [(129, 272, 1040), (17, 48, 4096), (1, 16, 16)])
def test_checked_gemm_s32_and_widen(M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = _i8(rng.integers(-127, 128, size=(M, K), dtype=np.int8))
    B = _i8(rng.integers(-127, 128, size=(N, K), dtype=np.int8))
    _both(lambda: cr.convrot_gemm_s32(A, B))
    _both(lambda: cr.convrot_widen_codes(A))


def test_checked_library_reports_no_stale_flag_after_release_calls():
    """Release calls never touch the checked library's flags: after a burst of
    release work the checked library still reads clean."""
    x = torch_bf16(synth.activations_bf16(3, 64, 1024, 2, 10.0))
    cr.convrot_quantize_activation(x, 128)
    prev = cr.select_library("checked")
    try:
        assert cr.convrot_get_error() == cr.OK
    finally:
        cr.select_library(prev)
    assert isinstance(cr.lib(), ctypes.CDLL)
