"""The allocation-free forward (`convrot_linear_fwd_noalloc`) against the
regular forward (`convrot_linear_fwd`).

The no-allocation entry point serves callers that cannot allocate device
memory where they run the layer (a host framework that only lends pointers,
a loop where a synchronising cudaMalloc is not allowed, a fixed memory
budget).  It keeps the activation codes in one library-owned device array, so
this file checks, through the C ABI, that two calls in a row with different
shapes both match the regular entry point, and that a problem larger than the
array is refused.  It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import REL_FRO_ORACLE, bits_of, f64, rel_fro, torch_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    cr.lib()


def _call_noalloc(x, Wq, sw, block, y, bias=None):
    L = cr.lib()
    M, K = x.shape
    N = Wq.shape[0]
    rc = L.convrot_linear_fwd_noalloc(ctypes.c_void_p(x.data_ptr()), M, K, ctypes.c_void_p(Wq.data_ptr()),
                                      ctypes.c_void_p(sw.data_ptr()), N, block,
                                      None if bias is None else ctypes.c_void_p(bias.data_ptr()),
                                      ctypes.c_void_p(y.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def test_noalloc_matches_regular_forward_on_two_calls():
    K, N, b = 1024, 528, 128
    W = synth.normal_bf16(21, synth.STREAM_W, N, K, 0.02)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    bias = torch_bf16(synth.normal_bf16(21, 9, 1, N, 0.1)[0])
    # first call: more rows; second call: fewer rows and other values, so stale
    # scratch contents from the first call would show up in the second
    for M, seed, use_bias in [(700, 22, False), (259, 23, True)]:
        x = torch_bf16(synth.activations_bf16(seed, M, K, 10, 30.0))
        bb = bias if use_bias else None
        ref = cr.convrot_linear_fwd(x, Wq, sw, b, bias=bb)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(x, Wq, sw, b, y, bb) == cr.OK
        torch.cuda.synchronize()
        assert cr.convrot_get_error() == cr.OK
        assert rel_fro(f64(bits_of(y)), f64(bits_of(ref))) <= REL_FRO_ORACLE
        assert torch.equal(y, ref)  # same kernels, same inputs: identical results


def _need(M, K):
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    return r(M * K * 2) + r(M * 4)


def test_noalloc_accepts_the_largest_problem_and_refuses_the_next():
    """The limit follows from convrot_linear_fwd_noalloc_max_bytes(): the largest M that
    fits at K = 4096 runs (and equals the regular forward), one row more is refused."""
    limit = cr.convrot_linear_fwd_noalloc_max_bytes()
    K, N, b = 4096, 16, 128
    M = limit // (2 * K)
    while _need(M + 1, K) <= limit:
        M += 1
    while _need(M, K) > limit:
        M -= 1
    assert M >= 8192  # 8192 tokens at K = 4096 fit, scales included
    x = torch_bf16(synth.activations_bf16(24, M + 1, K, 10, 30.0))
    W = synth.normal_bf16(24, synth.STREAM_W, N, K, 0.02)
    Wq, sw = cr.convrot_quantize_weight(torch_bf16(W), b)
    y = torch.empty((M + 1, N), dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(x[:M], Wq, sw, b, y[:M]) == cr.OK
    torch.cuda.synchronize()
    assert cr.convrot_get_error() == cr.OK
    assert torch.equal(y[:M], cr.convrot_linear_fwd(x[:M], Wq, sw, b))
    assert _call_noalloc(x, Wq, sw, b, y) == cr.ERR_UNSUPPORTED
    assert cr.convrot_get_error() == cr.OK
