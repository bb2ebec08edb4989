"""Failure detection without a GPU fault: a pipeline wait that never completes
must end at its limit, be reported to the host as CONVROT_ERR_TIMEOUT, and
leave the CUDA context usable (the next GEMM is still bit-exact)."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import int8_rotated_quantized_gb300 as cr  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cr._build.build()
    cr.lib()


def test_bounded_wait_reports_timeout_and_context_survives():
    assert cr.convrot_get_error() == cr.OK
    st = cr._stream(None)
    assert cr.lib().convrot_selftest_wait_timeout(20_000_000, st) == cr.OK  # 20 ms
    assert cr.convrot_get_error() == cr.ERR_TIMEOUT
    assert cr.convrot_get_error() == cr.OK  # the word was cleared
    rng = np.random.default_rng(3)
    A = rng.integers(-127, 128, size=(130, 256), dtype=np.int8)
    B = rng.integers(-127, 128, size=(48, 256), dtype=np.int8)
    C = cr.convrot_gemm_s32(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda())
    np.testing.assert_array_equal(C.cpu().numpy(), oracle.gemm_s32(A, B))
    assert cr.convrot_get_error() == cr.OK


def test_selftest_rejects_bad_limits():
    st = cr._stream(None)
    assert cr.lib().convrot_selftest_wait_timeout(0, st) == cr.ERR_INVALID_ARG
    assert cr.lib().convrot_selftest_wait_timeout(20_000_000_000, st) == cr.ERR_INVALID_ARG


def _fault_inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    xq = torch.from_numpy(rng.integers(-127, 128, size=(M, K)).astype(np.float16)).cuda()
    Wq = torch.from_numpy(rng.integers(-127, 128, size=(N, K), dtype=np.int8)).cuda()
    sx = torch.from_numpy(rng.uniform(1e-3, 2e-3, size=M).astype(np.float32)).cuda()
    sw = torch.from_numpy(rng.uniform(1e-4, 2e-4, size=N).astype(np.float32)).cuda()
    return xq, sx, Wq, sw


def _gemm_fault(widened, xq, sx, W, sw, y, limit_ns, skip, producer):
    M, K = xq.shape
    N = W.shape[0]
    return cr.lib().convrot_selftest_gemm_fault(widened, cr._ptr(xq), cr._ptr(sx), M, K, cr._ptr(W), cr._ptr(sw), N,
                                                cr._ptr(y), limit_ns, skip, producer, cr._stream(None))


# (M, N, K, skip in tiles, stages): one tile per CTA with the copies of stage 5 missing, and
# several tiles per CTA (or CTA pair) with the copies missing in its third tile, after two tiles
# have gone through the epilogue. A stage holds one K block of 64 in the single-CTA kernel
# (widened = 0) and two in the pair kernel (widened = 1).
@pytest.mark.parametrize("M,N,K,skip", [(1024, 512, 2048, (0, 5)), (4096, 4096, 1024, (2, 3))])
@pytest.mark.parametrize("widened", [0, 1])
@pytest.mark.parametrize("producer", [0, 1])
def test_gemm_abort_path_ends_at_the_limit_and_frees_the_sm(M, N, K, skip, widened, producer):
    """A copy the GEMM waits for never arrives (a test-only switch skips it in the named
    producer): the consumer's wait gives up after 20 ms, every role of the CTA stops,
    in-flight copies and MMAs drain, the tensor memory is freed, the host reads
    CONVROT_ERR_TIMEOUT, and the next GEMM on the same SMs is bit-identical to the one
    before (the widened-weight mode is the one the training step runs; the other mode
    also exercises the converter warps)."""
    import time
    assert cr.convrot_get_error() == cr.OK
    xq, sx, Wq, sw = _fault_inputs(M, N, K, M + N + K)
    W = cr.convrot_widen_codes(Wq) if widened else Wq
    run = cr.convrot_gemm_dequant_w16 if widened else cr.convrot_gemm_dequant
    before = run(xq, sx, W, sw)
    assert cr.convrot_get_error() == cr.OK
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    # the switch is inert when the iteration is never reached
    assert _gemm_fault(widened, xq, sx, W, sw, y, 20_000_000, 1 << 30, producer) == cr.OK
    assert cr.convrot_get_error() == cr.OK
    assert torch.equal(y, before)
    stages_per_tile = (K // 64) // (2 if widened else 1)
    t0 = time.perf_counter()
    assert _gemm_fault(widened, xq, sx, W, sw, y, 20_000_000, skip[0] * stages_per_tile + skip[1], producer) == cr.OK
    assert cr.convrot_get_error() == cr.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 1.5  # ended by the 20 ms limit, not the default 2 s
    assert cr.convrot_get_error() == cr.OK
    after = run(xq, sx, W, sw)
    assert cr.convrot_get_error() == cr.OK
    assert torch.equal(after, before)


def test_gemm_fault_selftest_rejects_bad_arguments():
    xq, sx, Wq, sw = _fault_inputs(64, 32, 64, 1)
    y = torch.zeros((64, 32), dtype=torch.bfloat16, device="cuda")
    assert _gemm_fault(0, xq, sx, Wq, sw, y, 0, 3, 0) == cr.ERR_INVALID_ARG
    assert _gemm_fault(0, xq, sx, Wq, sw, y, 20_000_000, 3, 2) == cr.ERR_INVALID_ARG
    assert _gemm_fault(0, xq, sx, Wq, sw, y, 20_000_000, -1, 0) == cr.ERR_INVALID_ARG
    assert _gemm_fault(2, xq, sx, Wq, sw, y, 20_000_000, 3, 0) == cr.ERR_INVALID_ARG
