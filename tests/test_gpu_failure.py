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
