"""Failure detection on the GPU without a GPU fault.

Every wait in the library's kernels is bounded; when one runs out the kernel
records it in a device error word and returns, and coalesce_device_status
reports COALESCE_ERR_DEVICE_TIMEOUT.  The self-test kernel waits on a barrier
that nothing arrives on (a flag that nothing sets) with a short limit; no
trap, bad address or endless loop is involved, and the context must stay
usable afterwards.
"""
import time

import pytest
import torch

import gemm_bias_activation_gb300 as g

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def test_bounded_wait_reports_timeout_and_context_survives():
    s = torch.cuda.current_stream().cuda_stream
    assert g.coalesce_device_status(s) == g.COALESCE_OK  # nothing pending
    t0 = time.perf_counter()
    assert g.coalesce_selftest_wait_timeout(50_000_000, s) == g.COALESCE_OK  # 50 ms limit
    st = g.coalesce_device_status(s)
    dt = time.perf_counter() - t0
    assert st == g.COALESCE_ERR_DEVICE_TIMEOUT, g.coalesce_status_string(st)
    assert "bounded wait" in g.coalesce_last_error()
    assert 0.045 < dt < 5.0, dt                   # it waited for the limit, then returned
    assert g.coalesce_device_status(s) == g.COALESCE_OK  # the word was cleared
    # The context is still usable: a GEMM runs and is correct.
    A = torch.eye(64, dtype=torch.bfloat16, device="cuda")
    B = torch.arange(64 * 64, dtype=torch.float32, device="cuda").reshape(64, 64).div(4096).to(torch.bfloat16)
    Y = g.gemm_bias_act(A, B, None, "none")
    g.device_status()
    assert torch.equal(Y, B)


def test_selftest_rejects_bad_limits():
    s = torch.cuda.current_stream().cuda_stream
    assert g.coalesce_selftest_wait_timeout(10, s) == g.COALESCE_ERR_INVALID_ARG
    assert g.coalesce_selftest_wait_timeout(100_000_000_000, s) == g.COALESCE_ERR_INVALID_ARG
