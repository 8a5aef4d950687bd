"""Fused vs unfused on the GPU (the "Coalesce" README's fusion study).

Unfused = coalesce_gemm_bias_act(bias=NULL, act=NONE) then the separate
in-place coalesce_bias_act pass.  For fp32 the two orders perform the same
fp32 operations in the same order, so the outputs must be bit-identical
(the README reports max |fused - unfused| = 0); for fp16/bf16 the unfused
order rounds the accumulator to the storage type first, so both are checked
against the fp64 oracle within the usual tolerance.
"""
import numpy as np
import pytest
import torch

import gemm_bias_activation_gb300 as g
import oracle
from gemm_bias_activation_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf", "softplus"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1000, 1032, 520), (2000, 2056, 264)])
def test_f32_fused_equals_unfused_bitwise(act, M, N, K):
    w = inputs.WORKLOADS["fp32_gemm_bias_gelu_256"]
    A, B, bias = (t.cuda() for t in inputs.gemm_inputs(w, seed=5, M=M, N=N, K=K))
    fused = g.gemm_bias_act(A, B, bias, act)
    unfused = g.gemm_then_bias_act(A, B, bias, act)
    g.device_status()
    assert torch.equal(fused.view(torch.int32), unfused.view(torch.int32))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("act", ["gelu_erf", "softplus", "relu"])
def test_half_unfused_matches_oracle(dtype, act):
    w = inputs.GemmWorkload("t", 513, 264, 1032, dtype, act, "ffn")
    A, B, bias = inputs.gemm_inputs(w, seed=6)
    Y = g.gemm_then_bias_act(A.cuda(), B.cuda(), bias.cuda(), act)
    g.device_status()
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), act)
    half_ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    # one extra rounding of the accumulator: allow a second half ulp
    assert (np.abs(f64(Y) - ref) <= 1e-2 + 2 * half_ulp * np.abs(ref)).all()


def test_bias_act_in_place_ragged_and_null_bias():
    for dtype in [torch.float32, torch.float16, torch.bfloat16]:
        M, N = 37, 40
        Y0 = torch.randn(M, N, dtype=torch.float32).to(dtype)
        bias = torch.randn(N, dtype=torch.float32).to(dtype)
        for b in [bias, None]:
            Y = Y0.clone().cuda()
            st = g.coalesce_bias_act(M, N, g._dtype_code(Y), Y.data_ptr(), None if b is None else b.cuda().data_ptr(),
                                     g.COALESCE_ACT_GELU_ERF, torch.cuda.current_stream().cuda_stream)
            assert st == 0
            g.device_status()
            ref = oracle.act_gelu_erf(f64(Y0) + (0.0 if b is None else f64(b)[None, :]))
            tol = 1e-6 if dtype == torch.float32 else (2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11)
            assert (np.abs(f64(Y) - ref) <= tol * np.maximum(1.0, np.abs(ref)) + 1e-6).all()
