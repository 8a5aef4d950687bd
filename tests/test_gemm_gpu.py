"""GPU parity: coalesce_gemm_bias_act (through the C ABI) against the fp64 oracle.

Tolerances (written here, derived from the arithmetic):
* fp32:      |gpu - ref| <= 1e-4 * max(1, |ref|)
* fp16/bf16: |gpu - ref| <= 1e-2 + half an output ulp of ref (2^-8 |ref| for
  bf16, 2^-11 |ref| for fp16).  With O(1) outputs a correctly rounded result
  can be up to half an ulp away from the exact value, which for bf16 exceeds
  1e-2 once |ref| >= 2.56; the ulp term admits exactly that rounding.
* integer-valued inputs (the "Coalesce" README's (i*7)%13 and (i*3)%11
  patterns, unscaled): fp32 accumulation is exact, so the output must equal
  the exact result rounded once to the output dtype, bit for bit.
"""
import numpy as np
import pytest
import torch

import gemm_bias_activation_gb300 as g
import oracle
from gemm_bias_activation_gb300 import inputs

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def tol(ref, dtype):
    a = np.abs(ref)
    if dtype == "f32":
        return 1e-4 * np.maximum(1.0, a)
    ulp_half = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    return 1e-2 + ulp_half * a


def check(gpu, ref, dtype, what=""):
    err = np.abs(gpu - ref)
    t = tol(ref, dtype)
    bad = err > t
    assert not np.any(np.isnan(gpu)), f"{what}: NaN in output"
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} over tolerance; max err {err.max():.3e} "
                           f"at {np.unravel_index(np.argmax(err - t), err.shape)}")
    return err.max()


def run(A, B, bias, act, canary=True):
    """Call through the C ABI with Y inside a guard band filled with a sentinel."""
    dev = A.device
    M, K = A.shape
    N = B.shape[1]
    pad = 4096
    store = torch.full((pad + M * N + pad,), float("nan"), dtype=A.dtype, device=dev)
    Y = store[pad:pad + M * N].view(M, N)
    st = g.coalesce_gemm_bias_act(M, N, K, g._dtype_code(A), A.data_ptr(), B.data_ptr(),
                                  0 if bias is None else bias.data_ptr(), Y.data_ptr(), g.ACT_CODES[act],
                                  torch.cuda.current_stream().cuda_stream)
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(torch.cuda.current_stream().cuda_stream) == 0
    if canary:
        head, tail = store[:pad], store[pad + M * N:]
        assert torch.isnan(head.float()).all() and torch.isnan(tail.float()).all(), "store outside Y"
    return Y


# ---------------------------------------------------------------- bit-exact integer cases
INT_SHAPES = [(128, 256, 64), (1, 8, 8), (7, 24, 16), (129, 264, 72), (300, 520, 264), (257, 1000, 1000),
              (1000, 136, 8), (64, 2048, 192), (1544, 1608, 72), (1000, 600, 72), (900, 800, 40)]


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("M,N,K", INT_SHAPES)
@pytest.mark.parametrize("act", ["none", "relu"])
def test_integer_patterns_bit_exact(dtype, M, N, K, act):
    A = inputs.integer_pattern((M, K), 7, 13, dtype).cuda()
    B = inputs.integer_pattern((K, N), 3, 11, dtype).cuda()
    bias = (torch.arange(N) % 9 - 40).to(DT[dtype]).cuda()
    Y = run(A, B, bias, act)
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), act)
    want = torch.from_numpy(ref).to(DT[dtype])  # one RNE rounding of the exact result
    got = Y.cpu()
    assert torch.equal(got.view(torch.int16 if dtype != "f32" else torch.int32),
                       want.view(torch.int16 if dtype != "f32" else torch.int32)), \
        f"max diff {np.abs(f64(got) - f64(want)).max()}"


# Several waves of persistent tiles (>= 2 x 152 output tiles), with an even
# and an odd number of row blocks, a ragged N and a ragged K.
WAVE_SHAPES = [(5120, 4096, 256), (4900, 4096, 136), (4224, 4000, 200)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", WAVE_SHAPES)
def test_many_waves_bit_exact(dtype, M, N, K):
    A = inputs.integer_pattern((M, K), 7, 13, dtype).cuda()
    B = inputs.integer_pattern((K, N), 3, 11, dtype).cuda()
    bias = (torch.arange(N) % 9 - 40).to(DT[dtype]).cuda()
    Y = run(A, B, bias, "relu")
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), "relu")
    want = torch.from_numpy(ref).to(DT[dtype])
    got = Y.cpu()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
        f"max diff {np.abs(f64(got) - f64(want)).max()}"


# Shapes the CTA-pair kernel takes (at least one 256 x 256 tile per SM pair):
# several tiles per pair, a ragged K, K below one k step, a single pair row,
# and ragged M and N: last pair rows whose odd CTA has no rows at all (257,
# 9999) or only some (4900), last column tiles with 8 or 40 valid columns.
PAIR_SHAPES = [(5120, 4096, 256), (4096, 4864, 72), (2560, 8192, 1000), (19456, 1024, 8), (256, 19456, 136),
               (4900, 4000, 72), (257, 19496, 64), (9999, 2056, 40)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", PAIR_SHAPES)
def test_cta_pair_kernel_bit_exact(dtype, M, N, K):
    A = inputs.integer_pattern((M, K), 7, 13, dtype).cuda()
    B = inputs.integer_pattern((K, N), 3, 11, dtype).cuda()
    bias = (torch.arange(N) % 9 - 40).to(DT[dtype]).cuda()
    Y = run(A, B, bias, "none")
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), "none")
    want = torch.from_numpy(ref).to(DT[dtype])
    got = Y.cpu()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
        f"max diff {np.abs(f64(got) - f64(want)).max()}"


@pytest.mark.parametrize("act", ["gelu_erf", "softplus", "relu"])
def test_cta_pair_kernel_random_sampled(act):
    w = inputs.GemmWorkload("t", 4096, 4864, 1000, "bf16", act, "ffn")
    A, B, bias = inputs.gemm_inputs(w, seed=13)
    Y = run(A.cuda(), B.cuda(), bias.cuda(), act)
    rows = _sample_rows(w.M, n=64, seed=3)
    ref = oracle.gemm_bias_act_rows(f64(A), f64(B), f64(bias), act, rows)
    check(f64(Y[rows]), ref, "bf16", f"pair kernel {act}")


def test_cta_pair_kernel_fp16_without_bias_sampled():
    w = inputs.GemmWorkload("t", 5120, 4096, 520, "f16", "gelu_erf", "ffn")
    A, B, _ = inputs.gemm_inputs(w, seed=21)
    Y = run(A.cuda(), B.cuda(), None, "gelu_erf")
    rows = _sample_rows(w.M, n=64, seed=4)
    ref = oracle.gemm_bias_act_rows(f64(A), f64(B), None, "gelu_erf", rows)
    check(f64(Y[rows]), ref, "f16", "pair kernel fp16 without bias")


def test_many_waves_random_gelu_sampled():
    w = inputs.GemmWorkload("t", 4900, 4000, 1000, "bf16", "gelu_erf", "ffn")
    A, B, bias = inputs.gemm_inputs(w, seed=9)
    Y = run(A.cuda(), B.cuda(), bias.cuda(), "gelu_erf")
    rows = _sample_rows(w.M, n=64, seed=2)
    ref = oracle.gemm_bias_act_rows(f64(A), f64(B), f64(bias), "gelu_erf", rows)
    check(f64(Y[rows]), ref, "bf16", "many-wave gelu")


# ---------------------------------------------------------------- random, all activations
SMALL_SHAPES = [(256, 256, 256), (300, 520, 264), (1, 8, 8), (130, 72, 40), (513, 264, 1032)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf", "softplus"])
@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
def test_half_random_parity(dtype, act, M, N, K):
    w = inputs.WORKLOADS["bf16_ffn_up_bias_gelu_16384x16384x4096"]
    w = inputs.GemmWorkload(w.name, M, N, K, dtype, act, "ffn")
    A, B, bias = inputs.gemm_inputs(w, seed=1)
    Y = run(A.cuda(), B.cuda(), bias.cuda(), act)
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), act)
    check(f64(Y), ref, dtype, f"{dtype} {act} {M}x{N}x{K}")


@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf", "softplus"])
# Shapes with fewer 128 x 128 tiles than a quarter of the SMs take the 64 x 64
# cluster split-K kernel; between a quarter and a half, the 128 x 128 kernel
# with K split over a CTA pair ((1024, 1024, 1024): 64 tiles; (1000, 600, 72):
# 40 tiles, five k slabs split three and two; (900, 800, 40): 56 tiles, three
# slabs, the last one ragged); (1300, 1200, 136) (110 tiles) and
# (2000, 2056, 264) take the 128 x 128 kernel whole.
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 264), (1, 4, 4), (130, 68, 36), (513, 260, 1028),
                                   (1300, 1200, 136), (2000, 2056, 264), (64, 64, 4096), (1024, 1024, 1024),
                                   (1000, 600, 72), (900, 800, 40)])
def test_f32_random_parity(act, M, N, K):
    w = inputs.WORKLOADS["fp32_gemm_bias_gelu_256"]
    A, B, bias = inputs.gemm_inputs(w, seed=2, M=M, N=N, K=K)
    Y = run(A.cuda(), B.cuda(), bias.cuda(), act)
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), act)
    check(f64(Y), ref, "f32", f"f32 {act} {M}x{N}x{K}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_bias_null_means_zero(dtype):
    w = inputs.GemmWorkload("t", 200, 264, 136, dtype, "gelu_erf", "uniform" if dtype == "f32" else "ffn")
    A, B, _ = inputs.gemm_inputs(w, seed=3)
    Y = run(A.cuda(), B.cuda(), None, "gelu_erf")
    ref = oracle.gemm_bias_act(f64(A), f64(B), None, "gelu_erf")
    check(f64(Y), ref, dtype, "bias=NULL")


def test_ones_times_inverse_n_closed_form():
    """A = 1, B = 1/N: the accumulator is exactly 1 and Y[:, j] = GELU(1 + bias[j])
    (the "Coalesce" README's fused-kernel test data)."""
    N = 256
    for dtype in ["bf16", "f16", "f32"]:
        A = torch.ones(192, N, dtype=DT[dtype]).cuda()
        B = torch.full((N, N), 1.0 / N, dtype=DT[dtype]).cuda()
        bias = (torch.linspace(-4, 2, N)).to(DT[dtype]).cuda()
        Y = run(A, B, bias, "gelu_erf")
        ref = oracle.act_gelu_erf(1.0 + f64(bias))[None, :].repeat(192, axis=0)
        check(f64(Y), ref, dtype, f"ones/N {dtype}")


def _sample_rows(M, n=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, M, size=n).tolist()) | {0, 1, 127, 128, M // 2, M - 129, M - 1}
    return sorted(rows)


# ---------------------------------------------------------------- square FP32 sweep, smaller sizes
# (the full-size workloads, 2048 and 4096 among them, are compared element by
# element in test_full_size_gpu.py)
@pytest.mark.parametrize("n", [512, 1024])
def test_f32_sweep_sizes(n):
    w = inputs.WORKLOADS[f"fp32_gemm_bias_gelu_{n}"]
    A, B, bias = inputs.gemm_inputs(w, seed=0)
    Y = g.gemm_bias_act(A.cuda(), B.cuda(), bias.cuda(), "gelu_erf")
    g.device_status()
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias), "gelu_erf")
    check(f64(Y), ref, "f32", f"f32 {n}")


def test_repeated_calls_identical():
    """Deterministic: the same inputs give the same bits on a second call."""
    w = inputs.GemmWorkload("t", 1000, 1032, 520, "bf16", "gelu_erf", "ffn")
    A, B, bias = (t.cuda() for t in inputs.gemm_inputs(w, seed=4))
    Y1 = run(A, B, bias, "gelu_erf").clone()
    Y2 = run(A, B, bias, "gelu_erf")
    assert torch.equal(Y1, Y2)
