"""Seeded random shapes through every compute entry point, against the fp64
oracle: GEMMs of every dtype and activation at sizes from one element to a
few hundred rows and columns (ragged in every dimension), chained MLPs of
random depth and widths (multiples of 8 up to 256, fp16 and bf16, with and
without biases), and training steps.  The shapes are drawn once from a fixed
seed, so every run checks the same cases.

Tolerances as in the dedicated tests:
* GEMM fp32: 1e-4 max(1, |ref|); fp16/bf16: 1e-2 + half an output ulp.
* MLP: 1e-2 + half an output ulp (2^-11 |ref| fp16, 2^-8 |ref| bf16) plus
  the first-order bound of what rounding every intermediate to the operand
  type (unit roundoff u) propagates to the output, as in test_mlp_ex_gpu:
  e_0 = 0; per layer e_{l-1} |W_l| plus fp32 summation (K 2^-24 (|h| |W| +
  |b|)), times the activation's Lipschitz constant, plus u |h_l|; at these
  widths and depths an fp16 chain stays far inside 1e-2 without it, but deep
  linear chains of 256-wide layers need not.
* Training: test_train_gpu.check_grads against the oracle's backward given
  the kernel's own stored activations.
"""
import numpy as np
import pytest
import torch

import gemm_bias_activation_gb300 as g
import oracle
from gemm_bias_activation_gb300 import inputs

from tests.test_train_gpu import backward, check_grads, forward_train
from tests.test_train_gpu import mk as mk_train

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ACTS = ["none", "relu", "gelu_erf", "softplus"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _gemm_cases(n=36):
    rng = np.random.default_rng(20261202)
    cases = []
    for i in range(n):
        dtype = ["f32", "f16", "bf16"][i % 3]
        step = 4 if dtype == "f32" else 8  # 16-byte rows
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 90)) * step
        K = int(rng.integers(1, 90)) * step
        act = ACTS[int(rng.integers(0, 4))]
        with_bias = bool(rng.integers(0, 4))  # one case in four without a bias
        cases.append((i, dtype, M, N, K, act, with_bias))
    return cases


@pytest.mark.parametrize("i,dtype,M,N,K,act,with_bias", _gemm_cases())
def test_random_gemm(i, dtype, M, N, K, act, with_bias):
    w = inputs.GemmWorkload("t", M, N, K, dtype, act, "uniform" if dtype == "f32" else "ffn")
    A, B, bias = inputs.gemm_inputs(w, seed=100 + i)
    b = bias.cuda() if with_bias else None
    Y = g.gemm_bias_act(A.cuda(), B.cuda(), b, act)
    g.device_status()
    ref = oracle.gemm_bias_act(f64(A), f64(B), f64(bias) if with_bias else None, act)
    err = np.abs(f64(Y) - ref)
    if dtype == "f32":
        t = 1e-4 * np.maximum(1.0, np.abs(ref))
    else:
        t = 1e-2 + (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) * np.abs(ref)
    assert not np.isnan(f64(Y)).any()
    assert (err <= t).all(), f"max err {err.max():.3e}, max err/tol {np.max(err / t):.2f}"


LIPSCHITZ = {"softplus": 1.0, "relu": 1.0, "none": 1.0}


def rounding_bound(x, Ws, bs, act, u):
    """First-order bound on |chain with intermediates rounded (unit roundoff
    u) - exact chain|; b entries may be None (zero)."""
    c = LIPSCHITZ[act]
    h = f64(x)
    e = np.zeros_like(h)
    for l, W in enumerate(Ws):
        W = f64(W)
        b = np.zeros(W.shape[1]) if bs is None or bs[l] is None else f64(bs[l])
        aW = np.abs(W)
        z = h @ W + b[None, :]
        ez = e @ aW + W.shape[0] * 2.0 ** -24 * (np.abs(h) @ aW + np.abs(b)[None, :])
        if l == len(Ws) - 1:
            return ez
        h = oracle.apply_act(z, act)
        e = c * ez + u * np.abs(h)


def _mlp_cases(n=24):
    rng = np.random.default_rng(4242)
    cases = []
    for i in range(n):
        dtype = "f16" if i % 3 else "bf16"
        L = int(rng.integers(1, 9))
        D, H, O = (int(rng.integers(1, 33)) * 8 for _ in range(3))
        rows = int(rng.integers(1, 3000))
        act = ["softplus", "relu", "none"][int(rng.integers(0, 3))] if dtype == "f16" else "softplus"
        with_bias = bool(rng.integers(0, 4))
        cases.append((i, dtype, rows, D, H, O, L, act, with_bias))
    return cases


@pytest.mark.parametrize("i,dtype,rows,D,H,O,L,act,with_bias", _mlp_cases())
def test_random_mlp(i, dtype, rows, D, H, O, L, act, with_bias):
    if L == 1:
        H = O  # a one-layer chain has no hidden width
    w = inputs.MlpWorkload("t", rows, D, H, L, dtype, 1.0 / max(D, H), 0.01 if with_bias else None, act, O)
    x, Ws, bs = inputs.mlp_inputs(w, seed=200 + i)
    out = g.mlp_fused(x.cuda(), [t.cuda() for t in Ws], [t.cuda() for t in bs] if with_bias else None, act)
    g.device_status()
    ref = oracle.mlp_chain(f64(x), [f64(t) for t in Ws], [f64(t) for t in bs], act)
    err = np.abs(f64(out) - ref)
    u = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    t = 1e-2 + u * np.abs(ref) + rounding_bound(x, Ws, bs if with_bias else None, act, u)
    assert not np.isnan(f64(out)).any()
    assert (err <= t).all(), f"max err {err.max():.3e}, max err/tol {np.max(err / t):.2f}"


def _train_cases(n=10):
    rng = np.random.default_rng(777)
    cases = []
    for i in range(n):
        dtype = "f16" if i % 2 else "bf16"
        L = int(rng.integers(1, 6))
        D, H, O = (int(rng.integers(1, 33)) * 8 for _ in range(3))
        rows = int(rng.integers(1, 2500))
        act = ["softplus", "relu"][int(rng.integers(0, 2))]
        cases.append((i, dtype, rows, D, H, O, L, act))
    return cases


@pytest.mark.parametrize("i,dtype,rows,D,H,O,L,act", _train_cases())
def test_random_training_step(i, dtype, rows, D, H, O, L, act):
    if L == 1:
        H = O
    x, Ws, bs, dout = mk_train(rows, D, H, O, L, dtype, seed=300 + i)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, act, dtype)
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, act, dtype)
    check_grads(x, Ws, dout, act, dtype, dx, dW, db, h_copy)
