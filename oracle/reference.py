"""Plain, slow, obviously-correct fp64 oracle (numpy / scipy on the CPU).

TEST INFRASTRUCTURE ONLY.  This module is the reference that the CUDA library is
checked against.  It is imported only by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the product path never touches it,
and it imports nothing from the product package.

What it computes, and the passages it follows
---------------------------------------------
* GEMM + bias + activation -- the "Coalesce" README, section "Fusion study
  (03_matmul_fused)": the fused kernel computes the same thing as "the same
  matmul followed by a separate elementwise kernel".  The oracle is that
  UNFUSED sequence, written out in three passes, all in fp64, from the
  dtype-rounded inputs widened exactly to fp64:

      pass 1  acc[i, j] = sum_k A[i, k] * B[k, j]       (library matmul)
      pass 2  z[i, j]   = acc[i, j] + bias[j]           (bias broadcast over rows)
      pass 3  y[i, j]   = act(z[i, j])

  Layouts are row-major A[M, K], B[K, N], bias[N], Y[M, N].
* GELU in the exact erf form -- the "Coalesce" README, "Notes for future
  sessions" (use erf, not the tanh approximation; PyTorch's default is the erf
  form): GELU(z) = z * Phi(z) = 0.5 * z * (1 + erf(z / sqrt(2))).
* Softplus -- the "MLP Megakernel" README, "Architecture" and "Ablation Study >
  Key findings": softplus(z) = log(1 + exp(z)) with beta = 1.  The oracle uses
  the exact identity log(1 + e^z) = max(z, 0) + log1p(exp(-|z|)), which is the
  same function evaluated without overflow.  (The page's "branchless" form
  x + log(1 + exp(-|x|)) is not softplus for x < 0; the page's threshold form
  where(x > 20, x, log(exp(x) + 1)) differs from the exact value by at most
  log1p(e^-20) ~ 2.1e-9.  Neither is used here: the oracle is the definition.)
* ReLU -- the "Coalesce" README, "MLIR pipeline (Phase 3)": max(z, 0).
* Chained MLP -- the "MLP Megakernel" README, "Architecture":
      out = softplus(softplus(x @ W1) @ W2) @ W3        (3 layers)
  and the 5-layer form, with a bias b_l added after every matmul (the
  workloads add biases; the page's formulas have none, and b_l = 0 recovers
  them).  W_l is stored [in, out] ("x @ W" form).  Intermediates are kept in
  fp64 (the plain definition); ``mlp_chain_fp16_mirror`` rounds each
  intermediate to fp16 as a diagnostic only, never for pass/fail.

* Training side of the chained MLP -- the "MLP Megakernel" README: "Full
  training" (forward + backward) and "Key ideas" (the backward differentiates
  softplus with its derivative sigmoid).  ``mlp_forward_train`` returns out and
  every intermediate activation; ``mlp_backward`` is the chain rule for the
  loss gradient dout = dLoss/dout, layer by layer from the last:

      g_{L}   = dout
      dW_l    = h_{l-1}^T g_l,   db_l = sum over rows of g_l
      g_{l-1} = (g_l W_l^T) * act'(z_{l-1})   (act' from the pre-activation:
                softplus' = sigmoid, ReLU' = [z > 0], identity' = 1)
      dx      = g_1 W_1^T

  all in fp64.

Parity pins (see tests/test_oracle.py): hand-worked 2x2/4x4 cases,
brute-force integer GEMMs, closed forms and textbook values of Phi, an
arbitrary-precision (mpmath) evaluation of erf and log(1 + e^z), the
fused-loop == unfused invariant, MLP special cases (identity weights,
L = 1 == GEMM), and the backward against central finite differences of
mlp_chain.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

ACTS = ("none", "relu", "gelu_erf", "softplus")

_INV_SQRT2 = 1.0 / math.sqrt(2.0)


def _f64(a) -> np.ndarray:
    """Exact widening of an fp16/bf16/fp32/fp64 array (or nested list) to fp64."""
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Activations (pass 3).  Elementwise on fp64 arrays.
# --------------------------------------------------------------------------
def act_none(z):
    """Identity: the epilogue adds the bias and applies nothing else."""
    return _f64(z)


def act_relu(z):
    """ReLU, max(z, 0) ("Coalesce" README, MLIR pipeline: matmul -> relu)."""
    return np.maximum(_f64(z), 0.0)


def act_gelu_erf(z):
    """GELU, exact erf form: 0.5 * z * (1 + erf(z / sqrt(2)))."""
    z = _f64(z)
    return 0.5 * z * (1.0 + _erf(z * _INV_SQRT2))


def act_softplus(z):
    """Softplus log(1 + e^z) (beta = 1), as max(z, 0) + log1p(exp(-|z|))."""
    z = _f64(z)
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


_ACT_FN = {
    "none": act_none,
    "relu": act_relu,
    "gelu_erf": act_gelu_erf,
    "softplus": act_softplus,
}


def apply_act(z, act: str):
    """Apply the named activation (one of ``ACTS``)."""
    try:
        fn = _ACT_FN[act]
    except KeyError:
        raise ValueError(f"unknown activation {act!r}; expected one of {ACTS}") from None
    return fn(z)


# --------------------------------------------------------------------------
# GEMM + bias + activation, unfused, in fp64.
# --------------------------------------------------------------------------
def _bias_vec(bias, n: int) -> np.ndarray:
    if bias is None:
        return np.zeros(n, dtype=np.float64)
    b = _f64(bias).reshape(-1)
    if b.shape[0] != n:
        raise ValueError(f"bias has {b.shape[0]} entries, expected N = {n}")
    return b


def gemm_bias_act(A, B, bias, act: str):
    """Y = act(A @ B + bias), three separate fp64 passes.

    A[M, K], B[K, N] row-major; bias[N] broadcast over rows, or None for zero.
    Returns an fp64 array Y[M, N].
    """
    A = _f64(A)
    B = _f64(B)
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch: A{A.shape} @ B{B.shape}")
    acc = A @ B                                   # pass 1: matmul
    z = acc + _bias_vec(bias, B.shape[1])[None, :]  # pass 2: bias
    return apply_act(z, act)                      # pass 3: activation


def gemm_bias_act_rows(A, B, bias, act: str, rows):
    """The rows ``rows`` of gemm_bias_act(A, B, bias, act), one by one.

    Each output row i depends only on A[i, :], B and bias, so a sample of rows
    of a full-size problem is computed exactly as the full problem would be.
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    return gemm_bias_act(_f64(A)[rows, :], B, bias, act)


def gemm_bias_act_fused_loops(A, B, bias, act: str):
    """Y = act(A @ B + bias) with explicit loops, k ascending, one element at a time.

    This is the "fused" order (accumulate, add bias, activate, store, per
    element).  Pure Python: tiny inputs only.  It exists for the invariant
    fused == unfused.
    """
    A = _f64(A)
    B = _f64(B)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("shape mismatch")
    b = _bias_vec(bias, N)
    fn = _ACT_FN[act]
    Y = np.empty((M, N), dtype=np.float64)
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                s += float(A[i, k]) * float(B[k, j])
            Y[i, j] = float(fn(np.float64(s + b[j])))
    return Y


# --------------------------------------------------------------------------
# Chained MLP.
# --------------------------------------------------------------------------
def _check_mlp(x, Ws, bs):
    L = len(Ws)
    if L < 1:
        raise ValueError("an MLP needs at least one layer")
    if bs is not None and len(bs) != L:
        raise ValueError("need one bias (or None) per layer")
    return L


def mlp_chain(x, Ws, bs, act: str = "softplus"):
    """out = h_{L-1} @ W_L + b_L with h_0 = x and h_l = act(h_{l-1} @ W_l + b_l).

    x[rows, D], W_1[D, H], W_l[H, H] (any [in, out] shapes that chain),
    b_l[out_l] or None (zero).  The last layer has a bias and no activation.
    All intermediates are fp64.
    """
    L = _check_mlp(x, Ws, bs)
    h = _f64(x)
    for l in range(L):
        W = _f64(Ws[l])
        b = None if bs is None else bs[l]
        z = h @ W + _bias_vec(b, W.shape[1])[None, :]
        h = z if l == L - 1 else apply_act(z, act)
    return h


def mlp_chain_rows(x, Ws, bs, rows, act: str = "softplus"):
    """Rows ``rows`` of mlp_chain (each output row depends on its input row only)."""
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    return mlp_chain(_f64(x)[rows, :], Ws, bs, act)


def mlp_chain_fp16_mirror(x, Ws, bs, act: str = "softplus"):
    """Diagnostic only: mlp_chain with every intermediate h_l rounded to fp16.

    Explains deviations of a kernel that keeps fp16 activations on chip.
    Never used to decide pass or fail.
    """
    L = _check_mlp(x, Ws, bs)
    h = _f64(x)
    for l in range(L):
        W = _f64(Ws[l])
        b = None if bs is None else bs[l]
        z = h @ W + _bias_vec(b, W.shape[1])[None, :]
        if l == L - 1:
            h = z
        else:
            h = apply_act(z, act).astype(np.float16).astype(np.float64)
    return h


# --------------------------------------------------------------------------
# Training side of the chained MLP.
# --------------------------------------------------------------------------
def act_derivative(z, act: str):
    """d act / dz at the pre-activation z: sigmoid for softplus, [z > 0] for
    ReLU, 1 for the identity (GELU is not trained by this library)."""
    z = np.asarray(z, dtype=np.float64)
    if act == "softplus":
        return 0.5 * (1.0 + np.tanh(0.5 * z))  # sigmoid(z), overflow-free
    if act == "relu":
        return (z > 0).astype(np.float64)
    if act == "none":
        return np.ones_like(z)
    raise ValueError(f"no derivative for {act!r}")


def act_derivative_from_output(h, act: str):
    """act'(z) written through the activation's output h = act(z), the form a
    backward pass evaluates when it keeps only the activations (the "MLP
    Megakernel" README, "Key ideas": the forward's activations are kept for the
    backward's derivative).  softplus: h = log(1 + e^z), so e^h = 1 + e^z and
    sigmoid(z) = e^z / (1 + e^z) = 1 - e^-h; ReLU: [z > 0] = [h > 0]; identity: 1."""
    h = np.asarray(h, dtype=np.float64)
    if act == "softplus":
        return -np.expm1(-h)
    if act == "relu":
        return (h > 0).astype(np.float64)
    if act == "none":
        return np.ones_like(h)
    raise ValueError(f"no derivative for {act!r}")


def mlp_forward_train(x, Ws, bs, act: str = "softplus"):
    """(out, [h_1 .. h_{L-1}], [z_1 .. z_L]) of mlp_chain, all fp64."""
    L = _check_mlp(x, Ws, bs)
    h = _f64(x)
    hs, zs = [], []
    for l in range(L):
        W = _f64(Ws[l])
        b = None if bs is None else bs[l]
        z = h @ W + _bias_vec(b, W.shape[1])[None, :]
        zs.append(z)
        if l == L - 1:
            return z, hs, zs
        h = apply_act(z, act)
        hs.append(h)


def mlp_backward(x, Ws, bs, dout, act: str = "softplus", derivs=None):
    """(dx, [dW_l], [db_l]) for the loss gradient dout = dLoss/dout, by the
    chain rule (see the module docstring), all fp64.

    ``derivs`` optionally supplies act'(z_l) for l = 1 .. L-1 instead of
    evaluating it here: ReLU's derivative [z > 0] is a decision, and a
    comparison with a kernel that decided it from its own (rounded) values
    must take the same decisions."""
    L = _check_mlp(x, Ws, bs)
    _, hs, zs = mlp_forward_train(x, Ws, bs, act)
    ins = [_f64(x)] + hs  # input of each layer
    g = _f64(dout)
    dWs, dbs = [None] * L, [None] * L
    dx = None
    for l in range(L - 1, -1, -1):
        W = _f64(Ws[l])
        dWs[l] = ins[l].T @ g
        dbs[l] = g.sum(axis=0)
        gin = g @ W.T
        if l > 0:
            d = act_derivative(zs[l - 1], act) if derivs is None else _f64(derivs[l - 1])
            g = gin * d
        else:
            dx = gin
    return dx, dWs, dbs


def mlp_backward_from_activations(x, Ws, hs, dout, act: str = "softplus"):
    """(dx, [dW_l], [db_l], [g_l]) given the stored activations hs = [h_1 ..
    h_{L-1}] (the inputs of layers 2 .. L) instead of recomputing them: the
    backward pass's own contract, whatever forward produced hs.  g_l =
    dLoss/dz_l for each layer (g_{L-1} = dout); each derivative comes from the
    stored activation (act_derivative_from_output).  All fp64."""
    L = len(Ws)
    if len(hs) != L - 1:
        raise ValueError("need L - 1 activations")
    ins = [_f64(x)] + [_f64(h) for h in hs]  # input of each layer
    g = _f64(dout)
    dWs, dbs, gs = [None] * L, [None] * L, [None] * L
    dx = None
    for l in range(L - 1, -1, -1):
        gs[l] = g
        W = _f64(Ws[l])
        dWs[l] = ins[l].T @ g
        dbs[l] = g.sum(axis=0)
        gin = g @ W.T
        if l > 0:
            g = gin * act_derivative_from_output(ins[l], act)
        else:
            dx = gin
    return dx, dWs, dbs, gs
