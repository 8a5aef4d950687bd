"""GPU parity: coalesce_mlp_fused (through the C ABI) against the fp64 oracle.

The oracle keeps every intermediate in fp64; the kernel rounds each
intermediate activation to fp16 on chip (the tensor cores take fp16
operands).  Tolerance, written here: |gpu - ref| <= 1e-2 + 2^-11 |ref| (the
1e-2 absolute bound of the fp16 workloads plus half an fp16 ulp of the
output).  The fp16-mirror oracle (intermediates rounded to fp16) is reported
when a case fails, as a diagnostic only.
"""
import math

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


def run(x, Ws, bs, act="softplus"):
    rows, D = x.shape
    H = Ws[0].shape[1]
    pad = 2048
    store = torch.full((pad + rows * H + pad,), float("nan"), dtype=torch.float16, device="cuda")
    out = store[pad:pad + rows * H].view(rows, H)
    xs = x.cuda()
    Wd = [w.cuda() for w in Ws]
    bd = None if bs is None else [None if b is None else b.cuda() for b in bs]
    st = g.coalesce_mlp_fused(rows, D, H, len(Ws), xs.data_ptr(), [w.data_ptr() for w in Wd],
                              None if bd is None else [None if b is None else b.data_ptr() for b in bd],
                              out.data_ptr(), g.ACT_CODES[act], torch.cuda.current_stream().cuda_stream)
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(torch.cuda.current_stream().cuda_stream) == 0
    assert torch.isnan(store[:pad].float()).all() and torch.isnan(store[pad + rows * H:].float()).all(), \
        "store outside out"
    return out


def check(gpu, ref, what, mirror=None):
    err = np.abs(gpu - ref)
    t = 1e-2 + 2.0 ** -11 * np.abs(ref)
    bad = err > t
    assert not np.isnan(gpu).any(), f"{what}: NaN"
    extra = ""
    if bad.any() and mirror is not None:
        extra = f"; vs fp16-mirror max err {np.abs(gpu - mirror).max():.3e}"
    assert not bad.any(), f"{what}: {bad.sum()}/{bad.size} over tol, max err {err.max():.3e}{extra}"
    return err.max()


def mk(rows, D, H, L, seed, b_var=0.01, w_var=None):
    w = inputs.MlpWorkload("t", rows, D, H, L, "f16", w_var if w_var is not None else 1.0 / H, b_var)
    return inputs.mlp_inputs(w, seed=seed)


@pytest.mark.parametrize("rows", [1, 127, 128, 129, 256, 1000, 4133])
@pytest.mark.parametrize("D,H,L", [(128, 128, 3), (64, 64, 5), (64, 128, 2), (128, 64, 4), (64, 64, 1),
                                   (256, 64, 2), (64, 192, 2), (64, 64, 8)])
def test_mlp_random_parity(rows, D, H, L):
    x, Ws, bs = mk(rows, D, H, L, seed=rows + 7 * L)
    out = run(x, Ws, bs)
    xs, Wn, bn = f64(x), [f64(w) for w in Ws], [f64(b) for b in bs]
    ref = oracle.mlp_chain(xs, Wn, bn, "softplus")
    check(f64(out), ref, f"mlp rows={rows} D={D} H={H} L={L}", oracle.mlp_chain_fp16_mirror(xs, Wn, bn))


@pytest.mark.parametrize("act", ["none", "relu", "gelu_erf"])
def test_mlp_other_activations(act):
    x, Ws, bs = mk(777, 128, 128, 3, seed=11)
    out = run(x, Ws, bs, act)
    ref = oracle.mlp_chain(f64(x), [f64(w) for w in Ws], [f64(b) for b in bs], act)
    check(f64(out), ref, f"act={act}")


def test_mlp_bias_null():
    x, Ws, _ = mk(300, 64, 64, 5, seed=3)
    out = run(x, Ws, None)
    ref = oracle.mlp_chain(f64(x), [f64(w) for w in Ws], None)
    check(f64(out), ref, "bias=NULL")


@pytest.mark.parametrize("L", [1, 3, 5])
def test_mlp_identity_weights_closed_form(L):
    """Identity W, zero b, x = ln k: out = ln(k + L - 1) (softplus(ln k) = ln(k + 1))."""
    D = H = 64
    rows = 200
    ks = torch.arange(1, D + 1, dtype=torch.float64) / 8.0
    x = torch.log(ks)[None, :].repeat(rows, 1).to(torch.float16)
    Ws = [torch.eye(D, dtype=torch.float16) for _ in range(L)]
    out = run(x, Ws, [None] * L)
    kx = np.exp(f64(x))  # the k that the fp16-rounded x encodes
    check(f64(out), np.log(kx + L - 1), f"identity L={L}")


def test_mlp_one_layer_matches_gemm_path():
    """L = 1 is a GEMM + bias with no activation: equal to coalesce_gemm_bias_act(act=none)."""
    x, Ws, bs = mk(1000, 128, 128, 1, seed=5)
    out = run(x, Ws, bs)
    Y = g.gemm_bias_act(x.cuda(), Ws[0].cuda(), bs[0].cuda(), "none")
    g.device_status()
    assert np.abs(f64(out) - f64(Y)).max() <= 2.0 ** -10 * max(1.0, np.abs(f64(Y)).max())


def test_mlp_repeated_calls_identical():
    x, Ws, bs = mk(5000, 64, 64, 5, seed=9)
    a = run(x, Ws, bs).clone()
    b = run(x, Ws, bs)
    assert torch.equal(a, b)


def test_softplus_epilogue_error_bound():
    """L = 2 with identity weights and zero biases: out = softplus(x) for each
    element, so the on-chip packed-fp16 softplus is checked directly against the
    fp64 definition over [-12, 12]: |err| <= 2e-3 + 2^-10 |ref| (one fp16 ulp of
    the value plus the polynomial's and ex2's share)."""
    D = 64
    rows = 1024
    x = torch.linspace(-12, 12, rows * D, dtype=torch.float64).reshape(rows, D).to(torch.float16)
    Ws = [torch.eye(D, dtype=torch.float16) for _ in range(2)]
    out = run(x, Ws, [None, None])
    ref = oracle.act_softplus(f64(x))
    err = np.abs(f64(out) - ref)
    assert (err <= 2e-3 + 2.0 ** -10 * np.abs(ref)).all(), f"max err {err.max():.3e}"


def test_softplus_log2_chain_error_bound():
    """L = 4 with identity weights and zero biases: out = softplus(softplus(
    softplus(x))), the fp16 chain that carries its activations in log2 units
    (four or more layers).  Per layer the packed softplus is within
    2e-3 + 2^-10 |h_l| of the exact value of its (rounded) argument and is
    1-Lipschitz, so the errors add.  The first layer's weights carry the
    factor log2 e, rounded to fp16 (relative error at most 2^-11), and its
    result is rounded to fp16 (2^-11): 2^-10 |x| in all; the last layer's
    weights carry ln 2 the same way, and its result is rounded once more:
    2^-10 |out|."""
    D = 64
    rows = 1024
    L = 4
    x = torch.linspace(-12, 12, rows * D, dtype=torch.float64).reshape(rows, D).to(torch.float16)
    Ws = [torch.eye(D, dtype=torch.float16) for _ in range(L)]
    out = run(x, Ws, [None] * L)
    xs = f64(x)
    h = xs
    tol = 2.0 ** -10 * np.abs(xs)
    for _ in range(L - 1):
        h = oracle.act_softplus(h)
        tol = tol + 2e-3 + 2.0 ** -10 * np.abs(h)
    tol = tol + 2.0 ** -10 * np.abs(h)
    err = np.abs(f64(out) - h)
    assert (err <= tol).all(), f"max err {err.max():.3e}, max err/tol {np.max(err / tol):.2f}"
