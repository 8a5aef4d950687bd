"""Pins for the fp64 oracle: it is checked against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a transposed
operand, a bias on the wrong axis, a dropped term, a wrong sign or scale in an
activation, an activation on the last MLP layer) fails at least one test;
``test_planted_mistakes_are_caught`` plants such slips and checks that.
"""
import math
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN, parse_matrix, read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- worked cases
@pytest.mark.parametrize("fixture", ["gemm_2x2_hand.txt", "gemm_2x2_relu_hand.txt"])
def test_hand_worked_2x2(fixture):
    g = read_golden(fixture)
    A = np.array(parse_matrix(g["A"]))
    B = np.array(parse_matrix(g["B"]))
    bias = np.array(parse_matrix(g["bias"])[0])
    Y = np.array(parse_matrix(g["Y"]))
    got = oracle.gemm_bias_act(A, B, bias, g["act"])
    assert np.array_equal(got, Y)
    assert np.array_equal(oracle.gemm_bias_act_fused_loops(A, B, bias, g["act"]), Y)


def _brute_int_gemm(A, B, bias, relu):
    M, K = len(A), len(A[0])
    N = len(B[0])
    out = [[0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = bias[j]
            for k in range(K):
                s += A[i][k] * B[k][j]
            out[i][j] = max(s, 0) if relu else s
    return out


@pytest.mark.parametrize("M,N,K", [(4, 4, 4), (5, 3, 7), (1, 9, 2), (13, 11, 17)])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_integer_pattern_brute_force(M, N, K, act):
    """The README's transposition-exposing patterns (i*7)%13, (i*3)%11, unscaled."""
    A = [[((i * K + k) * 7) % 13 for k in range(K)] for i in range(M)]
    B = [[((k * N + j) * 3) % 11 for j in range(N)] for k in range(K)]
    bias = [(j % 5) - 40 for j in range(N)]  # negative offsets so relu bites
    want = np.array(_brute_int_gemm(A, B, bias, act == "relu"), dtype=np.float64)
    got = oracle.gemm_bias_act(np.array(A), np.array(B), np.array(bias), act)
    assert np.array_equal(got, want)


def test_mlp_two_layer_hand():
    g = read_golden("mlp_2layer_hand.txt")
    consts = {"LN3M1": math.log(3.0) - 1.0}
    x = np.array(parse_matrix(g["x"]))
    W1 = np.array(parse_matrix(g["W1"]))
    W2 = np.array(parse_matrix(g["W2"]))
    b1 = np.array(parse_matrix(g["b1"], consts)[0])
    b2 = np.array(parse_matrix(g["b2"])[0])
    want = np.array(parse_matrix(g["out"]))
    got = oracle.mlp_chain(x, [W1, W2], [b1, b2], "softplus")
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


# ---------------------------------------------------------------- GELU
def test_gelu_normal_cdf_table():
    """GELU(x) = x * Phi(x) against a printed table of the normal CDF."""
    with open(os.path.join(GOLDEN, "normal_cdf_table.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    xs = np.array([float(r[0]) for r in rows])
    phi = np.array([float(r[1]) for r in rows])
    np.testing.assert_allclose(oracle.act_gelu_erf(xs), xs * phi, rtol=1e-14, atol=1e-16)


def test_gelu_closed_forms():
    assert oracle.act_gelu_erf(0.0) == 0.0
    assert oracle.act_gelu_erf(10.0) == 10.0
    assert abs(oracle.act_gelu_erf(-10.0)) < 1e-20
    x = np.linspace(-6, 6, 241)
    # Phi(x) + Phi(-x) = 1  =>  GELU(x) - GELU(-x) = x
    np.testing.assert_allclose(oracle.act_gelu_erf(x) - oracle.act_gelu_erf(-x), x, atol=1e-14)
    # GELU(x) -> x for x >> 0 and -> 0 for x << 0
    assert abs(oracle.act_gelu_erf(8.0) - 8.0) < 1e-13
    assert abs(oracle.act_gelu_erf(-8.0)) < 1e-13


def test_gelu_against_arbitrary_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for x in [-5.5, -2.25, -0.7, -1e-3, 1e-4, 0.3, 1.7, 4.2]:
        want = float(mpmath.mpf(x) * mpmath.ncdf(x))
        assert abs(float(oracle.act_gelu_erf(x)) - want) <= 1e-15 * max(1.0, abs(want))


# ---------------------------------------------------------------- softplus / relu
def test_softplus_closed_forms():
    assert float(oracle.act_softplus(0.0)) == pytest.approx(math.log(2.0), abs=1e-16)
    # softplus(ln k) = ln(1 + k)
    for k in [0.5, 1.0, 2.0, 3.0, 10.0, 1e6]:
        assert float(oracle.act_softplus(math.log(k))) == pytest.approx(math.log1p(k), rel=1e-15)
    x = np.linspace(-30, 30, 601)   # beyond |x| ~ 36 the excess is below one fp64 ulp
    sp = oracle.act_softplus(x)
    assert np.all(sp > np.maximum(x, 0.0))
    np.testing.assert_allclose(sp - oracle.act_softplus(-x), x, atol=1e-13)
    assert float(oracle.act_softplus(800.0)) == 800.0          # no overflow
    assert float(oracle.act_softplus(-800.0)) == 0.0           # underflows to 0, not NaN


def test_softplus_against_arbitrary_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for z in [-30.0, -5.0, -1.0, -1e-3, 0.0, 1e-3, 0.7, 5.0, 19.9, 20.1, 30.0]:
        want = float(mpmath.log(1 + mpmath.exp(z)))
        assert abs(float(oracle.act_softplus(z)) - want) <= 2e-16 * max(1.0, abs(want))


def test_relu_and_none():
    x = np.array([-2.0, -0.0, 0.0, 3.5])
    assert np.array_equal(oracle.act_relu(x), np.array([0.0, 0.0, 0.0, 3.5]))
    assert np.array_equal(oracle.act_none(x), x)


def test_apply_act_rejects_unknown():
    with pytest.raises(ValueError):
        oracle.apply_act(np.zeros(2), "gelu_tanh")


# ---------------------------------------------------------------- P1 pattern
def test_ones_times_inverse_n_gives_unit_accumulator():
    """A = 1, B = 1/N (N a power of two): the accumulator is exactly 1 and
    Y[:, j] = GELU(1 + bias[j]) ("Coalesce" README, Notes: B = 1/N so GELU
    sees values where the curve bends).  Checked against the Phi table."""
    N = 8
    A = np.ones((3, N))
    B = np.full((N, N), 1.0 / N)
    bias = np.array([-1.0, -0.5, 0.0, 0.5, 1.0, 2.0, -2.0, -3.0])
    z = 1.0 + bias
    phi = {0.0: 0.5, 0.5: 0.69146246127401310364, 1.0: 0.84134474606854294859,
           1.5: 0.933192798731141934, 2.0: 0.9772498680518207928, 3.0: 0.99865010196836990547,
           -1.0: 0.15865525393145705141, -2.0: 0.0227501319481792072}
    want = np.array([v * phi[v] for v in z])
    got = oracle.gemm_bias_act(A, B, bias, "gelu_erf")
    for row in got:
        np.testing.assert_allclose(row, want, rtol=1e-14, atol=1e-16)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("act", list(oracle.ACTS))
def test_fused_equals_unfused_integer_exact(act):
    rng = np.random.default_rng(5)
    A = rng.integers(-4, 5, size=(6, 9)).astype(np.float64)
    B = rng.integers(-4, 5, size=(9, 7)).astype(np.float64)
    bias = rng.integers(-3, 4, size=7).astype(np.float64)
    fused = oracle.gemm_bias_act_fused_loops(A, B, bias, act)
    unfused = oracle.gemm_bias_act(A, B, bias, act)
    assert np.array_equal(fused, unfused)


@pytest.mark.parametrize("act", list(oracle.ACTS))
def test_fused_equals_unfused_random(act):
    rng = np.random.default_rng(7)
    A = rng.uniform(-1, 1, size=(5, 33)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(33, 6)).astype(np.float32)
    bias = rng.uniform(-1, 1, size=6).astype(np.float32)
    fused = oracle.gemm_bias_act_fused_loops(A, B, bias, act)
    unfused = oracle.gemm_bias_act(A, B, bias, act)
    np.testing.assert_allclose(fused, unfused, rtol=1e-13, atol=1e-13)


def test_bias_none_is_zero_bias():
    rng = np.random.default_rng(1)
    A, B = rng.normal(size=(4, 5)), rng.normal(size=(5, 3))
    assert np.array_equal(oracle.gemm_bias_act(A, B, None, "relu"),
                          oracle.gemm_bias_act(A, B, np.zeros(3), "relu"))


def test_rows_sample_matches_full():
    rng = np.random.default_rng(2)
    A, B, bias = rng.normal(size=(50, 40)), rng.normal(size=(40, 30)), rng.normal(size=30)
    rows = [0, 7, 49, 13]
    full = oracle.gemm_bias_act(A, B, bias, "gelu_erf")
    np.testing.assert_allclose(oracle.gemm_bias_act_rows(A, B, bias, "gelu_erf", rows), full[rows],
                               rtol=1e-13, atol=1e-13)


def test_shape_checks():
    with pytest.raises(ValueError):
        oracle.gemm_bias_act(np.zeros((2, 3)), np.zeros((4, 2)), None, "none")
    with pytest.raises(ValueError):
        oracle.gemm_bias_act(np.zeros((2, 3)), np.zeros((3, 2)), np.zeros(3), "none")


# ---------------------------------------------------------------- MLP
@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_mlp_identity_weights_closed_form(L):
    """Identity W, zero b: out = softplus^(L-1)(x); with x = ln k, softplus(ln k)
    = ln(k + 1), so out = ln(k + L - 1) exactly (no activation on the last layer)."""
    ks = np.array([1.0, 2.0, 3.0, 7.0, 0.25])
    x = np.log(ks)[None, :].repeat(3, axis=0)
    D = ks.size
    Ws = [np.eye(D) for _ in range(L)]
    out = oracle.mlp_chain(x, Ws, [None] * L, "softplus")
    np.testing.assert_allclose(out, np.log(ks + L - 1)[None, :].repeat(3, axis=0), rtol=1e-14)


def test_mlp_one_layer_is_gemm_bias_none():
    rng = np.random.default_rng(3)
    x, W, b = rng.normal(size=(9, 8)), rng.normal(size=(8, 8)), rng.normal(size=8)
    np.testing.assert_allclose(oracle.mlp_chain(x, [W], [b]), oracle.gemm_bias_act(x, W, b, "none"),
                               rtol=1e-14, atol=1e-14)


def test_mlp_chain_is_composition_of_gemm_bias_act():
    """Layer by layer, the chain equals GEMM+bias+softplus calls with a final act=none."""
    rng = np.random.default_rng(4)
    x = rng.normal(size=(6, 8))
    Ws = [rng.normal(size=(8, 8)) / 3 for _ in range(3)]
    bs = [rng.normal(size=8) for _ in range(3)]
    h = oracle.gemm_bias_act(x, Ws[0], bs[0], "softplus")
    h = oracle.gemm_bias_act(h, Ws[1], bs[1], "softplus")
    h = oracle.gemm_bias_act(h, Ws[2], bs[2], "none")
    np.testing.assert_allclose(oracle.mlp_chain(x, Ws, bs), h, rtol=1e-13, atol=1e-13)
    rows = [5, 0, 2]
    np.testing.assert_allclose(oracle.mlp_chain_rows(x, Ws, bs, rows), h[rows], rtol=1e-13, atol=1e-13)


def test_mlp_mirror_rounds_intermediates_only():
    rng = np.random.default_rng(6)
    x = rng.normal(size=(4, 8))
    Ws = [rng.normal(size=(8, 8)) / 3 for _ in range(2)]
    bs = [None, None]
    exact = oracle.mlp_chain(x, Ws, bs)
    mirror = oracle.mlp_chain_fp16_mirror(x, Ws, bs)
    assert not np.array_equal(exact, mirror)
    np.testing.assert_allclose(mirror, exact, atol=5e-3)
    # one layer: nothing to round
    assert np.array_equal(oracle.mlp_chain_fp16_mirror(x, Ws[:1], bs[:1]), oracle.mlp_chain(x, Ws[:1], bs[:1]))


# ---------------------------------------------------------------- planted slips
def _pins_pass(gemm, gelu, softplus, mlp):
    """Re-run the core pins against substitute oracle functions; True if all pass."""
    try:
        g = read_golden("gemm_2x2_hand.txt")
        A = np.array(parse_matrix(g["A"]))
        B = np.array(parse_matrix(g["B"]))
        bias = np.array(parse_matrix(g["bias"])[0])
        if not np.array_equal(gemm(A, B, bias, "none"), np.array(parse_matrix(g["Y"]))):
            return False
        xs = np.array([0.5, 1.0, 2.0, -1.0])
        phi = np.array([0.69146246127401310364, 0.84134474606854294859, 0.9772498680518207928,
                        0.15865525393145705141])
        if not np.allclose(gelu(xs), xs * phi, rtol=1e-12, atol=0):
            return False
        if abs(float(softplus(0.0)) - math.log(2.0)) > 1e-15:
            return False
        if abs(float(softplus(-3.0)) - math.log1p(math.exp(-3.0))) > 1e-15:
            return False
        ks = np.array([1.0, 2.0, 3.0])
        out = mlp(np.log(ks)[None, :], [np.eye(3)] * 3, [None] * 3)
        if not np.allclose(out, np.log(ks + 2)[None, :], rtol=1e-13):
            return False
        return True
    except Exception:
        return False


def test_planted_mistakes_are_caught():
    good = (oracle.gemm_bias_act, oracle.act_gelu_erf, oracle.act_softplus, oracle.mlp_chain)
    assert _pins_pass(*good)

    def gemm_transposed_b(A, B, bias, act):
        return oracle.gemm_bias_act(A, np.asarray(B).T, bias, act)

    def gemm_bias_on_rows(A, B, bias, act):
        return oracle.apply_act(np.asarray(A, float) @ np.asarray(B, float) + np.asarray(bias)[:, None], act)

    def gemm_no_bias(A, B, bias, act):
        return oracle.gemm_bias_act(A, B, None, act)

    def gelu_tanh(x):
        x = np.asarray(x, float)
        return 0.5 * x * (1 + np.tanh(math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3)))

    def gelu_no_sqrt2(x):
        from scipy.special import erf
        x = np.asarray(x, float)
        return 0.5 * x * (1 + erf(x))

    def softplus_branchless_misprint(x):
        x = np.asarray(x, float)
        return x + np.log1p(np.exp(-np.abs(x)))

    def mlp_act_on_last(x, Ws, bs):
        h = np.asarray(x, float)
        for W in Ws:
            h = oracle.act_softplus(h @ W)
        return h

    def mlp_one_layer_short(x, Ws, bs):
        return oracle.mlp_chain(x, Ws[:-1], bs[:-1])

    for slip in [
        (gemm_transposed_b, good[1], good[2], good[3]),
        (gemm_bias_on_rows, good[1], good[2], good[3]),
        (gemm_no_bias, good[1], good[2], good[3]),
        (good[0], gelu_tanh, good[2], good[3]),
        (good[0], gelu_no_sqrt2, good[2], good[3]),
        (good[0], good[1], softplus_branchless_misprint, good[3]),
        (good[0], good[1], good[2], mlp_act_on_last),
        (good[0], good[1], good[2], mlp_one_layer_short),
    ]:
        assert not _pins_pass(*slip), slip


# ---------------------------------------------------------------- training side: the backward
def _fd_grads(x, Ws, bs, dout, act, eps=1e-6):
    """Central finite differences of loss = sum(dout * mlp_chain(...)) w.r.t.
    every weight, bias and input entry (tiny shapes only)."""
    def loss(x_, W_, b_):
        return float((oracle.mlp_chain(x_, W_, b_, act) * dout).sum())

    def grad_of(arr, f):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = f()
            arr[idx] = old - eps
            lm = f()
            arr[idx] = old
            g[idx] = (lp - lm) / (2 * eps)
        return g

    dW = [grad_of(W, lambda: loss(x, Ws, bs)) for W in Ws]
    db = [grad_of(b, lambda: loss(x, Ws, bs)) for b in bs]
    dx = grad_of(x, lambda: loss(x, Ws, bs))
    return dx, dW, db


@pytest.mark.parametrize("act", ["softplus", "relu", "none"])
@pytest.mark.parametrize("shapes", [[(3, 4), (4, 2)], [(4, 5), (5, 5), (5, 3)], [(2, 3)], [(3, 6), (6, 6), (6, 6), (6, 2)]])
def test_mlp_backward_matches_finite_differences(act, shapes):
    """The chain rule of mlp_backward against central differences of mlp_chain
    itself (an independent route to the same gradients)."""
    rng = np.random.default_rng(len(shapes) * 13 + len(act))
    x = rng.normal(size=(5, shapes[0][0]))
    Ws = [rng.normal(size=s) * 0.7 for s in shapes]
    bs = [rng.normal(size=s[1]) * 0.3 for s in shapes]
    dout = rng.normal(size=(5, shapes[-1][1]))
    dx, dW, db = oracle.mlp_backward(x, Ws, bs, dout, act)
    fx, fW, fb = _fd_grads(x, Ws, bs, dout, act)
    assert np.allclose(dx, fx, rtol=1e-6, atol=1e-7)
    for a, b in zip(dW, fW):
        assert np.allclose(a, b, rtol=1e-6, atol=1e-7)
    for a, b in zip(db, fb):
        assert np.allclose(a, b, rtol=1e-6, atol=1e-7)


def test_mlp_backward_planted_slips_are_caught():
    """Plausible mistakes in a backward (transposed weight in the data
    gradient, derivative taken at the output instead of the pre-activation,
    bias gradient averaged instead of summed) disagree with the finite
    differences; the test above would catch each of them."""
    rng = np.random.default_rng(7)
    shapes = [(3, 4), (4, 4), (4, 2)]
    x = rng.normal(size=(6, 3))
    Ws = [rng.normal(size=s) * 0.7 for s in shapes]
    bs = [rng.normal(size=s[1]) * 0.3 for s in shapes]
    dout = rng.normal(size=(6, 2))
    fx, fW, fb = _fd_grads(x, Ws, bs, dout, "softplus")
    _, hs, zs = oracle.mlp_forward_train(x, Ws, bs, "softplus")
    # derivative at the output instead of the pre-activation
    g = dout
    g1 = (g @ Ws[2].T) * oracle.act_derivative(hs[1], "softplus")
    assert not np.allclose(hs[0].T @ g1, fW[1], rtol=1e-3)
    # transposed use of a square weight in the data gradient
    g1t = (g @ Ws[2].T) * oracle.act_derivative(zs[1], "softplus")
    g0t = (g1t @ Ws[1]) * oracle.act_derivative(zs[0], "softplus")
    assert not np.allclose(x.T @ g0t, fW[0], rtol=1e-3)
    # averaged bias gradient
    assert not np.allclose(dout.mean(axis=0), fb[2], rtol=1e-3)


def test_act_derivative_textbook_values():
    """sigmoid(0) = 1/2, sigmoid(z) + sigmoid(-z) = 1, ReLU' and identity'."""
    z = np.linspace(-30, 30, 601)
    s = oracle.act_derivative(z, "softplus")
    assert oracle.act_derivative(np.array([0.0]), "softplus")[0] == 0.5
    assert np.allclose(s + oracle.act_derivative(-z, "softplus"), 1.0, atol=1e-15)
    assert np.allclose(s, 1.0 / (1.0 + np.exp(-z)), rtol=1e-14)
    assert (oracle.act_derivative(np.array([-1.0, 2.0]), "relu") == [0.0, 1.0]).all()
    assert (oracle.act_derivative(z, "none") == 1.0).all()


def test_act_derivative_from_output_matches_pre_activation_form():
    """softplus' written through the output h = softplus(z) equals sigmoid(z)
    (two different formulas: 1 - e^-h against the tanh form of the sigmoid),
    over a range wide enough that h is tiny (z << 0) and e^-h underflows
    (z >> 0); ReLU' and identity' agree on h = act(z)."""
    z = np.linspace(-40, 40, 801)
    for act in ("softplus", "relu", "none"):
        h = oracle.apply_act(z, act)
        a = oracle.act_derivative_from_output(h, act)
        b = oracle.act_derivative(z, act)
        # the tanh form of the sigmoid rounds to 0 below z ~ -37: absolute agreement
        assert np.allclose(a, b, rtol=1e-12, atol=1e-16), act
    # h small: 1 - e^-h ~ h (the form keeps relative precision there)
    h = np.array([1e-12, 1e-6])
    assert np.allclose(oracle.act_derivative_from_output(h, "softplus"), h, rtol=1e-6)


@pytest.mark.parametrize("act", ["softplus", "relu", "none"])
def test_mlp_backward_from_activations_matches_chain_rule(act):
    """Given the forward's own activations, the stored-activation backward
    equals mlp_backward (pinned to finite differences above); given other
    activations it differs, so the activations are really used."""
    rng = np.random.default_rng(17)
    shapes = [(4, 6), (6, 6), (6, 3)]
    x = rng.normal(size=(7, 4))
    Ws = [rng.normal(size=s) * 0.7 for s in shapes]
    bs = [rng.normal(size=s[1]) * 0.3 for s in shapes]
    dout = rng.normal(size=(7, 3))
    _, hs, _ = oracle.mlp_forward_train(x, Ws, bs, act)
    rx, rW, rb = oracle.mlp_backward(x, Ws, bs, dout, act)
    dx, dW, db, gs = oracle.mlp_backward_from_activations(x, Ws, hs, dout, act)
    assert np.allclose(dx, rx, rtol=1e-12, atol=1e-14)
    for a, b in zip(dW + db, rW + rb):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    assert np.array_equal(gs[-1], dout) and np.allclose(db[0], gs[0].sum(axis=0))
    perturbed = [h + 0.25 for h in hs]
    _, pW, _, _ = oracle.mlp_backward_from_activations(x, Ws, perturbed, dout, act)
    assert not np.allclose(pW[1], rW[1], rtol=1e-3)
