"""GPU parity for the training side: coalesce_gemm_ex (transposed operands,
fp32 accumulation, activation-derivative epilogue) and the chained MLP's
coalesce_mlp_forward_train / coalesce_mlp_backward, against the fp64 oracle.

Tolerances, written here:

* Integer-valued operands: every product and partial sum is an exact fp32
  integer (|sum| < 2^24), so the result must equal the exact value bit for
  bit, whatever the order of the (atomic) additions.
* DACT epilogue: (A B) * act'(aux) rounded once to fp16: 1e-2 + 2^-11 |ref|
  against fp64 on the same inputs, as for the forward GEMM.
* Gradients: against the oracle's backward given the kernel's stored
  activations (the backward's contract; the forward's accuracy is tested on
  its own).  Each output is a sum of products whose operands the GPU holds in
  fp16/bf16 (unit roundoff u = 2^-11 / 2^-8), with fp32 sums: (L + 3) u S,
  S = the sum of the absolute values of its terms, plus the first-order
  propagation of the data gradients' roundings down the chain (check_grads),
  which dominates when few rows are summed; for dx also + u |ref|, its final
  rounding.
"""
import numpy as np
import pytest
import torch

import gemm_bias_activation_gb300 as g
import oracle
from gemm_bias_activation_gb300 import inputs

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}
U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def stream():
    return torch.cuda.current_stream().cuda_stream


def gemm_ex(M, N, K, dtype, flags, A, B, Y, bias=None, aux=None, act="none"):
    st = g.coalesce_gemm_ex(M, N, K, g._dtype_code(A), flags, A.data_ptr(), B.data_ptr(),
                            None if bias is None else bias.data_ptr(), None if aux is None else aux.data_ptr(),
                            Y.data_ptr(), g.ACT_CODES[act], stream())
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(stream()) == 0


def ints(shape, lo, hi, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=gen).to(DT[dtype])


# ---------------------------------------------------------------- transposed operands (store mode), bit-exact
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 136, 72), (520, 264, 1032), (64, 1000, 200), (8, 24, 40)])
def test_transposed_operands_exact(dtype, ta, tb, M, N, K):
    A = ints((M, K), -3, 3, dtype, 1)
    B = ints((K, N), -2, 2, dtype, 2)
    Ad = (A.t().contiguous() if ta else A).cuda()
    Bd = (B.t().contiguous() if tb else B).cuda()
    Y = torch.full((M, N), float("nan"), dtype=DT[dtype], device="cuda")
    flags = (g.COALESCE_GEMM_TRANS_A if ta else 0) | (g.COALESCE_GEMM_TRANS_B if tb else 0)
    gemm_ex(M, N, K, dtype, flags, Ad, Bd, Y)
    want = torch.from_numpy(f64(A) @ f64(B)).to(DT[dtype])
    assert torch.equal(Y.cpu(), want)


# ---------------------------------------------------------------- fp32 accumulation (split K, atomic), bit-exact
@pytest.mark.parametrize("ta", [True, False])
@pytest.mark.parametrize("M,N,K", [(64, 64, 65536), (128, 128, 100000), (200, 136, 4096), (256, 192, 40000),
                                   (136, 64, 72), (8, 16, 5000)])
def test_accum_f32_exact(ta, M, N, K):
    A = ints((M, K), -3, 3, "f16", 3)
    B = ints((K, N), -2, 2, "f16", 4)
    Ad = (A.t().contiguous() if ta else A).cuda()
    Y0 = ints((M, N), -50, 50, "f16", 5).float()
    Y = Y0.cuda()
    flags = g.COALESCE_GEMM_ACCUM_F32 | (g.COALESCE_GEMM_TRANS_A if ta else 0)
    gemm_ex(M, N, K, "f16", flags, Ad, B.cuda(), Y)
    want = f64(Y0) + f64(A) @ f64(B)  # |sum| < 2^24: exact in fp32
    assert np.array_equal(f64(Y), want)


# ---------------------------------------------------------------- derivative epilogue
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("act", ["softplus", "relu", "none"])
@pytest.mark.parametrize("in_place", [False, True])
def test_dact_epilogue(dtype, act, in_place):
    M, N, K = 777, 200, 136
    gA = inputs.normal((M, K), 6, 1, dtype, 1.0)
    W = inputs.normal((N, K), 6, 2, dtype, 1.0 / K)  # given as Bt [N, K]
    hz = inputs.normal((M, N), 6, 3, dtype, 4.0)
    h = torch.from_numpy(oracle.apply_act(f64(hz), act)).to(DT[dtype])  # an activation's output
    hd = h.cuda()
    Y = hd if in_place else torch.empty((M, N), dtype=DT[dtype], device="cuda")
    gemm_ex(M, N, K, dtype, g.COALESCE_GEMM_DACT | g.COALESCE_GEMM_TRANS_B, gA.cuda(), W.cuda(), Y, aux=hd, act=act)
    hv = f64(h)
    d = -np.expm1(-hv) if act == "softplus" else (hv > 0).astype(np.float64) if act == "relu" else np.ones_like(hv)
    ref = (f64(gA) @ f64(W).T) * d
    tol = 1e-2 + (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11) * np.abs(ref)
    err = np.abs(f64(Y) - ref)
    assert (err <= tol).all(), f"max err {err.max():.3e}"


# ---------------------------------------------------------------- MLP training
def mk(rows, D, H, O, L, dtype, seed):
    w = inputs.MlpWorkload("t", rows, D, H, L, dtype, 1.0 / H, 0.01, "softplus", O)
    x, Ws, bs = inputs.mlp_inputs(w, seed=seed)
    dout = inputs.normal((rows, O), seed, 99, dtype, 1.0)
    return x, Ws, bs, dout


def forward_train(x, Ws, bs, H, O, act, dtype):
    rows, D = x.shape
    L = len(Ws)
    xd, Wd, bd = x.cuda(), [w.cuda() for w in Ws], [b.cuda() for b in bs]
    hs = [torch.empty((rows, H), dtype=DT[dtype], device="cuda") for _ in range(L - 1)]
    out = torch.empty((rows, O), dtype=DT[dtype], device="cuda")
    st = g.coalesce_mlp_forward_train(rows, D, H, O, L, g._dtype_code(x), xd.data_ptr(), [w.data_ptr() for w in Wd],
                                      [b.data_ptr() for b in bd], [h.data_ptr() for h in hs], out.data_ptr(),
                                      g.ACT_CODES[act], stream())
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(stream()) == 0
    return xd, Wd, hs, out


GUARD = 256  # NaN elements after every output, which no call may write


def _guarded(shape, dtype):
    n = 1
    for d in shape:
        n *= d
    store = torch.full((n + GUARD,), float("nan"), dtype=dtype, device="cuda")
    return store[:n].view(*shape), store


def backward(xd, Wd, hs, dout, H, O, act, dtype, want_dx=True, want_db=True):
    rows, D = xd.shape
    L = len(Wd)
    dW, db, stores = [], [], []
    for w in Wd:
        t, st_ = _guarded((w.shape[0], w.shape[1]), torch.float32)
        dW.append(t)
        stores.append(st_)
        t, st_ = _guarded((w.shape[1],), torch.float32)
        db.append(t)
        stores.append(st_)
    dx = None
    if want_dx:
        dx, st_ = _guarded((rows, D), DT[dtype])
        stores.append(st_)
    dd = dout.cuda()
    st = g.coalesce_mlp_backward(rows, D, H, O, L, g._dtype_code(xd), xd.data_ptr(), [w.data_ptr() for w in Wd],
                                 [h.data_ptr() for h in hs], dd.data_ptr(), None if dx is None else dx.data_ptr(),
                                 [t.data_ptr() for t in dW], [t.data_ptr() for t in db] if want_db else None,
                                 g.ACT_CODES[act], stream())
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(stream()) == 0
    for st_ in stores:
        assert torch.isnan(st_[-GUARD:].float()).all(), "write beyond an output"
    return dx, dW, db


def check_grads(x, Ws, dout, act, dtype, dx, dW, db, gpu_h):
    """Against the oracle's backward given the kernel's own stored activations
    gpu_h (copies taken before the backward, which may overwrite them): the
    backward's contract is the gradient for the activations it is handed, and
    it takes every derivative from them, as the oracle does here.

    Tolerance (first order): E_l bounds |g_l(kernel) - g_l| elementwise.
    E_{L-1} = 0 (dout is exact); the kernel forms g_{l-1} = (g_l W_l^T) * d
    in fp32 from its g_l and rounds it to dtype, so
      E_{l-1} = (E_l |W_l|^T + N_l 2^-24 |g_l| |W_l|^T) |d| + 2^-21 |g_l W_l^T| + u |g_{l-1}|.
    Each gradient then carries the propagated error of its g plus (L + 3) u S
    for its own sums (S = the sum of the absolute values of its terms)."""
    L = len(Ws)
    u = U[dtype]
    xs, Wn, dn = f64(x), [f64(w) for w in Ws], f64(dout)
    hs = [f64(h) for h in gpu_h]
    rdx, rdW, rdb, gs = oracle.mlp_backward_from_activations(xs, Wn, hs, dn, act)
    ins = [xs] + hs
    E = [None] * L
    E[L - 1] = np.zeros_like(dn)
    for l in range(L - 1, 0, -1):
        aW = np.abs(Wn[l]).T
        d = np.abs(oracle.act_derivative_from_output(ins[l], act))
        N = Wn[l].shape[1]
        E[l - 1] = (E[l] @ aW + N * 2.0 ** -24 * (np.abs(gs[l]) @ aW)) * d + \
            2.0 ** -21 * np.abs(gs[l] @ Wn[l].T) + u * np.abs(gs[l - 1])
    c = (L + 3) * u
    for l in range(L if dW is not None else 0):
        S = np.abs(ins[l]).T @ np.abs(gs[l])
        tol = c * S + np.abs(ins[l]).T @ E[l] + 1e-30
        err = np.abs(f64(dW[l]) - rdW[l])
        assert (err <= tol).all(), f"dW[{l}] max err/tol {np.max(err / tol):.2f}"
        if db is not None:
            tolb = c * np.abs(gs[l]).sum(axis=0) + E[l].sum(axis=0) + 1e-30
            errb = np.abs(f64(db[l]) - rdb[l])
            assert (errb <= tolb).all(), f"db[{l}] max err/tol {np.max(errb / tolb):.2f}"
    if dx is not None:
        aW0 = np.abs(Wn[0]).T
        tolx = c * (np.abs(gs[0]) @ aW0) + E[0] @ aW0 + u * np.abs(rdx) + 1e-30
        errx = np.abs(f64(dx) - rdx)
        assert (errx <= tolx).all(), f"dx max err/tol {np.max(errx / tolx):.2f}"


def forward_error_bound(x, Ws, bs, act, dtype):
    """First-order bounds on how far the kernel's forward activations and
    output can be from the exact fp64 chain: ([eh_0 .. eh_{L-1}], e_out), eh_l
    for the input of layer l (eh_0 = 0: x is exact).

    Per layer the fp32 accumulation adds e_{l-1} |W_l| + K 2^-24 (|h| |W_l| +
    |b_l|).  An fp16 softplus rounds z to fp16 (u |z|) and evaluates on packed
    fp16 pairs, within 2e-3 + 2^-10 |h| of softplus of that value
    (test_mlp_gpu.py's test_softplus_epilogue_error_bound pins this);
    softplus is 1-Lipschitz.  A bf16 softplus runs in fp32 (__expf/__logf,
    ~1e-6) and rounds h to bf16 (u |h|).  The output adds its own rounding
    u |out|."""
    u = U[dtype]
    h = f64(x)
    e = np.zeros_like(h)
    ehs = [e]
    L = len(Ws)
    for l in range(L):
        W = f64(Ws[l])
        b = np.zeros(W.shape[1]) if bs is None or bs[l] is None else f64(bs[l])
        aW = np.abs(W)
        z = h @ W + b[None, :]
        ez = e @ aW + W.shape[0] * 2.0 ** -24 * (np.abs(h) @ aW + np.abs(b)[None, :])
        if l == L - 1:
            return ehs, ez + u * np.abs(z)
        assert act == "softplus"
        h = oracle.act_softplus(z)
        if dtype == "f16":
            e = ez + u * np.abs(z) + 2e-3 + 2.0 ** -10 * np.abs(h)
        else:
            e = ez + 1e-6 + u * np.abs(h)
        ehs.append(e)


def check_step_end_to_end(x, Ws, bs, dout, dtype, out, dx, dW, db):
    """A whole training step (forward storing activations, then backward)
    against the oracle's backward on the exact fp64 chain, softplus.

    The tolerance is the backward's own bound (check_grads, for the
    activations it is handed) plus what the forward's activation error eh_l
    (forward_error_bound) propagates into the gradients, to first order:
      Dg_{L-1} = 0,
      Dg_{l-1} = (Dg_l |W_l|^T) |act'(h_l)| + |g_l W_l^T| e^-h_l eh_l
        (softplus' = 1 - e^-h, whose derivative in h is e^-h),
      dW_l: eh_l^T |g_l| + |in_l|^T Dg_l,   db_l: the row sum of Dg_l,
      dx: Dg_0 |W_1|^T."""
    L = len(Ws)
    u = U[dtype]
    xs, Wn, bn, dn = f64(x), [f64(w) for w in Ws], [f64(b) for b in bs], f64(dout)
    rout, rhs, _ = oracle.mlp_forward_train(xs, Wn, bn, "softplus")
    rdx, rdW, rdb = oracle.mlp_backward(xs, Wn, bn, dn, "softplus")
    _, _, _, gs = oracle.mlp_backward_from_activations(xs, Wn, rhs, dn, "softplus")
    ehs, e_out = forward_error_bound(x, Ws, bs, "softplus", dtype)
    ins = [xs] + rhs
    # the forward's output
    err = np.abs(f64(out) - rout)
    tol = 1e-2 + u * np.abs(rout) + (0.0 if dtype == "f16" else e_out)
    assert (err <= tol).all(), f"out: max err/tol {np.max(err / tol):.2f}"
    # the backward's own rounding (as check_grads), around the exact activations
    E = [None] * L
    E[L - 1] = np.zeros_like(dn)
    for l in range(L - 1, 0, -1):
        aW = np.abs(Wn[l]).T
        d = np.abs(oracle.act_derivative_from_output(ins[l], "softplus"))
        E[l - 1] = (E[l] @ aW + Wn[l].shape[1] * 2.0 ** -24 * (np.abs(gs[l]) @ aW)) * d + \
            2.0 ** -21 * np.abs(gs[l] @ Wn[l].T) + u * np.abs(gs[l - 1])
    # what the forward's activation error propagates
    Dg = [None] * L
    Dg[L - 1] = np.zeros_like(dn)
    for l in range(L - 1, 0, -1):
        d = np.abs(oracle.act_derivative_from_output(ins[l], "softplus"))
        Dg[l - 1] = (Dg[l] @ np.abs(Wn[l]).T) * d + np.abs(gs[l] @ Wn[l].T) * np.exp(-ins[l]) * ehs[l]
    c = (L + 3) * u
    for l in range(L):
        tolw = c * (np.abs(ins[l]).T @ np.abs(gs[l])) + np.abs(ins[l]).T @ (E[l] + Dg[l]) + \
            ehs[l].T @ np.abs(gs[l]) + 1e-30
        errw = np.abs(f64(dW[l]) - rdW[l])
        assert (errw <= tolw).all(), f"dW[{l}]: max err/tol {np.max(errw / tolw):.2f}"
        tolb = c * np.abs(gs[l]).sum(axis=0) + (E[l] + Dg[l]).sum(axis=0) + 1e-30
        errb = np.abs(f64(db[l]) - rdb[l])
        assert (errb <= tolb).all(), f"db[{l}]: max err/tol {np.max(errb / tolb):.2f}"
    aW0 = np.abs(Wn[0]).T
    tolx = c * (np.abs(gs[0]) @ aW0) + (E[0] + Dg[0]) @ aW0 + u * np.abs(rdx) + 1e-30
    errx = np.abs(f64(dx) - rdx)
    assert (errx <= tolx).all(), f"dx: max err/tol {np.max(errx / tolx):.2f}"


# (128, 128, 128, 6) and (256, 256, 256, 2) stream their weights through the
# fused forward (192 and 256 KiB) and take the GEMM-form backward; (72, 136,
# 40, 3) and (8, 24, 16, 2) run the fused forward on widths padded to 64.
TRAIN_SHAPES = [(128, 128, 128, 3), (64, 64, 64, 5), (64, 128, 192, 3), (256, 64, 128, 2), (64, 64, 256, 1),
                (72, 136, 40, 3), (128, 128, 128, 6), (256, 256, 256, 2), (8, 24, 16, 2)]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,H,O,L", TRAIN_SHAPES)
def test_forward_train_matches_oracle(dtype, D, H, O, L):
    rows = 1500
    x, Ws, bs, _ = mk(rows, D, H, O, L, dtype, seed=D + O + L)
    _, _, hs, out = forward_train(x, Ws, bs, H, O, "softplus", dtype)
    rout, rhs, _ = oracle.mlp_forward_train(f64(x), [f64(w) for w in Ws], [f64(b) for b in bs], "softplus")
    # every stored activation and the output are a GEMM + bias + softplus of
    # the previous stored value: compare each against the oracle layer applied
    # to the GPU's own input, with the GEMM tolerance
    ins = [f64(x)] + [f64(h) for h in hs]
    tol_u = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    for l in range(L):
        z = ins[l] @ f64(Ws[l]) + f64(bs[l])[None, :]
        ref = z if l == L - 1 else oracle.act_softplus(z)
        got = f64(out) if l == L - 1 else ins[l + 1]
        err = np.abs(got - ref)
        assert (err <= 1e-2 + tol_u * np.abs(ref)).all(), f"layer {l}: max err {err.max():.3e}"
    assert np.isfinite(f64(out)).all() and len(rhs) == L - 1
    # and the output against the exact fp64 chain: the stated bound for fp16,
    # plus the propagated rounding of the bf16 intermediates for bf16
    extra = 0.0 if dtype == "f16" else forward_error_bound(x, Ws, bs, "softplus", dtype)[1]
    err = np.abs(f64(out) - rout)
    tol = 1e-2 + tol_u * np.abs(rout) + extra
    assert (err <= tol).all(), f"out vs the fp64 chain: max err {err.max():.3e}, max err/tol {np.max(err / tol):.2f}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,H,O,L", TRAIN_SHAPES)
def test_backward_matches_oracle(dtype, D, H, O, L):
    rows = 3000
    x, Ws, bs, dout = mk(rows, D, H, O, L, dtype, seed=2 * D + L)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", dtype)
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, "softplus", dtype)
    check_grads(x, Ws, dout, "softplus", dtype, dx, dW, db, h_copy)


# shapes the fused backward kernel takes (K_l <= 128, the dW accumulators
# within 512 TMEM columns, widths rounded up to 64), among them one and two
# column groups, a two-slot ring (L = 1, wide output), rows beyond K_l, and
# widths that are not multiples of 64 (dW, db and dx clipped to them)
@pytest.mark.parametrize("rows", [1, 129, 5000])
@pytest.mark.parametrize("D,H,O,L", [(128, 64, 64, 4), (128, 128, 64, 2), (64, 128, 128, 2), (128, 128, 256, 1),
                                     (64, 64, 128, 3), (72, 40, 24, 3), (8, 24, 16, 2), (120, 56, 200, 1),
                                     (40, 104, 8, 3)])
def test_backward_fused_shapes(rows, D, H, O, L):
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=rows + 3 * D + O + L)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", "f16")
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, "softplus", "f16")
    check_grads(x, Ws, dout, "softplus", "f16", dx, dW, db, h_copy)


@pytest.mark.parametrize("act", ["softplus", "relu"])
def test_backward_fused_padded_bf16(act):
    rows, D, H, O, L = 2000, 72, 40, 24, 3
    x, Ws, bs, dout = mk(rows, D, H, O, L, "bf16", seed=17)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, act, "bf16")
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, act, "bf16")
    check_grads(x, Ws, dout, act, "bf16", dx, dW, db, h_copy)


def test_backward_fused_deepest_chain():
    """7 layers of 64: one 64-column acc2 plus seven 64-column dW accumulators
    fill the 512 TMEM columns exactly (the fused kernel's largest chain)."""
    rows, D, H, O, L = 3000, 64, 64, 64, 7
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=31)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", "f16")
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, "softplus", "f16")
    check_grads(x, Ws, dout, "softplus", "f16", dx, dW, db, h_copy)


def test_backward_some_bias_gradients_null():
    """db entries may be NULL one by one: the others are still produced, and
    the NULL ones are never written."""
    rows, D, H, O, L = 2500, 128, 128, 128, 3
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=32)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", "f16")
    h_copy = [h.clone() for h in hs]
    dW = [torch.empty((w.shape[0], w.shape[1]), dtype=torch.float32, device="cuda") for w in Wd]
    db = [torch.empty((w.shape[1],), dtype=torch.float32, device="cuda") for w in Wd]
    dx = torch.empty((rows, D), dtype=torch.float16, device="cuda")
    dd = dout.cuda()
    st = g.coalesce_mlp_backward(rows, D, H, O, L, g.COALESCE_F16, xd.data_ptr(), [w.data_ptr() for w in Wd],
                                 [h.data_ptr() for h in hs], dd.data_ptr(), dx.data_ptr(), [t.data_ptr() for t in dW],
                                 [db[0].data_ptr(), None, db[2].data_ptr()], g.ACT_CODES["softplus"], stream())
    assert st == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(stream()) == 0
    check_grads(x, Ws, dout, "softplus", "f16", dx, dW, None, h_copy)
    _, _, rdb, gs = oracle.mlp_backward_from_activations(f64(x), [f64(w) for w in Ws], [f64(h) for h in h_copy],
                                                         f64(dout), "softplus")
    for l in (0, 2):
        tol = (L + 3) * U["f16"] * np.abs(gs[l]).sum(axis=0) + 1e-3
        assert (np.abs(f64(db[l]) - rdb[l]) <= tol).all(), f"db[{l}]"


@pytest.mark.parametrize("act", ["relu", "none"])
def test_backward_other_activations(act):
    rows, D, H, O, L = 2000, 64, 128, 64, 3
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=5)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, act, "f16")
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, act, "f16")
    check_grads(x, Ws, dout, act, "f16", dx, dW, db, h_copy)


def test_backward_many_rows_split_k():
    """2^17 rows: the weight gradients' K = rows is split over every SM."""
    rows, D, H, O, L = 1 << 17, 128, 128, 128, 3
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=11)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", "f16")
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, H, O, "softplus", "f16", want_dx=False)
    check_grads(x, Ws, dout, "softplus", "f16", None, dW, db, h_copy)


def test_backward_optional_outputs_null():
    rows, D, H, O, L = 700, 64, 64, 64, 2
    x, Ws, bs, dout = mk(rows, D, H, O, L, "f16", seed=12)
    xd, Wd, hs, _ = forward_train(x, Ws, bs, H, O, "softplus", "f16")
    h_copy = [h.clone() for h in hs]
    dx, dW, _ = backward(xd, Wd, hs, dout, H, O, "softplus", "f16", want_dx=False, want_db=False)
    check_grads(x, Ws, dout, "softplus", "f16", None, dW, None, h_copy)


def test_training_step_full_size_workload():
    """The bench's training workload (3-layer, 128 wide, 2^20 rows, seed 0):
    every dW, db and dx entry against the fp64 oracle's backward for the
    stored activations."""
    w = inputs.WORKLOADS["fp16_mlp3_softplus_128w_2p20rows_train"]
    x, Ws, bs = inputs.mlp_inputs(w, seed=0)
    dout = inputs.normal((w.rows, w.out_width), 0, 99, w.dtype, 1.0)
    xd, Wd, hs, out = forward_train(x, Ws, bs, w.H, w.out_width, w.act, w.dtype)
    assert torch.isfinite(out.float()).all()
    h_copy = [h.clone() for h in hs]
    dx, dW, db = backward(xd, Wd, hs, dout, w.H, w.out_width, w.act, w.dtype)
    check_grads(x, Ws, dout, w.act, w.dtype, dx, dW, db, h_copy)


@pytest.mark.parametrize("rows,D,H,L", [(65536, 128, 128, 3), (65536, 64, 64, 5), (4133, 128, 128, 3),
                                        (1, 64, 64, 5)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_training_step_end_to_end(rows, D, H, L, dtype):
    """The whole step (fused forward storing activations, then the backward)
    against the oracle's gradients of the exact fp64 chain, on the two timed
    chain shapes (3 layers of 128, 5 of 64) with W ~ N(0, 1/H) and
    b ~ N(0, 0.01) (variances)."""
    x, Ws, bs, dout = mk(rows, D, H, H, L, dtype, seed=rows + L)
    xd, Wd, hs, out = forward_train(x, Ws, bs, H, H, "softplus", dtype)
    out_h = out.clone()
    dx, dW, db = backward(xd, Wd, hs, dout, H, H, "softplus", dtype)
    check_step_end_to_end(x, Ws, bs, dout, dtype, out_h, dx, dW, db)
