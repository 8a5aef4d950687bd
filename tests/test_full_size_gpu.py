"""Whole-output parity at the workloads' full sizes, through the C ABI, in the
launch configurations the bench times.

"Fuse Elementwise Ops", "Correctness requirements": the fused kernel must
match the unfused sequence everywhere, the last partial tile included.  Here
every element of every full-size output is compared with the fp64 oracle, not
a sample of rows.  The oracle is evaluated in row blocks (each output row
depends only on its own input row, so a block is computed exactly as the whole
problem would be).

Tolerances (as in the other parity tests, written here):

* bf16 / fp16 outputs: |gpu - ref| <= 1e-2 + half an output ulp of ref
  (2^-8 |ref| for bf16, 2^-11 |ref| for fp16).  The raw max |err| and the
  number of elements over a plain 1e-2 are printed as well: for bf16, a
  correctly rounded output above |ref| = 2.56 can be more than 1e-2 from the
  exact value, which is what the ulp term admits.
* fp32 outputs: |gpu - ref| <= 1e-4 max(1, |ref|).
"""
import numpy as np
import pytest
import torch

import gemm_bias_activation_gb300 as g
import oracle
from gemm_bias_activation_gb300 import inputs

pytestmark = pytest.mark.gpu

HALF_ULP = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


class Stats:
    """Running comparison over row blocks of one output."""

    def __init__(self, dtype, what):
        self.dtype, self.what = dtype, what
        self.n = self.bad = self.over_plain = 0
        self.max_err = self.max_ratio = 0.0
        self.first_bad = None

    def add(self, got, ref, row0):
        err = np.abs(got - ref)
        a = np.abs(ref)
        if self.dtype == "f32":
            tol = 1e-4 * np.maximum(1.0, a)
        else:
            tol = 1e-2 + HALF_ULP[self.dtype] * a
            self.over_plain += int((err > 1e-2).sum())
        assert not np.isnan(got).any(), f"{self.what}: NaN in rows {row0}.."
        bad = err > tol
        if bad.any() and self.first_bad is None:
            i, j = np.unravel_index(np.argmax(bad), bad.shape)
            self.first_bad = (row0 + i, j, got[i, j], ref[i, j])
        self.bad += int(bad.sum())
        self.n += err.size
        self.max_err = max(self.max_err, float(err.max()))
        self.max_ratio = max(self.max_ratio, float((err / tol).max()))

    def finish(self):
        print(f"\n{self.what}: {self.n} elements, max |err| {self.max_err:.3e}, max err/tol {self.max_ratio:.3f}, "
              f"over plain 1e-2: {self.over_plain}")
        assert self.bad == 0, f"{self.what}: {self.bad} of {self.n} over tolerance, first (row, col, gpu, ref) " \
                              f"{self.first_bad}"


def test_ffn_up_projection_full_output():
    """bf16 X[16384,4096] @ W[4096,16384] + bias, GELU_erf: all 2^28 outputs."""
    w = inputs.WORKLOADS["bf16_ffn_up_bias_gelu_16384x16384x4096"]
    A, B, bias = inputs.gemm_inputs(w, seed=0)
    Y = g.gemm_bias_act(A.cuda(), B.cuda(), bias.cuda(), "gelu_erf")
    g.device_status()
    Yh = Y.cpu()
    del Y
    A64, B64, b64 = f64(A), f64(B), f64(bias)
    st = Stats("bf16", "ffn 16384x16384x4096")
    blk = 1024
    for r0 in range(0, w.M, blk):
        ref = oracle.gemm_bias_act(A64[r0:r0 + blk], B64, b64, "gelu_erf")
        st.add(f64(Yh[r0:r0 + blk]), ref, r0)
    st.finish()


@pytest.mark.parametrize("n", [2048, 4096])
def test_f32_sweep_full_output(n):
    """FP32 square GEMM + bias + GELU_erf at the sweep's two largest sizes: every output."""
    w = inputs.WORKLOADS[f"fp32_gemm_bias_gelu_{n}"]
    A, B, bias = inputs.gemm_inputs(w, seed=0)
    Y = g.gemm_bias_act(A.cuda(), B.cuda(), bias.cuda(), "gelu_erf")
    g.device_status()
    st = Stats("f32", f"fp32 {n}^3")
    st.add(f64(Y), oracle.gemm_bias_act(f64(A), f64(B), f64(bias), "gelu_erf"), 0)
    st.finish()


@pytest.mark.parametrize("name", ["fp16_mlp3_softplus_128w_2p20rows", "fp16_mlp5_softplus_64w_2p22rows"])
def test_mlp_full_output(name):
    """The two chained-MLP workloads (2^20 rows x 128, 3 layers; 2^22 rows x 64,
    5 layers): every output element against the fp64 chain."""
    w = inputs.WORKLOADS[name]
    x, Ws, bs = inputs.mlp_inputs(w, seed=0)
    xd, Wd, bd = x.cuda(), [t.cuda() for t in Ws], [t.cuda() for t in bs]
    out = torch.empty((w.rows, w.H), dtype=xd.dtype, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = g.coalesce_mlp_fused(w.rows, w.D, w.H, w.L, xd.data_ptr(), [t.data_ptr() for t in Wd],
                              [t.data_ptr() for t in bd], out.data_ptr(), g.ACT_CODES[w.act], stream)
    assert rc == 0, g.coalesce_last_error()
    assert g.coalesce_device_status(stream) == 0
    oh = out.cpu()
    del out, xd
    W64, b64 = [f64(t) for t in Ws], [f64(t) for t in bs]
    st = Stats(w.dtype, name)
    blk = 1 << 18
    for r0 in range(0, w.rows, blk):
        ref = oracle.mlp_chain(f64(x[r0:r0 + blk]), W64, b64, w.act)
        st.add(f64(oh[r0:r0 + blk]), ref, r0)
    st.finish()
