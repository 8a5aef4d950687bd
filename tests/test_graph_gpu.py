"""The entry points inside a CUDA graph (the small-M, launch-bound regime).

A call allocates nothing and never synchronises the host, so a sequence of
calls can be captured once and replayed; replays must give the same bits as
eager calls.  The "MLP Megakernel" README (Ablation Study) shows why this
matters at small row counts: there the launch, not the kernel, dominates.
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


@pytest.mark.parametrize("rows", [64, 1024, 8192])
def test_mlp_graph_replay_matches_eager(rows):
    w = inputs.WORKLOADS["fp16_mlp3_softplus_128w_2p20rows"]
    x, Ws, bs = inputs.mlp_inputs(w, seed=2, rows=rows)
    x, Ws, bs = x.cuda(), [t.cuda() for t in Ws], [t.cuda() for t in bs]
    eager = g.mlp_fused(x, Ws, bs)
    g.device_status()
    out = torch.empty_like(eager)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.mlp_fused(x, Ws, bs, out=out)
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    g.device_status()
    assert torch.equal(out, eager)
    ref = oracle.mlp_chain(f64(x), [f64(t) for t in Ws], [f64(t) for t in bs])
    assert (np.abs(f64(out) - ref) <= 1e-2 + 2.0 ** -11 * np.abs(ref)).all()


def test_gemm_graph_replay_matches_eager():
    for dtype in ["bf16", "f32"]:
        wname = "bf16_ffn_up_bias_gelu_16384x16384x4096" if dtype == "bf16" else "fp32_gemm_bias_gelu_256"
        w = inputs.WORKLOADS[wname]
        A, B, bias = (t.cuda() for t in inputs.gemm_inputs(w, seed=3, M=320, N=264, K=136))
        eager = g.gemm_bias_act(A, B, bias, "gelu_erf")
        unfused_eager = g.gemm_then_bias_act(A, B, bias, "gelu_erf")
        g.device_status()
        Y = torch.empty_like(eager)
        Y2 = torch.empty_like(eager)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.gemm_bias_act(A, B, bias, "gelu_erf", out=Y)
            g.gemm_then_bias_act(A, B, bias, "gelu_erf", out=Y2)
        graph.replay()
        torch.cuda.synchronize()
        g.device_status()
        assert torch.equal(Y, eager)
        assert torch.equal(Y2, unfused_eager)


def test_cta_pair_gemm_graph_replay_matches_eager():
    """The CTA-pair kernel (cluster launch) captured into a graph, its first
    call made during the capture, replays to the eager call's bits."""
    w = inputs.WORKLOADS["bf16_ffn_up_bias_gelu_16384x16384x4096"]
    A, B, bias = (t.cuda() for t in inputs.gemm_inputs(w, seed=5, M=4096, N=4864, K=128))
    out = torch.empty((4096, 4864), dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gemm_bias_act(A, B, bias, "gelu_erf", out=out)
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    g.device_status()
    eager = g.gemm_bias_act(A, B, bias, "gelu_erf")
    g.device_status()
    assert torch.equal(out, eager)


def test_training_step_graph_replay_matches_eager():
    """Forward (activations stored) + backward captured in one graph: the
    forward output and dx equal the eager call bit for bit; dW and db are fp32
    sums over the rows whose addition order differs between calls (atomic and
    TMA reduce-add across CTAs).  Two orders of the same n fp32 additions
    differ by at most 2 n 2^-24 S (first order), S the sum of the terms'
    magnitudes, computed here from the stored activations."""
    w = inputs.MlpWorkload("t", 3000, 64, 128, 3, "f16", 1.0 / 128, 0.01, "softplus", 64)
    x, Ws, bs = (t for t in inputs.mlp_inputs(w, seed=4))
    x, Ws, bs = x.cuda(), [t.cuda() for t in Ws], [t.cuda() for t in bs]
    dout = inputs.normal((w.rows, 64), 4, 99, "f16", 1.0).cuda()
    out_e, hs_e = g.mlp_forward_train(x, Ws, bs)
    h_host = [f64(h) for h in hs_e]  # the backward consumes hs_e
    dx_e, dW_e, db_e = g.mlp_backward(x, Ws, hs_e, dout)
    g.device_status()
    out = torch.empty_like(out_e)
    hs = [torch.empty_like(h) for h in hs_e]
    dx = torch.empty_like(dx_e)
    dW = [torch.empty_like(t) for t in dW_e]
    db = [torch.empty_like(t) for t in db_e]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.mlp_forward_train(x, Ws, bs, hs=hs, out=out)
        g.mlp_backward(x, Ws, hs, dout, dW=dW, db=db, dx=dx)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    g.device_status()
    assert torch.equal(out, out_e)
    assert torch.equal(dx, dx_e)
    _, _, _, gs = oracle.mlp_backward_from_activations(f64(x), [f64(t) for t in Ws], h_host, f64(dout), "softplus")
    ins = [f64(x)] + h_host
    bound = 2.0 * w.rows * 2.0 ** -24
    for l in range(w.L):
        s_dw = np.abs(ins[l]).T @ np.abs(gs[l])
        s_db = np.abs(gs[l]).sum(axis=0)
        assert (np.abs(f64(dW[l]) - f64(dW_e[l])) <= bound * s_dw + 1e-30).all(), f"dW[{l}]"
        assert (np.abs(f64(db[l]) - f64(db_e[l])) <= bound * s_db + 1e-30).all(), f"db[{l}]"
