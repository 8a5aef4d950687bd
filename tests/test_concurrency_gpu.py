"""Concurrent use of the C ABI: several host threads, each with its own CUDA
stream, call the GEMM and the chained MLP at once.  The library keeps no
per-call global state besides the bounded-wait error word, so every result
must equal, bit for bit, the same call made alone (both kernels are
deterministic: no atomics, a fixed summation order)."""
import threading

import pytest
import torch

import gemm_bias_activation_gb300 as g
from gemm_bias_activation_gb300 import inputs

pytestmark = pytest.mark.gpu

THREADS = 4
CALLS = 12


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    g.build()
    g.load_library()
    torch.cuda.set_device(0)


def _gemm_case(i):
    """Even threads: a GEMM of one CTA per tile; odd threads: one large
    enough for the CTA-pair kernel (cluster launches from several streams)."""
    w = inputs.WORKLOADS["bf16_ffn_up_bias_gelu_16384x16384x4096"]
    if i % 2:
        A, B, bias = inputs.gemm_inputs(w, seed=100 + i, M=4096 + 256 * i, N=4864, K=64)
    else:
        A, B, bias = inputs.gemm_inputs(w, seed=100 + i, M=1000 + 37 * i, N=520, K=264)
    return A.cuda(), B.cuda(), bias.cuda()


def _mlp_case(i):
    w = inputs.WORKLOADS["fp16_mlp3_softplus_128w_2p20rows"]
    x, Ws, bs = inputs.mlp_inputs(w, seed=200 + i, rows=3000 + 129 * i)
    return x.cuda(), [t.cuda() for t in Ws], [t.cuda() for t in bs]


def test_threads_and_streams_give_the_single_call_bits():
    gemms = [_gemm_case(i) for i in range(THREADS)]
    mlps = [_mlp_case(i) for i in range(THREADS)]
    want_y = [g.gemm_bias_act(A, B, bias, "gelu_erf") for A, B, bias in gemms]
    want_o = [g.mlp_fused(x, Ws, bs) for x, Ws, bs in mlps]
    torch.cuda.synchronize()
    got = [None] * THREADS
    errors = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            A, B, bias = gemms[i]
            x, Ws, bs = mlps[i]
            with torch.cuda.stream(s):
                ys = [torch.empty((A.shape[0], B.shape[1]), dtype=A.dtype, device="cuda") for _ in range(CALLS)]
                os_ = [torch.empty((x.shape[0], Ws[-1].shape[1]), dtype=x.dtype, device="cuda") for _ in range(CALLS)]
                start.wait()
                for c in range(CALLS):
                    g.gemm_bias_act(A, B, bias, "gelu_erf", out=ys[c], stream=s)
                    g.mlp_fused(x, Ws, bs, out=os_[c], stream=s)
            s.synchronize()
            got[i] = (ys, os_)
        except Exception as e:  # reported by the main thread
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    g.device_status()
    for i in range(THREADS):
        ys, os_ = got[i]
        for c in range(CALLS):
            assert torch.equal(ys[c], want_y[i]), (i, c)
            assert torch.equal(os_[c], want_o[i]), (i, c)
