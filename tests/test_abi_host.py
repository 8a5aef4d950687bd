"""Host-only checks of the C ABI: the library builds and loads, exports every
symbol the header declares, and rejects bad arguments before touching CUDA.

No call here reaches a kernel launch: every argument set is invalid, and the
library validates arguments before its first CUDA call.
"""
import ctypes
import os
import re

import pytest

import gemm_bias_activation_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coalesce.h")

FAKE = 0x7F0000000000  # 16-byte aligned; never dereferenced (the call fails validation first)


@pytest.fixture(scope="module")
def lib():
    g.build()
    return g.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coalesce_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(g.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_header_enums_match_binding():
    text = open(HEADER).read()
    vals = dict(re.findall(r"(COALESCE_\w+)\s*=\s*(-?\d+)", text))
    for name, v in vals.items():
        assert getattr(g, name) == int(v), name


def test_status_strings(lib):
    for st in [0, -1, -2, -3, -4, -5, 17]:
        s = g.coalesce_status_string(st)
        assert isinstance(s, str) and s
    assert g.coalesce_status_string(0) == "ok"


GEMM_OK = dict(M=64, N=64, K=64, dtype=g.COALESCE_BF16, A=FAKE, B=FAKE + (1 << 24), bias=FAKE + (2 << 24),
               Y=FAKE + (3 << 24), act=g.COALESCE_ACT_GELU_ERF, stream=None)


@pytest.mark.parametrize("change,expect", [
    (dict(M=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(N=-3), g.COALESCE_ERR_INVALID_ARG),
    (dict(K=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(dtype=7), g.COALESCE_ERR_INVALID_ARG),
    (dict(act=9), g.COALESCE_ERR_INVALID_ARG),
    (dict(act=-1), g.COALESCE_ERR_INVALID_ARG),
    (dict(A=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(B=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(Y=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(A=FAKE + 8), g.COALESCE_ERR_MISALIGNED),
    (dict(Y=FAKE + (3 << 24) + 2), g.COALESCE_ERR_MISALIGNED),
    (dict(bias=FAKE + (2 << 24) + 4), g.COALESCE_ERR_MISALIGNED),
    (dict(K=60), g.COALESCE_ERR_MISALIGNED),          # 60 * 2 B is not a multiple of 16
    (dict(N=100), g.COALESCE_ERR_MISALIGNED),
    (dict(dtype=g.COALESCE_F32, N=66), g.COALESCE_ERR_MISALIGNED),
    (dict(Y=FAKE + 64), g.COALESCE_ERR_INVALID_ARG),  # Y overlaps A
    (dict(M=1 << 31), g.COALESCE_ERR_UNSUPPORTED),
])
def test_gemm_rejects(lib, change, expect):
    a = dict(GEMM_OK, **change)
    st = g.coalesce_gemm_bias_act(a["M"], a["N"], a["K"], a["dtype"], a["A"], a["B"], a["bias"], a["Y"], a["act"],
                                  a["stream"])
    assert st == expect, (change, st, g.coalesce_last_error())


MLP_OK = dict(rows=256, D=128, H=128, L=3, x=FAKE, W=[FAKE + (1 << 24)] * 3, b=None, out=FAKE + (2 << 24),
              act=g.COALESCE_ACT_SOFTPLUS)


@pytest.mark.parametrize("change,expect", [
    (dict(rows=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(L=0, W=[]), g.COALESCE_ERR_INVALID_ARG),
    (dict(x=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(out=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(W=[FAKE, 0, FAKE]), g.COALESCE_ERR_INVALID_ARG),
    (dict(act=11), g.COALESCE_ERR_INVALID_ARG),
    (dict(D=100), g.COALESCE_ERR_MISALIGNED),              # rows of 200 bytes
    (dict(H=264), g.COALESCE_ERR_UNSUPPORTED),             # wider than 256
    (dict(H=512), g.COALESCE_ERR_UNSUPPORTED),
    (dict(L=9, W=[FAKE] * 9), g.COALESCE_ERR_UNSUPPORTED),   # at most 8 layers
    (dict(x=FAKE + 4), g.COALESCE_ERR_MISALIGNED),
    (dict(b=[FAKE + 2, None, None]), g.COALESCE_ERR_MISALIGNED),
    (dict(out=FAKE + 1024), g.COALESCE_ERR_INVALID_ARG),   # out overlaps x
])
def test_mlp_rejects(lib, change, expect):
    a = dict(MLP_OK, **change)
    st = g.coalesce_mlp_fused(a["rows"], a["D"], a["H"], a["L"], a["x"], a["W"], a["b"], a["out"], a["act"], None)
    assert st == expect, (change, st, g.coalesce_last_error())


def test_last_error_mentions_the_problem(lib):
    g.coalesce_gemm_bias_act(0, 1, 1, 0, FAKE, FAKE, None, FAKE, 0, None)
    assert "invalid argument" in g.coalesce_last_error()


def test_tensor_wrappers_fail_loudly_without_cuda():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    a = torch.zeros(8, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.gemm_bias_act(a, a)


@pytest.mark.parametrize("limit", [0, 999, 10_000_000_001])
def test_selftest_rejects_out_of_range_limits(lib, limit):
    assert g.coalesce_selftest_wait_timeout(limit, None) == g.COALESCE_ERR_INVALID_ARG


@pytest.mark.parametrize("iters,sink,flop", [(0, FAKE, True), (7, FAKE, True), (12, FAKE, True),
                                              ((1 << 40) + 8, FAKE, True), (8, 0, True), (8, FAKE, False)])
def test_measure_ffma_rejects(lib, iters, sink, flop):
    out = ctypes.c_double(-1.0)
    st = lib.coalesce_measure_ffma(iters, sink or None, ctypes.byref(out) if flop else None, None)
    assert st == g.COALESCE_ERR_INVALID_ARG
    assert out.value == -1.0


@pytest.mark.parametrize("args,expect", [
    ((0, 8, 0, FAKE, None, 0), g.COALESCE_ERR_INVALID_ARG),
    ((8, 8, 5, FAKE, None, 0), g.COALESCE_ERR_INVALID_ARG),
    ((8, 8, 0, 0, None, 0), g.COALESCE_ERR_INVALID_ARG),
    ((8, 8, 0, FAKE, None, 7), g.COALESCE_ERR_INVALID_ARG),
    ((8, 6, 0, FAKE, None, 0), g.COALESCE_ERR_MISALIGNED),
    ((8, 8, 2, FAKE + 8, None, 0), g.COALESCE_ERR_MISALIGNED),
    ((8, 8, 2, FAKE, FAKE + 16, 0), g.COALESCE_ERR_INVALID_ARG),  # bias overlaps Y
])
def test_bias_act_rejects(lib, args, expect):
    assert g.coalesce_bias_act(*args, None) == expect


MLPX_OK = dict(rows=256, D=128, H=128, O=64, L=3, dtype=g.COALESCE_BF16, x=FAKE, W=[FAKE + (1 << 24)] * 3, b=None,
               out=FAKE + (2 << 24), act=g.COALESCE_ACT_SOFTPLUS)


@pytest.mark.parametrize("change,expect", [
    (dict(O=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(dtype=5), g.COALESCE_ERR_INVALID_ARG),
    (dict(dtype=g.COALESCE_F32), g.COALESCE_ERR_UNSUPPORTED),
    (dict(O=100), g.COALESCE_ERR_MISALIGNED),
    (dict(D=4), g.COALESCE_ERR_MISALIGNED),
    (dict(O=320), g.COALESCE_ERR_UNSUPPORTED),
    (dict(H=320, O=256, D=128), g.COALESCE_ERR_UNSUPPORTED),       # hidden width over 256
    (dict(b=[FAKE, FAKE + 8, None]), g.COALESCE_ERR_MISALIGNED),
    (dict(out=FAKE + 4096), g.COALESCE_ERR_INVALID_ARG),        # out overlaps x
    (dict(W=[FAKE, None, FAKE]), g.COALESCE_ERR_INVALID_ARG),
])
def test_mlp_ex_rejects(lib, change, expect):
    a = dict(MLPX_OK, **change)
    st = g.coalesce_mlp_fused_ex(a["rows"], a["D"], a["H"], a["O"], a["L"], a["dtype"], a["x"], a["W"], a["b"],
                                 a["out"], a["act"], None)
    assert st == expect, (change, st, g.coalesce_last_error())


GEX_OK = dict(M=128, N=128, K=256, dtype=g.COALESCE_F16, flags=g.COALESCE_GEMM_TRANS_A, A=FAKE, B=FAKE + (1 << 24),
              bias=None, aux=None, Y=FAKE + (2 << 24), act=g.COALESCE_ACT_NONE)


@pytest.mark.parametrize("change,expect", [
    (dict(flags=16), g.COALESCE_ERR_INVALID_ARG),
    (dict(flags=g.COALESCE_GEMM_ACCUM_F32 | g.COALESCE_GEMM_DACT), g.COALESCE_ERR_INVALID_ARG),
    (dict(flags=g.COALESCE_GEMM_ACCUM_F32, act=g.COALESCE_ACT_RELU), g.COALESCE_ERR_INVALID_ARG),
    (dict(flags=g.COALESCE_GEMM_ACCUM_F32, bias=FAKE + (3 << 24)), g.COALESCE_ERR_INVALID_ARG),
    (dict(flags=g.COALESCE_GEMM_DACT), g.COALESCE_ERR_INVALID_ARG),                      # no aux
    (dict(aux=FAKE + (3 << 24)), g.COALESCE_ERR_INVALID_ARG),                           # aux without DACT
    (dict(dtype=g.COALESCE_F32), g.COALESCE_ERR_UNSUPPORTED),
    (dict(flags=g.COALESCE_GEMM_DACT, aux=FAKE + (3 << 24), act=g.COALESCE_ACT_GELU_ERF), g.COALESCE_ERR_UNSUPPORTED),
    (dict(M=100), g.COALESCE_ERR_MISALIGNED),           # TRANS_A: A's rows are M long
    (dict(flags=g.COALESCE_GEMM_TRANS_B, K=100), g.COALESCE_ERR_MISALIGNED),
    (dict(flags=g.COALESCE_GEMM_DACT, aux=FAKE + (2 << 24) + 64), g.COALESCE_ERR_INVALID_ARG),  # partial overlap
])
def test_gemm_ex_rejects(lib, change, expect):
    a = dict(GEX_OK, **change)
    st = g.coalesce_gemm_ex(a["M"], a["N"], a["K"], a["dtype"], a["flags"], a["A"], a["B"], a["bias"], a["aux"],
                            a["Y"], a["act"], None)
    assert st == expect, (change, st, g.coalesce_last_error())


TRAIN_OK = dict(rows=1024, D=64, H=64, O=64, L=3, dtype=g.COALESCE_F16, x=FAKE, W=[FAKE + (1 << 24)] * 3,
                h=[FAKE + (2 << 24), FAKE + (3 << 24)], dout=FAKE + (4 << 24), dx=FAKE + (5 << 24),
                dW=[FAKE + (6 << 24)] * 3, db=None, act=g.COALESCE_ACT_SOFTPLUS)


@pytest.mark.parametrize("change,expect", [
    (dict(rows=0), g.COALESCE_ERR_INVALID_ARG),
    (dict(act=g.COALESCE_ACT_GELU_ERF), g.COALESCE_ERR_UNSUPPORTED),
    (dict(dtype=g.COALESCE_F32), g.COALESCE_ERR_UNSUPPORTED),
    (dict(L=9, W=[FAKE] * 9, dW=[FAKE] * 9, h=[FAKE] * 8), g.COALESCE_ERR_UNSUPPORTED),
    (dict(H=60), g.COALESCE_ERR_MISALIGNED),
    (dict(dW=[FAKE, None, FAKE]), g.COALESCE_ERR_INVALID_ARG),
    (dict(dx=FAKE + 8), g.COALESCE_ERR_MISALIGNED),
    (dict(dx=FAKE + 4096), g.COALESCE_ERR_INVALID_ARG),   # dx overlaps x
])
def test_mlp_backward_rejects(lib, change, expect):
    a = dict(TRAIN_OK, **change)
    st = g.coalesce_mlp_backward(a["rows"], a["D"], a["H"], a["O"], a["L"], a["dtype"], a["x"], a["W"], a["h"],
                                 a["dout"], a["dx"], a["dW"], a["db"], a["act"], None)
    assert st == expect, (change, st, g.coalesce_last_error())


def test_mlp_forward_train_rejects_relu_free_gelu(lib):
    a = TRAIN_OK
    st = g.coalesce_mlp_forward_train(a["rows"], a["D"], a["H"], a["O"], a["L"], a["dtype"], a["x"], a["W"], None,
                                      a["h"], a["dout"], g.COALESCE_ACT_GELU_ERF, None)
    assert st == g.COALESCE_ERR_UNSUPPORTED


def test_last_error_is_per_thread(lib):
    """Each host thread reads the message of its own last rejected call."""
    import threading

    cases = [(dict(M=0), "must be >= 1"), (dict(act=11), "activation"), (dict(dtype=9), "dtype"), (dict(A=0), "NULL")]
    seen = {}
    barrier = threading.Barrier(len(cases))

    def worker(i, change):
        a = dict(GEMM_OK, **change)
        barrier.wait()
        for _ in range(200):
            st = g.coalesce_gemm_bias_act(a["M"], a["N"], a["K"], a["dtype"], a["A"], a["B"], a["bias"], a["Y"],
                                          a["act"], None)
            assert st == g.COALESCE_ERR_INVALID_ARG
        seen[i] = g.coalesce_last_error()

    ts = [threading.Thread(target=worker, args=(i, c)) for i, (c, _) in enumerate(cases)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for i, (_, word) in enumerate(cases):
        assert word in seen[i], (i, seen[i])
