"""GB300 (sm_103a) fused GEMM + bias + activation and chained MLP.

A thin Python binding over the C ABI of ``libcoalesce.so`` (``include/coalesce.h``).
The functions named like the C entry points marshal arguments and call them;
every step of the computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams only.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from ._build import LIB_PATH, build  # noqa: F401

# Enumerations mirrored from include/coalesce.h
COALESCE_F32, COALESCE_F16, COALESCE_BF16 = 0, 1, 2
COALESCE_ACT_NONE, COALESCE_ACT_RELU, COALESCE_ACT_GELU_ERF, COALESCE_ACT_SOFTPLUS = 0, 1, 2, 3
COALESCE_OK = 0
COALESCE_ERR_INVALID_ARG = -1
COALESCE_ERR_UNSUPPORTED = -2
COALESCE_ERR_MISALIGNED = -3
COALESCE_ERR_CUDA = -4
COALESCE_ERR_DEVICE_TIMEOUT = -5
COALESCE_GEMM_TRANS_A, COALESCE_GEMM_TRANS_B, COALESCE_GEMM_ACCUM_F32, COALESCE_GEMM_DACT = 1, 2, 4, 8

ACT_CODES = {"none": COALESCE_ACT_NONE, "relu": COALESCE_ACT_RELU, "gelu_erf": COALESCE_ACT_GELU_ERF,
             "softplus": COALESCE_ACT_SOFTPLUS}

# Every symbol include/coalesce.h declares.
EXPORTED_SYMBOLS = (
    "coalesce_gemm_bias_act",
    "coalesce_gemm_ex",
    "coalesce_mlp_forward_train",
    "coalesce_mlp_backward",
    "coalesce_bias_act",
    "coalesce_mlp_fused",
    "coalesce_mlp_fused_ex",
    "coalesce_device_status",
    "coalesce_selftest_wait_timeout",
    "coalesce_measure_ffma",
    "coalesce_status_string",
    "coalesce_last_error",
    "coalesce_shutdown",
)


class CoalesceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib_or_none()
        text = lib.coalesce_status_string(status).decode() if lib else str(status)
        detail = lib.coalesce_last_error().decode() if lib else ""
        super().__init__(f"{where}: {text} ({status}): {detail}")


_LIB: Optional[ctypes.CDLL] = None


def _lib_or_none() -> Optional[ctypes.CDLL]:
    return _LIB


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcoalesce.so (built by ``build()``); raise if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with gemm_bias_activation_gb300.build()")
    L = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    L.coalesce_gemm_bias_act.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, i32, vp]
    L.coalesce_gemm_bias_act.restype = i32
    L.coalesce_gemm_ex.argtypes = [i64, i64, i64, i32, ctypes.c_uint, vp, vp, vp, vp, vp, i32, vp]
    L.coalesce_gemm_ex.restype = i32
    pp = ctypes.POINTER(vp)
    L.coalesce_mlp_forward_train.argtypes = [i64, i64, i64, i64, i32, i32, vp, pp, pp, pp, vp, i32, vp]
    L.coalesce_mlp_forward_train.restype = i32
    L.coalesce_mlp_backward.argtypes = [i64, i64, i64, i64, i32, i32, vp, pp, pp, vp, vp, pp, pp, i32, vp]
    L.coalesce_mlp_backward.restype = i32
    L.coalesce_bias_act.argtypes = [i64, i64, i32, vp, vp, i32, vp]
    L.coalesce_bias_act.restype = i32
    L.coalesce_mlp_fused.argtypes = [i64, i64, i64, i32, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, i32, vp]
    L.coalesce_mlp_fused.restype = i32
    L.coalesce_mlp_fused_ex.argtypes = [i64, i64, i64, i64, i32, i32, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                                        i32, vp]
    L.coalesce_mlp_fused_ex.restype = i32
    L.coalesce_device_status.argtypes = [vp]
    L.coalesce_device_status.restype = i32
    L.coalesce_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    L.coalesce_selftest_wait_timeout.restype = i32
    L.coalesce_measure_ffma.argtypes = [i64, vp, ctypes.POINTER(ctypes.c_double), vp]
    L.coalesce_measure_ffma.restype = i32
    L.coalesce_status_string.argtypes = [i32]
    L.coalesce_status_string.restype = ctypes.c_char_p
    L.coalesce_last_error.argtypes = []
    L.coalesce_last_error.restype = ctypes.c_char_p
    L.coalesce_shutdown.argtypes = []
    L.coalesce_shutdown.restype = None
    _LIB = L
    return L


# --------------------------------------------------------------------------
# Raw C-ABI calls (same names and argument order as include/coalesce.h).
# Pointers are integers (device addresses); `stream` is a cudaStream_t as int.
# --------------------------------------------------------------------------
def coalesce_gemm_bias_act(M: int, N: int, K: int, dtype: int, A: int, B: int, bias: Optional[int], Y: int,
                           act: int, stream: Optional[int]) -> int:
    return load_library().coalesce_gemm_bias_act(M, N, K, dtype, A, B, bias or None, Y, act, stream or None)


def coalesce_gemm_ex(M: int, N: int, K: int, dtype: int, flags: int, A: int, B: int, bias: Optional[int],
                     aux: Optional[int], Y: int, act: int, stream: Optional[int]) -> int:
    return load_library().coalesce_gemm_ex(M, N, K, dtype, flags, A, B, bias or None, aux or None, Y, act,
                                           stream or None)


def _ptr_array(ptrs: Optional[Sequence[Optional[int]]], n: int):
    return None if ptrs is None else (ctypes.c_void_p * n)(*[p or None for p in ptrs])


def coalesce_mlp_forward_train(rows: int, D: int, H: int, O: int, L: int, dtype: int, x: int, W: Sequence[int],
                               b: Optional[Sequence[Optional[int]]], h: Sequence[int], out: int, act: int,
                               stream: Optional[int]) -> int:
    return load_library().coalesce_mlp_forward_train(rows, D, H, O, L, dtype, x, _ptr_array(W, L), _ptr_array(b, L),
                                                     _ptr_array(h, max(L - 1, 1)), out, act, stream or None)


def coalesce_mlp_backward(rows: int, D: int, H: int, O: int, L: int, dtype: int, x: int, W: Sequence[int],
                          h: Sequence[int], dout: int, dx: Optional[int], dW: Sequence[int],
                          db: Optional[Sequence[Optional[int]]], act: int, stream: Optional[int]) -> int:
    return load_library().coalesce_mlp_backward(rows, D, H, O, L, dtype, x, _ptr_array(W, L),
                                                _ptr_array(h, max(L - 1, 1)), dout, dx or None, _ptr_array(dW, L),
                                                _ptr_array(db, L), act, stream or None)


def coalesce_bias_act(M: int, N: int, dtype: int, Y: int, bias: Optional[int], act: int,
                      stream: Optional[int]) -> int:
    return load_library().coalesce_bias_act(M, N, dtype, Y, bias or None, act, stream or None)


def coalesce_mlp_fused(rows: int, D: int, H: int, L: int, x: int, W: Sequence[int],
                       b: Optional[Sequence[Optional[int]]], out: int, act: int, stream: Optional[int]) -> int:
    wa = (ctypes.c_void_p * L)(*W)
    ba = None if b is None else (ctypes.c_void_p * L)(*[p or None for p in b])
    return load_library().coalesce_mlp_fused(rows, D, H, L, x, wa, ba, out, act, stream or None)


def coalesce_mlp_fused_ex(rows: int, D: int, H: int, O: int, L: int, dtype: int, x: int, W: Sequence[int],
                          b: Optional[Sequence[Optional[int]]], out: int, act: int, stream: Optional[int]) -> int:
    wa = (ctypes.c_void_p * L)(*W)
    ba = None if b is None else (ctypes.c_void_p * L)(*[p or None for p in b])
    return load_library().coalesce_mlp_fused_ex(rows, D, H, O, L, dtype, x, wa, ba, out, act, stream or None)


def coalesce_device_status(stream: Optional[int]) -> int:
    return load_library().coalesce_device_status(stream or None)


def coalesce_selftest_wait_timeout(limit_ns: int, stream: Optional[int]) -> int:
    return load_library().coalesce_selftest_wait_timeout(limit_ns, stream or None)


def coalesce_status_string(status: int) -> str:
    return load_library().coalesce_status_string(status).decode()


def coalesce_last_error() -> str:
    return load_library().coalesce_last_error().decode()


def coalesce_shutdown() -> None:
    load_library().coalesce_shutdown()


# --------------------------------------------------------------------------
# Tensor conveniences (argument marshalling only).
# --------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch

    codes = {torch.float32: COALESCE_F32, torch.float16: COALESCE_F16, torch.bfloat16: COALESCE_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _check(status: int, where: str) -> None:
    if status != COALESCE_OK:
        raise CoalesceError(status, where)


def _stream_handle(stream) -> int:
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def gemm_bias_act(A, B, bias=None, act: str = "gelu_erf", out=None, stream=None):
    """Y = act(A @ B + bias) through coalesce_gemm_bias_act; A[M,K], B[K,N] contiguous CUDA tensors."""
    import torch

    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous (row-major)")
    M, K = A.shape
    K2, N = B.shape
    if K != K2 or A.dtype != B.dtype or (bias is not None and (bias.dtype != A.dtype or bias.numel() != N)):
        raise ValueError("shape or dtype mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=A.dtype, device=A.device)
    st = coalesce_gemm_bias_act(M, N, K, _dtype_code(A), A.data_ptr(), B.data_ptr(),
                                None if bias is None else bias.data_ptr(), out.data_ptr(), ACT_CODES[act],
                                _stream_handle(stream))
    _check(st, "coalesce_gemm_bias_act")
    return out


def gemm_then_bias_act(A, B, bias=None, act: str = "gelu_erf", out=None, stream=None):  # noqa: D401
    """The UNFUSED sequence: GEMM without bias or activation, then the separate
    in-place bias + activation pass (coalesce_bias_act).  For fusion studies."""
    Y = gemm_bias_act(A, B, None, "none", out=out, stream=stream)
    M, N = Y.shape
    st = coalesce_bias_act(M, N, _dtype_code(Y), Y.data_ptr(), None if bias is None else bias.data_ptr(),
                           ACT_CODES[act], _stream_handle(stream))
    _check(st, "coalesce_bias_act")
    return Y


def mlp_fused(x, Ws, bs=None, act: str = "softplus", out=None, stream=None):
    """Chained MLP through coalesce_mlp_fused_ex.

    x[rows, D], W_l [in, out] (D -> H -> ... -> H -> O), b_l [out_l] or None;
    all fp16 or all bf16, contiguous CUDA tensors.  Returns out[rows, O].
    """
    import torch

    rows, D = x.shape
    L = len(Ws)
    H = Ws[0].shape[1] if L > 1 else Ws[-1].shape[1]  # no hidden layer when L = 1
    O = Ws[-1].shape[1]
    if out is None:
        out = torch.empty((rows, O), dtype=x.dtype, device=x.device)
    st = coalesce_mlp_fused_ex(rows, D, H, O, L, _dtype_code(x), x.data_ptr(), [w.data_ptr() for w in Ws],
                               None if bs is None else [None if b is None else b.data_ptr() for b in bs],
                               out.data_ptr(), ACT_CODES[act], _stream_handle(stream))
    _check(st, "coalesce_mlp_fused_ex")
    return out


def mlp_forward_train(x, Ws, bs=None, act: str = "softplus", hs=None, out=None, stream=None):
    """Training forward through coalesce_mlp_forward_train: returns (out, hs),
    hs the L-1 stored activations [rows, H] (pass them to mlp_backward)."""
    import torch

    rows, D = x.shape
    L = len(Ws)
    H = Ws[0].shape[1] if L > 1 else Ws[-1].shape[1]
    O = Ws[-1].shape[1]
    if hs is None:
        hs = [torch.empty((rows, H), dtype=x.dtype, device=x.device) for _ in range(L - 1)]
    if out is None:
        out = torch.empty((rows, O), dtype=x.dtype, device=x.device)
    st = coalesce_mlp_forward_train(rows, D, H, O, L, _dtype_code(x), x.data_ptr(), [w.data_ptr() for w in Ws],
                                    None if bs is None else [None if b is None else b.data_ptr() for b in bs],
                                    [h.data_ptr() for h in hs], out.data_ptr(), ACT_CODES[act], _stream_handle(stream))
    _check(st, "coalesce_mlp_forward_train")
    return out, hs


def mlp_backward(x, Ws, hs, dout, act: str = "softplus", want_dx: bool = True, want_db: bool = True, dW=None,
                 db=None, dx=None, stream=None):
    """Backward through coalesce_mlp_backward: returns (dx, [dW_l], [db_l]) with
    dW_l, db_l fp32; consumes hs (overwritten with gradients)."""
    import torch

    rows, D = x.shape
    L = len(Ws)
    H = Ws[0].shape[1] if L > 1 else Ws[-1].shape[1]
    O = Ws[-1].shape[1]
    if dW is None:
        dW = [torch.empty(w.shape, dtype=torch.float32, device=x.device) for w in Ws]
    if want_db and db is None:
        db = [torch.empty((w.shape[1],), dtype=torch.float32, device=x.device) for w in Ws]
    if want_dx and dx is None:
        dx = torch.empty_like(x)
    st = coalesce_mlp_backward(rows, D, H, O, L, _dtype_code(x), x.data_ptr(), [w.data_ptr() for w in Ws],
                               [h.data_ptr() for h in hs], dout.data_ptr(), dx.data_ptr() if want_dx else None,
                               [t.data_ptr() for t in dW], [t.data_ptr() for t in db] if want_db else None,
                               ACT_CODES[act], _stream_handle(stream))
    _check(st, "coalesce_mlp_backward")
    return (dx if want_dx else None), dW, (db if want_db else None)


def device_status(stream=None) -> None:
    """Synchronise and raise if a kernel's bounded wait ran out."""
    _check(coalesce_device_status(_stream_handle(stream)), "coalesce_device_status")
