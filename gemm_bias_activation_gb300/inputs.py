"""Seeded synthetic inputs for the GEMM + bias + activation and chained-MLP workloads.

This module only draws random numbers and rounds them to the storage dtype
(round-to-nearest-even, exactly what ``Tensor.to`` does).  It holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can be fed the
same bits from it.

Recipe (every tensor gets its own generator seeded from (seed, tensor id)):

* FP32 GEMM workloads: A[M, K], B[K, N], bias[N] ~ U(-1, 1), drawn in fp32.
* bf16 FFN up-projection: X[M, K] ~ N(0, 1), W[K, N] ~ N(0, 1/K) and
  bias[N] ~ N(0, 0.02), where the second argument of N(., .) is the VARIANCE
  (1/K makes the pre-activation unit variance only as a variance), drawn in
  fp32 and rounded to bf16.
* fp16 chained MLP: x[rows, D] ~ N(0, 1), W_l ~ N(0, 1/H) (variance) and
  b_l ~ N(0, 0.01) (variance) or b_l = 0, drawn in fp32 and rounded to fp16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Tuple

import torch

_TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def _gen(seed: int, tensor_id: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed((seed * 1_000_003 + tensor_id * 7919 + 17) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def uniform(shape, seed: int, tensor_id: int, dtype: str, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    """U(lo, hi) drawn in fp32, rounded RNE to ``dtype``."""
    t = torch.rand(shape, generator=_gen(seed, tensor_id), dtype=torch.float32)
    t.mul_(hi - lo).add_(lo)
    return t.to(torch_dtype(dtype))


def normal(shape, seed: int, tensor_id: int, dtype: str, variance: float = 1.0) -> torch.Tensor:
    """N(0, variance) drawn in fp32, rounded RNE to ``dtype``."""
    t = torch.randn(shape, generator=_gen(seed, tensor_id), dtype=torch.float32)
    if variance != 1.0:
        t.mul_(math.sqrt(variance))
    return t.to(torch_dtype(dtype))


def integer_pattern(shape, mult: int, mod: int, dtype: str) -> torch.Tensor:
    """Small-integer test pattern value[i] = (i * mult) % mod over the flat index.

    The "Coalesce" README (Notes for future sessions) uses (i*7)%13 and
    (i*3)%11 so that a transposed or shifted index shows up as a wrong value
    (A = 1, B = 1 would hide it).  Used unscaled, products and sums stay small
    integers that fp32 accumulates exactly, so a GEMM on them is bit-exact.
    """
    n = 1
    for s in shape:
        n *= s
    idx = torch.arange(n, dtype=torch.int64)
    return ((idx * mult) % mod).to(torch.float32).reshape(shape).to(torch_dtype(dtype))


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class GemmWorkload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # "f32" | "f16" | "bf16" (A, B, bias and Y share it)
    act: str            # "none" | "relu" | "gelu_erf" | "softplus"
    dist: str           # "uniform" | "ffn"
    bias_variance: float = 0.02

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def bytes_moved(self) -> float:
        """Algorithmic HBM bytes: read A, B, bias once, write Y once."""
        e = 4 if self.dtype == "f32" else 2
        return float(e * (self.M * self.K + self.K * self.N + self.N + self.M * self.N))


@dataclasses.dataclass(frozen=True)
class MlpWorkload:
    name: str
    rows: int
    D: int
    H: int
    L: int
    dtype: str                    # "f16" | "bf16"
    w_variance: float
    b_variance: Optional[float]   # None means b_l = 0
    act: str = "softplus"
    O: Optional[int] = None       # output width of the last layer; None means H
    train: bool = False           # a training step: forward with stored activations + backward

    @property
    def out_width(self) -> int:
        return self.H if self.O is None else self.O

    def layer_shapes(self) -> List[Tuple[int, int]]:
        """[in, out] of each W_l: D -> H -> ... -> H -> out_width."""
        return [(self.D if l == 0 else self.H, self.out_width if l == self.L - 1 else self.H) for l in range(self.L)]

    def flops(self) -> float:
        return 2.0 * self.rows * sum(k * n for k, n in self.layer_shapes())

    def bytes_moved(self) -> float:
        """Algorithmic HBM bytes: x in, out once; weights and biases once."""
        e = 2
        w = sum(k * n + n for k, n in self.layer_shapes())
        return float(e * (self.rows * self.D + self.rows * self.out_width + w))

    def train_bytes_moved(self) -> float:
        """Algorithmic HBM bytes of one training step, each tensor moved once:
        the forward reads x and writes every stored activation and the output;
        the backward reads dout, every stored activation and x, and writes dx
        (the fused backward keeps every data gradient on chip).  Weights,
        biases and their gradients are negligible and left out."""
        e, r = 2, self.rows
        fwd = self.D + (self.L - 1) * self.H + self.out_width
        bwd = self.out_width + (self.L - 1) * self.H + self.D + self.D
        return float(e * r * (fwd + bwd))

    def train_flops(self) -> float:
        """Forward GEMMs plus the two backward GEMMs (dW and the data gradient) per layer."""
        return 3.0 * self.flops()


WORKLOADS = {
    w.name: w
    for w in [
        GemmWorkload("fp32_gemm_bias_gelu_256", 256, 256, 256, "f32", "gelu_erf", "uniform"),
        GemmWorkload("fp32_gemm_bias_gelu_512", 512, 512, 512, "f32", "gelu_erf", "uniform"),
        GemmWorkload("fp32_gemm_bias_gelu_1024", 1024, 1024, 1024, "f32", "gelu_erf", "uniform"),
        GemmWorkload("fp32_gemm_bias_gelu_2048", 2048, 2048, 2048, "f32", "gelu_erf", "uniform"),
        GemmWorkload("fp32_gemm_bias_gelu_4096", 4096, 4096, 4096, "f32", "gelu_erf", "uniform"),
        GemmWorkload("bf16_ffn_up_bias_gelu_16384x16384x4096", 16384, 16384, 4096, "bf16", "gelu_erf", "ffn"),
        MlpWorkload("fp16_mlp3_softplus_128w_2p20rows", 1 << 20, 128, 128, 3, "f16", 1.0 / 128, 0.01),
        MlpWorkload("fp16_mlp5_softplus_64w_2p22rows", 1 << 22, 64, 64, 5, "f16", 1.0 / 64, None),
        MlpWorkload("fp16_mlp3_softplus_128w_2p20rows_train", 1 << 20, 128, 128, 3, "f16", 1.0 / 128, 0.01,
                    train=True),
    ]
}


def gemm_inputs(w: GemmWorkload, seed: int = 0, M: Optional[int] = None, N: Optional[int] = None,
                K: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(A, B, bias) on the CPU for workload ``w`` (optionally at another shape)."""
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    if w.dist == "uniform":
        A = uniform((M, K), seed, 1, w.dtype)
        B = uniform((K, N), seed, 2, w.dtype)
        bias = uniform((N,), seed, 3, w.dtype)
    elif w.dist == "ffn":
        A = normal((M, K), seed, 1, w.dtype, 1.0)
        B = normal((K, N), seed, 2, w.dtype, 1.0 / K)
        bias = normal((N,), seed, 3, w.dtype, w.bias_variance)
    else:
        raise ValueError(w.dist)
    return A, B, bias


def mlp_inputs(w: MlpWorkload, seed: int = 0, rows: Optional[int] = None
               ) -> Tuple[torch.Tensor, List[torch.Tensor], List[Optional[torch.Tensor]]]:
    """(x, [W_l], [b_l]) on the CPU for MLP workload ``w``; W_l is [in, out]."""
    rows = w.rows if rows is None else rows
    x = normal((rows, w.D), seed, 1, w.dtype, 1.0)
    Ws, bs = [], []
    for l, (fan_in, fan_out) in enumerate(w.layer_shapes()):
        Ws.append(normal((fan_in, fan_out), seed, 10 + l, w.dtype, w.w_variance))
        if w.b_variance is None:
            bs.append(torch.zeros(fan_out, dtype=torch_dtype(w.dtype)))
        else:
            bs.append(normal((fan_out,), seed, 30 + l, w.dtype, w.b_variance))
    return x, Ws, bs
