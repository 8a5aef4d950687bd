"""fp64 CPU oracle for the fused GEMM + bias + activation and the chained MLP.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.
"""
from .reference import (  # noqa: F401
    ACTS,
    act_derivative,
    act_derivative_from_output,
    act_gelu_erf,
    act_none,
    act_relu,
    act_softplus,
    apply_act,
    gemm_bias_act,
    gemm_bias_act_fused_loops,
    gemm_bias_act_rows,
    mlp_chain,
    mlp_chain_fp16_mirror,
    mlp_chain_rows,
    mlp_backward,
    mlp_backward_from_activations,
    mlp_forward_train,
)
