"""GB300 (sm_103a) unified-precision FP8 linear layer.

The compute lives in the C-ABI library ``libjetfp8.so`` (``include/jet_fp8.h``),
built in-tree from ``csrc/`` by ``build.build()``.  ``binding`` is a thin
ctypes layer over it; ``workloads`` draws the seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    JetError,
    device_status,
    gemm_fp8_dgrad,
    gemm_fp8_fwd,
    gemm_fp8_fwd_grouped,
    gemm_fp8_wgrad,
    jet_gemm_fp8_dgrad,
    jet_gemm_fp8_fwd,
    jet_gemm_fp8_fwd_grouped,
    jet_gemm_fp8_wgrad,
    jet_quant_act_1x128,
    jet_quant_dual_1x128_128x1,
    jet_quant_w_128x128,
    jet_requant_128x1,
    jet_swiglu_quant_1x128,
    jet_token_mismatch_masked,
    jet_token_mult_prob_error,
    load,
    quant_act_1x128,
    quant_dual_1x128_128x1,
    quant_w_128x128,
    requant_128x1,
    selftest_bounded_wait,
    selftest_quotient,
    swiglu_quant_1x128,
    token_mismatch_masked,
    token_mult_prob_error,
    workspace_bytes,
)
