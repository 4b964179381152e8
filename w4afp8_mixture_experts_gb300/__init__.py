"""GB300 (sm_103a) W4AFP8 mixture-of-experts hot path: a C-ABI CUDA library and its binding.

int4 weights (fp32 scales per 128 along K) x FP8 E4M3 activations (per token
per 128 columns): routing, permutation, quantisation, grouped GEMMs, SiLU-and-Mul
requantisation, combine, and the dense W4AFP8 Linear.  See include/w4a8moe.h.
"""
from ._binding import (  # noqa: F401
    MoeLayout, W4A8Error, device_error, fp8_quant_per_token_group, fp8_quant_scatter_per_token_group,
    linear_split_k, linear_workspace_bytes, load,
    moe_permute, moe_permute_ep, moe_route_topk, moe_unpermute_combine, moe_workspace_layout, scale_ld,
    silu_mul_requant, w4a8_grouped_gemm, w4a8_grouped_gemm_silu, w4a8_linear, w4a8_moe_forward, w4a8_moe_forward_ep,
    w4a8_moe_forward_noalloc, w4a8_prepack_weights,
)
