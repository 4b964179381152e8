"""CPU oracle of the W4AFP8 MoE hot path (numpy, float64).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py, never by the CUDA library or its Python binding.
See oracle/moe.py for the definition of every step and its citation.
"""
from . import e4m3  # noqa: F401
from .moe import (  # noqa: F401
    GROUP, bf16_bits, bf16_value, dequant, grouped_gemm, linear, moe_layer, moe_tokens,
    pack_int4, permute, quant_per_token_group, round_bf16, route_topk, silu, silu_mul,
    silu_mul_requant, unpack_int4, unpermute_combine, w4a8_gemm,
)
