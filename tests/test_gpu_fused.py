"""GPU parity of the w13 GEMM with SiLU-and-Mul requantisation fused into its epilogue.

The fused entry point computes, for 128-row tiles, gate and up blocks of the same 128 h-columns in one
CTA and requantises h = silu(gate) * up there; its codes, scales and corrections must equal the unfused
path's (the GEMM writing Y13, then the SiLU-and-Mul kernel) bit for bit, and the unfused path is the one
the stage tests pin to the oracle.  Also checked against the oracle's SiLU-and-Mul requantisation of the
oracle's Y13 within the requantisation gate (codes decided in fp32; exp may differ in the last bit).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bf16_from_bits, prepacked, rel_fro, scales_from_gpu_layout, to_dev
import inputs

pytestmark = pytest.mark.gpu


def _plan(lib, M, E, K):
    th = ctypes.c_int()
    return lib.load().w4a8_grouped_gemm_plan(M, E, K, ctypes.byref(th))


@pytest.mark.parametrize("counts,I,K", [
    ([300, 129, 0, 700, 61], 256, 1024),      # ragged chunks, an empty expert, a chunk of fewer than 64 rows
    ([1000, 1024, 999], 128, 512),             # two stages per tile, the smallest fused K
    ([513, 640], 512, 2048),
    ([257, 384, 300, 1], 256, 7168),          # an expert of one row in a wide plan
])
def test_fused_equals_unfused(lib, counts, I, K):
    rng = np.random.default_rng(sum(counts) + I + K)
    E = len(counts)
    seg = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(seg[-1])
    assert _plan(lib, M, E, K) == 2  # wide tiles only: the fused epilogue runs
    xb = inputs.to_bf16_bits((rng.standard_normal((M, K)) * rng.uniform(0.2, 5, (M, 1))).astype(np.float32))
    aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    packed = rng.integers(0, 256, size=(E, 2 * I, K // 2), dtype=np.uint8)
    ws = rng.uniform(0.005, 0.02, size=(E, K // 128, 2 * I)).astype(np.float32)
    B, bs, sg = prepacked(lib, packed), to_dev(ws), to_dev(seg)
    qf, sf, cf = lib.w4a8_grouped_gemm_silu(aq, a_s, a_c, B, bs, sg, fused=True)
    qu, su, cu = lib.w4a8_grouped_gemm_silu(aq, a_s, a_c, B, bs, sg, fused=False)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert torch.equal(qf, qu)
    assert torch.equal(sf[:, :M], su[:, :M]) and torch.equal(cf[:, :M], cu[:, :M])
    # the oracle: SiLU-and-Mul requantisation of its own bf16 Y13
    y13 = oracle.round_bf16(oracle.grouped_gemm(aq.cpu().numpy(), scales_from_gpu_layout(a_s, M), seg,
                                                lambda e: oracle.unpack_int4(packed[e]), lambda e: ws[e].T))
    rq, rs = oracle.silu_mul_requant(y13)
    got_q = qf.cpu().numpy()
    assert (got_q != rq).mean() <= 1e-3
    assert rel_fro(oracle.dequant(got_q, scales_from_gpu_layout(sf, M)), oracle.dequant(rq, rs)) <= 1e-3


def test_fused_entry_without_caller_corrections(lib):
    rng = np.random.default_rng(11)
    counts, I, K = [400, 300], 256, 1024
    E = len(counts)
    seg = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(seg[-1])
    xb = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    packed = rng.integers(0, 256, size=(E, 2 * I, K // 2), dtype=np.uint8)
    ws = rng.uniform(0.005, 0.02, size=(E, K // 128, 2 * I)).astype(np.float32)
    B, bs, sg = prepacked(lib, packed), to_dev(ws), to_dev(seg)
    q1, s1, c1 = lib.w4a8_grouped_gemm_silu(aq, a_s, a_c, B, bs, sg)
    q2, s2, c2 = lib.w4a8_grouped_gemm_silu(aq, a_s, None, B, bs, sg)
    assert torch.equal(q1, q2) and torch.equal(s1[:, :M], s2[:, :M]) and torch.equal(c1[:, :M], c2[:, :M])
    assert lib.device_error() == 0


def test_unfused_plan_takes_the_separate_kernels(lib):
    # a narrow-tile plan (few rows per expert): the entry point runs the GEMM and then the SiLU-and-Mul
    # kernel, with the same results as calling them one after the other
    rng = np.random.default_rng(5)
    counts, I, K = [3, 0, 9, 1, 16], 256, 512
    E = len(counts)
    seg = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M = int(seg[-1])
    assert _plan(lib, M, E, K) == 1
    xb = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    packed = rng.integers(0, 256, size=(E, 2 * I, K // 2), dtype=np.uint8)
    ws = rng.uniform(0.005, 0.02, size=(E, K // 128, 2 * I)).astype(np.float32)
    B, bs, sg = prepacked(lib, packed), to_dev(ws), to_dev(seg)
    q, s, c = lib.w4a8_grouped_gemm_silu(aq, a_s, a_c, B, bs, sg)
    y13 = lib.w4a8_grouped_gemm(aq, a_s, a_c, B, bs, sg)
    q2, s2, c2 = lib.silu_mul_requant(y13)
    assert torch.equal(q, q2) and torch.equal(s[:, :M], s2[:, :M]) and torch.equal(c[:, :M], c2[:, :M])
