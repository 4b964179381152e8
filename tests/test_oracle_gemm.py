"""Pins of the int4 x FP8 GEMM, the int4 packing, bf16 rounding and SiLU."""
import math
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import e4m3


def test_pack_order_hand_worked():
    # element k=0 -> bits 0-3, k=1 -> bits 4-7, two's complement
    assert oracle.pack_int4([[1, -2]]).tolist() == [[0xE1]]
    assert oracle.pack_int4([[-8, 7, 0, -1]]).tolist() == [[0x78, 0xF0]]
    assert oracle.unpack_int4(np.array([[0x78, 0xF0]], np.uint8)).tolist() == [[-8, 7, 0, -1]]


def test_pack_round_trip():
    v = np.random.default_rng(0).integers(-8, 8, size=(7, 256))
    assert np.array_equal(oracle.unpack_int4(oracle.pack_int4(v)), v)
    b = np.arange(256, dtype=np.uint8)[None, :]
    assert np.array_equal(oracle.pack_int4(oracle.unpack_int4(b)), b)


def _random_operands(rng, M, N, K):
    x = (rng.standard_normal((M, K)) * rng.uniform(0.1, 10, (M, 1))).astype(np.float32)
    aq, a_s = oracle.quant_per_token_group(x)
    w = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    ws = rng.uniform(0.005, 0.02, size=(N, K // 128)).astype(np.float32)
    return aq, a_s, w, ws


@pytest.mark.parametrize("M,N,K", [(1, 3, 128), (5, 7, 384), (16, 40, 1024)])
def test_grouped_form_equals_dense_dequantised_matmul(M, N, K):
    rng = np.random.default_rng(M * N + K)
    aq, a_s, w, ws = _random_operands(rng, M, N, K)
    y = oracle.w4a8_gemm(aq, a_s, w, ws)
    Af = oracle.dequant(aq, a_s)                                        # code * a_s
    Wf = w.astype(np.float64) * np.repeat(ws.astype(np.float64), 128, axis=1)  # int4 * w_s
    ref = Af @ Wf.T
    assert np.linalg.norm(y - ref) <= 1e-12 * np.linalg.norm(ref)


def test_brute_force_tiny():
    rng = np.random.default_rng(7)
    M, N, K = 2, 3, 256
    aq, a_s, w, ws = _random_operands(rng, M, N, K)
    y = oracle.w4a8_gemm(aq, a_s, w, ws)
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for g in range(K // 128):
                part = 0.0
                for kk in range(g * 128, (g + 1) * 128):
                    part += e4m3.DECODE_TABLE[aq[m, kk]] * int(w[n, kk])
                tot += float(a_s[m, g]) * float(ws[n, g]) * part
            assert abs(y[m, n] - tot) <= 1e-12 * max(1.0, abs(tot))


def test_integer_special_case_is_exact():
    # all scales 1, activation codes of small integers, weights in {-1, 0, 1}:
    # an integer matrix product, checked exactly with Python integers.
    rng = np.random.default_rng(11)
    M, N, K = 6, 9, 384
    a_int = rng.integers(-2, 3, size=(M, K))
    aq = e4m3.encode(a_int.astype(np.float32))
    a_s = np.ones((M, K // 128), np.float32)
    w = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    ws = np.ones((N, K // 128), np.float32)
    y = oracle.w4a8_gemm(aq, a_s, w, ws)
    for m in range(M):
        for n in range(N):
            assert y[m, n] == sum(int(a_int[m, kk]) * int(w[n, kk]) for kk in range(K))


def test_power_of_two_scales_are_exact():
    rng = np.random.default_rng(12)
    M, N, K = 3, 4, 256
    a_int = rng.integers(-7, 8, size=(M, K))
    aq = e4m3.encode(a_int.astype(np.float32))
    a_s = np.array([[2.0 ** -3, 2.0 ** 1]] * M, np.float32)
    w = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    ws = np.array([[2.0 ** -5, 2.0 ** -6]] * N, np.float32)
    y = oracle.w4a8_gemm(aq, a_s, w, ws)
    for m in range(M):
        for n in range(N):
            s0 = sum(int(a_int[m, kk]) * int(w[n, kk]) for kk in range(128))
            s1 = sum(int(a_int[m, kk]) * int(w[n, kk]) for kk in range(128, 256))
            assert y[m, n] == s0 * 2.0 ** -8 + s1 * 2.0 ** -5


def test_grouped_gemm_routes_rows_by_segment():
    rng = np.random.default_rng(13)
    K, N = 256, 8
    aq, a_s, _, _ = _random_operands(rng, 10, N, K)
    W = {e: rng.integers(-8, 8, size=(N, K)).astype(np.int8) for e in range(3)}
    S = {e: rng.uniform(0.005, 0.02, size=(N, 2)).astype(np.float32) for e in range(3)}
    seg = np.array([0, 4, 4, 10])
    y = oracle.grouped_gemm(aq, a_s, seg, W.__getitem__, S.__getitem__)
    assert np.array_equal(y[:4], oracle.w4a8_gemm(aq[:4], a_s[:4], W[0], S[0]))
    assert np.array_equal(y[4:], oracle.w4a8_gemm(aq[4:], a_s[4:], W[2], S[2]))


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(14)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000),
                        [0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3e-39, -2.5e-40]])
    ours = oracle.round_bf16(x)
    # torch rounds fp32 -> bf16; compare on values that are exact in fp32 first
    x32 = x.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x32).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x32), ref)
    # ties: 1 + 2**-8 is halfway between 1 and 1 + 2**-7 -> even (1.0); 1 + 3*2**-8 -> 1 + 2**-6
    assert ours[-4] == 1.0 and ours[-3] == 1.0 + 2.0 ** -6
    assert oracle.bf16_bits(np.array([1.0, -2.0])).tolist() == [0x3F80, 0xC000]


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(64.0) == 64.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(-64.0) + 64.0 * math.exp(-64.0)) < 1e-40
    assert oracle.silu(-1000.0) == 0.0
    x = np.random.default_rng(15).standard_normal(1000) * 8
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    assert np.allclose(oracle.silu(x), ref, rtol=1e-14, atol=1e-300)


def test_silu_mul_uses_gate_then_up():
    y = np.array([[64.0, 0.0, 3.0, 5.0]])  # I = 2: gate = [64, 0], up = [3, 5]
    assert oracle.silu_mul(y).tolist() == [[192.0, 0.0]]
