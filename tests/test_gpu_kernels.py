"""GPU parity of the routing, permutation, quantisation, SiLU-requant and combine kernels.

Each kernel runs through the C ABI (the Python binding only marshals) and is
compared element by element with the CPU oracle on the same seeded inputs.
"""
import random

import numpy as np
import pytest
import torch

import inputs
import oracle
from gpu_util import (bf16_from_bits, bf16_ulp_diff, bits_of_bf16, decode_prepacked, f64_of_bf16, rel_fro,
                      scales_from_gpu_layout, to_dev)

pytestmark = pytest.mark.gpu


def test_generator_twin_is_bit_exact(lib):
    for seed, stream, start, n in [(0, 1, 0, 4099), (3, 2, 12345, 1000), (7, 4, 1 << 33, 517)]:
        g = inputs.gpu_packed_int4(seed, stream, (n,), start=start).cpu().numpy()
        assert np.array_equal(g, inputs.packed_int4(seed, stream, start, n))
        s = inputs.gpu_scales(seed, stream, (n,), start=start).cpu().numpy()
        assert np.array_equal(s, inputs.scales(seed, stream, start, n))


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (333, 8, 2), (64, 256, 8), (257, 384, 8), (40, 1000, 32),
                                   (17, 5, 5), (9, 33, 1)])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk(lib, T, E, k, renorm):
    rng = np.random.default_rng(T * 1000 + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, : min(E, 6)] = lg[0, 0]  # ties
    if T > 3:
        lg[3] = np.round(lg[3])    # many ties
    ids, w = lib.moe_route_topk(to_dev(lg), k, renorm)
    rid, rw = oracle.route_topk(lg, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    got = w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - rw) / np.abs(rw)) <= 1e-6


def _distinct_ids(rng, T, E, k, skew=None):
    ids = np.empty((T, k), np.int32)
    for t in range(T):
        if skew is not None:
            p = skew / skew.sum()
            ids[t] = rng.choice(E, size=k, replace=False, p=p)
        else:
            ids[t] = rng.choice(E, size=k, replace=False)
    return ids


# from 8192 pairs the permutation runs over several CTAs (count pass + placement pass)
@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 8, 2), (64, 256, 8), (1000, 384, 8), (4096, 16, 4),
                                   (2049, 1024, 3), (1024, 256, 8), (8192, 256, 8), (4096, 1024, 8),
                                   (3001, 7, 3)])
def test_permute(lib, T, E, k):
    rng = np.random.default_rng(T + E + k)
    ids = _distinct_ids(rng, T, E, k)
    seg, s2d, d2s = lib.moe_permute(to_dev(ids), E)
    rs, rs2d, rd2s = oracle.permute(ids, E)
    assert np.array_equal(seg.cpu().numpy(), rs)
    assert np.array_equal(s2d.cpu().numpy(), rs2d)
    assert np.array_equal(d2s.cpu().numpy(), rd2s)


def test_permute_skewed_and_empty(lib):
    rng = np.random.default_rng(5)
    E = 64
    skew = np.zeros(E)
    skew[[3, 7, 8, 40, 41, 42, 63]] = [100, 1, 1, 5, 5, 5, 30]
    ids = _distinct_ids(rng, 3000, E, 4, skew)
    seg, s2d, d2s = lib.moe_permute(to_dev(ids), E)
    rs, rs2d, rd2s = oracle.permute(ids, E)
    assert np.array_equal(seg.cpu().numpy(), rs)
    assert np.array_equal(s2d.cpu().numpy(), rs2d)
    assert np.array_equal(d2s.cpu().numpy(), rd2s)


def _bf16_rows(rng, M, K):
    x = rng.standard_normal((M, K)).astype(np.float32) * rng.uniform(0.01, 30, (M, 1)).astype(np.float32)
    if M > 2:
        x[1] = 0.0                              # all-zero row
        x[2, 5] = 3.0e4                         # a spike
    if M > 4:
        x[4, :] = np.float32(1e-30)             # tiny values
    if M > 6:
        x[5, 7] = 3.0e38                        # near the bf16 maximum: scale ~7e35
        x[6, 0::2] = -0.0                       # signed zeros: codes 0x80 / 0x00
        x[6, 1::2] = 0.0
    return inputs.to_bf16_bits(x)


# 1200 x 7168 has more than 65536 groups: the four-lanes-per-group kernel (sixteen below that)
@pytest.mark.parametrize("M,K", [(1, 128), (37, 256), (300, 7168), (1024, 2048), (1200, 7168)])
def test_quant(lib, M, K):
    rng = np.random.default_rng(M + K)
    xb = _bf16_rows(rng, M, K)
    q, s, c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    rq, rs = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(xb))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(scales_from_gpu_layout(s, M), rs)
    _check_gcorr(scales_from_gpu_layout(c, M), rq, rs)


def _check_gcorr(gc, codes, scales):
    # -1/2 * scale * S with S the exact sum of the group's E4M3 values, rounded once to fp32, then one
    # fp32 product: bit for bit
    M, K = codes.shape
    S = oracle.e4m3.decode(codes).reshape(M, K // 128, 128).sum(axis=2)
    ref = (np.float32(-0.5) * (scales.astype(np.float32) * S.astype(np.float32))).astype(np.float32)
    assert np.array_equal(gc, ref)


def test_gcorr_sum_is_exact_past_the_fp32_grid(lib):
    # Groups whose code sum passes 2^15 while holding values on the 2^-9 grid: a running fp32 sum would
    # round there, the exact sum must not (the correction is rounded once, at the end).
    K = 256
    x = np.zeros((4, K), np.float32)
    x[:, :100] = 1.0                                  # codes 448 (0x7E)
    x[:, 100:128] = np.float32(1.0 / 448 * 0.40625)  # tiny codes with fine bits
    x[1, 128:] = -1.0
    x[2, :128] *= -1
    x[3, 1:128:2] = np.float32(3.0 / 448 * 0.0078125)
    xb = inputs.to_bf16_bits(x)
    q, s, c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    rq, rs = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(xb))
    assert np.array_equal(q.cpu().numpy(), rq)
    S = oracle.e4m3.decode(rq).reshape(4, 2, 128).sum(axis=2)
    assert np.abs(S).max() > 2 ** 15
    _check_gcorr(scales_from_gpu_layout(c, 4), rq, rs)


def test_quant_gather(lib):
    rng = np.random.default_rng(9)
    T, K, k = 50, 512, 3
    xb = _bf16_rows(rng, T, K)
    ids = _distinct_ids(rng, T, 16, k)
    _, _, d2s = oracle.permute(ids, 16)
    q, s, c = lib.fp8_quant_per_token_group(bf16_from_bits(xb), to_dev(d2s.astype(np.int32)), k)
    rq, rs = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(xb))
    tok = d2s // k
    assert np.array_equal(q.cpu().numpy(), rq[tok])
    assert np.array_equal(scales_from_gpu_layout(s, T * k), rs[tok])


@pytest.mark.parametrize("M,I", [(3, 128), (77, 512), (512, 2048), (4200, 2048)])
def test_silu_mul_requant(lib, M, I):
    # Codes are decided in fp32 on both sides, but exp differs in the last bit between the
    # device and numpy, so a code may move by one step on a rounding tie.
    rng = np.random.default_rng(M + I)
    gu = rng.standard_normal((M, 2 * I)).astype(np.float32) * 4
    gu[0, :I] = 0.0
    if M > 1:
        gu[1, :I] = -200.0                      # silu(-200) ~ 0
    gub = inputs.to_bf16_bits(gu)
    q, s, c = lib.silu_mul_requant(bf16_from_bits(gub))
    rq, rs = oracle.silu_mul_requant(inputs.bf16_bits_to_f32(gub).astype(np.float64))
    gq = q.cpu().numpy()
    gs = scales_from_gpu_layout(s, M)
    assert np.max(np.abs(gs.astype(np.float64) - rs) / rs) <= 1e-6
    diff = gq != rq
    assert diff.mean() <= 1e-3
    if diff.any():
        step = np.abs(gq[diff].astype(np.int32) - rq[diff].astype(np.int32))
        assert np.all((step == 1) | ((gq[diff] & 0x7F) == 0) & ((rq[diff] & 0x7F) <= 1))
    assert rel_fro(oracle.dequant(gq, gs), oracle.dequant(rq, rs)) <= 1e-3
    _check_gcorr(scales_from_gpu_layout(c, M), gq, gs)


@pytest.mark.parametrize("T,k,H", [(1, 1, 8), (64, 8, 7168), (300, 2, 256), (129, 32, 64)])
def test_combine(lib, T, k, H):
    rng = np.random.default_rng(T + k + H)
    P = T * k
    yb = inputs.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    s2d = rng.permutation(P).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    out = lib.moe_unpermute_combine(bf16_from_bits(yb), to_dev(s2d), to_dev(w))
    ref = oracle.round_bf16(oracle.unpermute_combine(inputs.bf16_bits_to_f32(yb), s2d, w, T, k))
    gb = bits_of_bf16(out)
    rb = oracle.bf16_bits(ref)
    ulp = bf16_ulp_diff(gb, rb)
    assert ulp.max() <= 1 and (ulp > 0).mean() <= 1e-2
    assert rel_fro(f64_of_bf16(out), ref) <= 1e-3


@pytest.mark.parametrize("rows,K", [(1, 8), (3, 256), (4096, 7168)])
def test_prepack_weights(lib, rows, K):
    # the prepacked bytes, read with the documented format, hold the same int4 values
    rng = np.random.default_rng(rows + K)
    packed = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    packed[0, :4] = [0x00, 0x88, 0x7F, 0xF8]
    got = lib.w4a8_prepack_weights(to_dev(packed)).cpu().numpy()
    assert np.array_equal(decode_prepacked(got), oracle.unpack_int4(packed))


@pytest.mark.parametrize("T,K,k,drop", [(1, 128, 1, 0.0), (64, 7168, 8, 0.0), (300, 512, 3, 0.0),
                                        (1000, 256, 8, 0.5), (5000, 1024, 4, 0.0)])
def test_quant_scatter_equals_gather(lib, T, K, k, drop):
    # quantising each source row once and scattering it through src2dst writes exactly what the gather
    # through dst2src writes (codes, scales, corrections), and matches the oracle on the placed rows
    rng = np.random.default_rng(T + K + k)
    x_bits = inputs.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    P = T * k
    s2d = rng.permutation(P).astype(np.int32)
    s2d[rng.random(P) < drop] = -1  # pairs of another expert-parallel shard
    PL = int((s2d >= 0).sum())
    keep = np.nonzero(s2d >= 0)[0]
    s2d[keep] = np.argsort(np.argsort(s2d[keep])).astype(np.int32)  # placed rows are 0 .. PL-1
    d2s = np.full(P, -1, np.int32)
    d2s[s2d[keep]] = keep.astype(np.int32)
    x = bf16_from_bits(x_bits)
    sq, ss, sc = lib.fp8_quant_scatter_per_token_group(x, to_dev(s2d), k, P)
    gq, gs, gc = lib.fp8_quant_per_token_group(x, to_dev(d2s), k)
    torch.cuda.synchronize()
    assert torch.equal(sq[:PL], gq[:PL]) and torch.equal(ss[:, :PL], gs[:, :PL]) and torch.equal(sc[:, :PL], gc[:, :PL])
    rq, rsc = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(x_bits))
    src = d2s[:PL] // k
    assert np.array_equal(sq[:PL].cpu().numpy(), rq[src])
    assert np.array_equal(ss[:, :PL].cpu().numpy().T, rsc[src])
    assert bool((sq[PL:] == 0).all())


def test_bounded_wait_gives_up_and_reports(lib):
    # a wait that nothing completes, with the GEMMs' bounded-wait routine and a 1 ms limit: it gives up,
    # the device error word carries the timeout bit (once: reading clears it), and the next GEMM is correct
    import ctypes
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.load().w4a8_test_wait_timeout(1_000_000, ctypes.c_void_p(flag.data_ptr()), st) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    assert lib.device_error() == 1
    assert lib.device_error() == 0
    rng = np.random.default_rng(3)
    M, N, K = 300, 256, 1024
    xb = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    packed = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    ws = rng.uniform(0.005, 0.02, size=(K // 128, N)).astype(np.float32)
    got = lib.w4a8_linear(aq, a_s, a_c, lib.w4a8_prepack_weights(to_dev(packed)), to_dev(ws))
    ref = oracle.linear(aq.cpu().numpy(), scales_from_gpu_layout(a_s, M), oracle.unpack_int4(packed), ws.T)
    assert rel_fro(got.float().cpu().numpy().astype(np.float64), ref) <= 1e-3
    assert lib.device_error() == 0
