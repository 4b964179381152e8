"""GPU parity of the int4 x FP8 grouped GEMM and the dense Linear (tcgen05 kernels).

Inputs are seeded; the oracle computes in float64 from the same E4M3 codes,
int4 values and fp32 scales, and its result is rounded once to bf16.  Each
GEMM stage must agree within a relative Frobenius error of 1e-3.
"""
import numpy as np
import pytest
import torch

import inputs
import oracle
from oracle import e4m3
from gpu_util import f64_of_bf16, gcorr_of, prepacked, rel_fro, scales_from_gpu_layout, scales_to_gpu_layout, to_dev

pytestmark = pytest.mark.gpu


def _acts(rng, M, K):
    x = rng.standard_normal((M, K)).astype(np.float32) * rng.uniform(0.1, 10, (M, 1)).astype(np.float32)
    return oracle.quant_per_token_group(x)


def _weights(rng, E, N, K):
    packed = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, size=(E, K // 128, N)).astype(np.float32)
    return packed, s


def _run_grouped(lib, aq, a_s, packed, ws, seg):
    return lib.w4a8_grouped_gemm(to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s)),
                                 prepacked(lib, packed), to_dev(ws), to_dev(seg.astype(np.int64)))


def _oracle_grouped(aq, a_s, packed, ws, seg):
    return oracle.round_bf16(oracle.grouped_gemm(aq, a_s, seg, lambda e: oracle.unpack_int4(packed[e]),
                                                 lambda e: ws[e].T))


@pytest.mark.parametrize("M", [16, 40, 300])  # M <= 32 per expert selects the small-M pipeline
def test_integer_case_is_exact(lib, M):
    # all scales 1, activations small integers, weights in {-1, 0, 1}: every product and
    # partial sum is an exact integer in fp32, so the device result must be exact.
    rng = np.random.default_rng(M)
    N, K = 256, 256
    a_int = rng.integers(-3, 4, size=(M, K))
    aq = e4m3.encode(a_int.astype(np.float32))
    a_s = np.ones((M, K // 128), np.float32)
    w = rng.integers(-1, 2, size=(1, N, K))
    packed = oracle.pack_int4(w)
    ws = np.ones((1, K // 128, N), np.float32)
    seg = np.array([0, M])
    got = f64_of_bf16(_run_grouped(lib, aq, a_s, packed, ws, seg))
    ref = oracle.round_bf16(a_int.astype(np.float64) @ w[0].T.astype(np.float64))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M", [13, 128])
def test_every_int4_value(lib, M):
    # one-hot activations pick single weights: C[j][n] = a * int4(W[n][j]) exactly
    N, K = 128, 128
    aq = np.zeros((M, K), np.uint8)
    aq[np.arange(M), np.arange(M)] = e4m3.encode(np.float32(2.0))
    a_s = np.ones((M, 1), np.float32)
    rng = np.random.default_rng(2)
    w = rng.integers(-8, 8, size=(1, N, K))
    w[0, :16, :16] = np.arange(-8, 8)[None, :]
    packed = oracle.pack_int4(w)
    ws = np.ones((1, 1, N), np.float32)
    got = f64_of_bf16(_run_grouped(lib, aq, a_s, packed, ws, np.array([0, M])))
    assert np.array_equal(got, 2.0 * w[0].T[:M].astype(np.float64))


@pytest.mark.parametrize("counts,N,K", [
    ([3, 0, 17, 1, 64, 2, 0, 9], 256, 256),          # decode-style tile (few rows per expert)
    ([40, 200, 0, 129, 5, 300, 1, 77], 384, 512),    # several token chunks per expert
    ([1] * 37, 128, 1024),
    ([0, 0, 0, 500], 128, 128),
    ([2, 0, 5, 1, 31, 3], 256, 4096),                # long K: the small-M pipeline with 4 MMA warps
    ([7, 1, 0, 16, 9], 128, 7168),
    ([500, 3, 0, 15, 16, 17, 40, 1], 256, 512),      # 32 to 128 rows per expert: experts <= 32 rows in their own launch
    ([300, 1, 16, 0, 2], 128, 4096),
    ([2000, 3, 0, 15], 128, 256),                    # >= 128 rows per expert: one launch, 128-wide tiles for all
    ([33, 32, 31, 0, 64, 20], 128, 1024),            # mean 30 rows: one side of the 32-row crossover or the other
])
def test_grouped_gemm(lib, counts, N, K):
    rng = np.random.default_rng(sum(counts) + N + K)
    E = len(counts)
    seg = np.concatenate([[0], np.cumsum(counts)])
    M = int(seg[-1])
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, E, N, K)
    got = f64_of_bf16(_run_grouped(lib, aq, a_s, packed, ws, seg))
    ref = _oracle_grouped(aq, a_s, packed, ws, seg)
    err = rel_fro(got, ref)
    assert err <= 1e-3, (err, np.abs(got - ref).max())
    assert lib.device_error() == 0


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (16, 256, 1536), (128, 384, 512), (300, 128, 2048),
                                   (1000, 256, 256)])
def test_linear(lib, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 1, N, K)
    got = f64_of_bf16(lib.w4a8_linear(to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s)),
                                      prepacked(lib, packed[0]), to_dev(ws[0])))
    ref = oracle.linear(aq, a_s, oracle.unpack_int4(packed[0]), ws[0].T)
    err = rel_fro(got, ref)
    assert err <= 1e-3, (err, np.abs(got - ref).max())
    assert lib.device_error() == 0


# Shapes with fewer 128-row weight tiles than SMs: K is split and a second kernel sums the
# fp32 partials (decode tiles for M <= 32, 128-row tiles above).
@pytest.mark.parametrize("M,N,K", [(1, 1024, 8192), (13, 512, 4096), (40, 256, 16384), (130, 256, 32768)])
def test_linear_split_k(lib, M, N, K):
    assert lib.linear_split_k(M, N, K) > 1
    rng = np.random.default_rng(M * 11 + N + K)
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 1, N, K)
    got = f64_of_bf16(lib.w4a8_linear(to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s)),
                                      prepacked(lib, packed[0]), to_dev(ws[0])))
    ref = oracle.linear(aq, a_s, oracle.unpack_int4(packed[0]), ws[0].T)
    err = rel_fro(got, ref)
    assert err <= 1e-3, (err, np.abs(got - ref).max())
    assert lib.device_error() == 0


def test_linear_split_k_workspace_contents_do_not_matter(lib):
    # The partial sums live in the caller's workspace: whatever it held before (bytes of 0xFF, random
    # bytes, the previous call's partials) the result is the same, bit for bit, and matches the oracle.
    M, N, K = 1, 1024, 8192
    assert lib.linear_split_k(M, N, K) > 1
    rng = np.random.default_rng(9)
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 1, N, K)
    args = (to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s)), prepacked(lib, packed[0]),
            to_dev(ws[0]))
    need = lib.linear_workspace_bytes(M, N, K)
    buf = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = [lib.w4a8_linear(*args, ws=buf).clone()]
    buf.copy_(torch.from_numpy(rng.integers(0, 256, need, dtype=np.uint8)))
    outs.append(lib.w4a8_linear(*args, ws=buf).clone())
    outs += [lib.w4a8_linear(*args, ws=buf).clone() for _ in range(3)]  # the words of the previous calls
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert all(torch.equal(o, outs[0]) for o in outs[1:])
    ref = oracle.linear(aq, a_s, oracle.unpack_int4(packed[0]), ws[0].T)
    assert rel_fro(f64_of_bf16(outs[0]), ref) <= 1e-3


def test_linear_split_k_needs_workspace(lib):
    M, N, K = 1, 1024, 8192
    rng = np.random.default_rng(5)
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 1, N, K)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.W4A8Error):
        lib.w4a8_linear(to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s)),
                        prepacked(lib, packed[0]), to_dev(ws[0]), ws=small)


def test_tile_configurations_agree_bit_for_bit(lib):
    # the same expert rows through the 16-wide tiles (few rows per expert), the 128-wide tiles (many) and
    # the two-launch split (in between): each output element is the same fp32 sequence of per-group MMA
    # partials and promotions, so the three give the same bf16 bits
    rng = np.random.default_rng(77)
    N, K, R = 256, 512, 10
    aq0, as0 = _acts(rng, R, K)
    big_q, big_s = _acts(rng, 300, K)
    packed, ws = _weights(rng, 2, N, K)
    outs = []
    for other in (0, 300, 200):  # M = 10 (16-wide), 310 (128-wide), 210 (split: expert 0 on 16-wide tiles)
        aq = np.concatenate([aq0, big_q[:other]])
        a_s = np.concatenate([as0, big_s[:other]])
        seg = np.array([0, R, R + other])
        outs.append(_run_grouped(lib, aq, a_s, packed, ws, seg)[:R].cpu())
    assert lib.device_error() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    ref = _oracle_grouped(aq0, as0, packed, ws, np.array([0, R, R]))
    assert rel_fro(f64_of_bf16(outs[0]), ref) <= 1e-3



def test_output_alignment_and_guard_band(lib):
    # The 128-wide tiles store 16-byte pieces of output rows, so the entry points take C only 16-byte
    # aligned: an output 2 or 6 bytes past such a boundary is refused (invalid argument) with nothing
    # written, and one 16 bytes past it gives the bits of a fresh allocation with nothing written outside
    # C, for the grouped GEMM (ragged chunks: 140 and 160 rows) and the dense Linear.
    import ctypes
    raw = lib.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rng = np.random.default_rng(91)
    M, N, K = 300, 256, 512
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 2, N, K)
    seg = np.array([0, 140, M])
    A, S, G = to_dev(aq), scales_to_gpu_layout(a_s), scales_to_gpu_layout(gcorr_of(aq, a_s))
    Bp, Bs, sg = prepacked(lib, packed), to_dev(ws), to_dev(seg.astype(np.int64))
    Bl, Bls = Bp[0].contiguous(), Bs[0].contiguous()
    assert lib.linear_split_k(M, N, K) == 1  # the Linear's tiles store C directly (no partials)
    want = lib.w4a8_grouped_gemm(A, S, G, Bp, Bs, sg)
    want_lin = lib.w4a8_linear(A, S, G, Bl, Bls)
    p = ctypes.c_void_p

    def grouped(C):
        return raw.w4a8_grouped_gemm(p(A.data_ptr()), p(S.data_ptr()), p(G.data_ptr()), S.shape[1],
                                     p(Bp.data_ptr()), p(Bs.data_ptr()), p(sg.data_ptr()), 2, N, K, M,
                                     p(C.data_ptr()), None, 0, st)

    def linear(C):
        return raw.w4a8_linear(p(A.data_ptr()), p(S.data_ptr()), p(G.data_ptr()), S.shape[1], p(Bl.data_ptr()),
                               p(Bls.data_ptr()), M, N, K, p(C.data_ptr()), None, 0, st)

    for off in (1, 3, 8):  # 2, 6 and 16 bytes past a 256-byte aligned allocation
        for call, ref in ((grouped, want), (linear, want_lin)):
            buf = torch.full((M * N + 16,), 7.0, dtype=torch.bfloat16, device="cuda")
            C = buf[off:off + M * N]
            rc = call(C)
            torch.cuda.synchronize()
            if off == 8:
                assert rc == 0
                assert torch.equal(C.view(M, N), ref)
                assert torch.all(buf[:off] == 7.0) and torch.all(buf[off + M * N:] == 7.0)
            else:
                assert rc == 1  # W4A8_ERR_INVALID_ARG
                assert torch.all(buf == 7.0)
    assert lib.device_error() == 0

# The dense Linear sweep at its own shapes: M in {1, 16, 128, 1024, 8192} x (N, K) in {(24576, 1536),
# (7168, 16384), (18432, 7168), (7168, 2048)}, with the bench's weights (counter-based generator, filled
# on the device) and x ~ N(0,1) quantised by the library.  Every row up to M = 128 and a seeded sample of
# 64 rows (first and last included) above is compared with the oracle at 1e-3 relative Frobenius per
# shape; the sampled rows' codes and scales must equal the oracle's quantisation bit for bit.
@pytest.mark.parametrize("N,K", inputs.LINEAR_NK)
def test_linear_sweep_shapes(lib, N, K):
    from gpu_util import bf16_from_bits, scales_from_gpu_layout
    seed, G = 0, K // 128
    W = lib.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_LIN_W, (N, K // 2)))
    S = inputs.gpu_scales(seed, inputs.STREAM_LIN_SCALE, (G, N))
    got, codes, scales, spans = [], [], [], []
    for M in inputs.LINEAR_M:
        rng = np.random.default_rng(1000 + M)
        x_bits = inputs.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
        aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(x_bits))
        C = lib.w4a8_linear(aq, a_s, a_c, W, S)
        if M <= 128:
            sel = np.arange(M)
        else:
            sel = np.sort(np.concatenate([[0, M - 1], rng.choice(np.arange(1, M - 1), 62, replace=False)]))
        idx = torch.from_numpy(sel).cuda()
        got.append(f64_of_bf16(C.index_select(0, idx)))
        rq, rs = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(x_bits[sel]))
        assert np.array_equal(aq.index_select(0, idx).cpu().numpy(), rq)
        assert np.array_equal(scales_from_gpu_layout(a_s, M)[sel], rs)
        codes.append(rq)
        scales.append(rs)
        spans.append((M, len(sel)))
        assert lib.device_error() == 0
    Wh = oracle.unpack_int4(inputs.packed_int4(seed, inputs.STREAM_LIN_W, 0, N * K // 2).reshape(N, K // 2))
    Sh = np.ascontiguousarray(inputs.scales(seed, inputs.STREAM_LIN_SCALE, 0, G * N).reshape(G, N).T)
    ref = oracle.linear(np.concatenate(codes), np.concatenate(scales), Wh, Sh)
    o = 0
    for (M, n), g in zip(spans, got):
        err = rel_fro(g, ref[o:o + n])
        print(f"Linear M={M} N={N} K={K} (split-K {lib.linear_split_k(M, N, K)}): "
              f"{n} rows, rel Frobenius {err:.2e}")
        assert err <= 1e-3, (M, err)
        o += n


# a_gcorr = NULL: the GEMM computes the activation corrections from the codes itself (into its
# workspace), with the quantisation kernels' arithmetic, so the result is the one it gives with the
# corrections the quantisation emits, bit for bit; and within the stage tolerance of the oracle.
@pytest.mark.parametrize("kind,M,N,K", [("grouped", 0, 256, 512), ("grouped", 3000, 128, 1024),
                                        ("linear", 1, 1024, 8192), ("linear", 200, 384, 2048),
                                        ("linear", 1000, 256, 256)])
def test_gemm_without_caller_corrections(lib, kind, M, N, K):
    from gpu_util import bf16_from_bits
    rng = np.random.default_rng(M + N + K)
    if kind == "grouped":
        counts = [40, 0, 7, 300, 1] if M == 0 else list(rng.multinomial(M, [0.5, 0.3, 0.2]))
        M = int(sum(counts))
        seg = np.concatenate([[0], np.cumsum(counts)])
    xb = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    aq, a_s, a_c = lib.fp8_quant_per_token_group(bf16_from_bits(xb))
    E = len(seg) - 1 if kind == "grouped" else 1
    packed, ws = _weights(rng, E, N, K)
    if kind == "grouped":
        B, bs, sg = prepacked(lib, packed), to_dev(ws), to_dev(seg.astype(np.int64))
        with_c = lib.w4a8_grouped_gemm(aq, a_s, a_c, B, bs, sg)
        without = lib.w4a8_grouped_gemm(aq, a_s, None, B, bs, sg)
        ref = _oracle_grouped(aq.cpu().numpy(), scales_from_gpu_layout(a_s, M), packed, ws, seg)
    else:
        B, bs = prepacked(lib, packed[0]), to_dev(ws[0])
        with_c = lib.w4a8_linear(aq, a_s, a_c, B, bs)
        without = lib.w4a8_linear(aq, a_s, None, B, bs)
        ref = oracle.linear(aq.cpu().numpy(), scales_from_gpu_layout(a_s, M), oracle.unpack_int4(packed[0]), ws[0].T)
    assert lib.device_error() == 0
    assert torch.equal(with_c, without)
    assert rel_fro(f64_of_bf16(without), ref) <= 1e-3


def test_gemm_without_corrections_needs_workspace(lib):
    rng = np.random.default_rng(3)
    M, N, K = 64, 128, 256
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, 1, N, K)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = lib.load().w4a8_linear(to_dev(aq).data_ptr(), scales_to_gpu_layout(a_s).data_ptr(), None,
                                scale_ld_of(M), prepacked(lib, packed[0]).data_ptr(), to_dev(ws[0]).data_ptr(),
                                M, N, K, C.data_ptr(), small.data_ptr(), small.numel(), None)
    assert rc == 1  # W4A8_ERR_INVALID_ARG: the corrections need (K/128) x ld fp32 of workspace
    assert lib.linear_workspace_bytes(M, N, K) >= (K // 128) * scale_ld_of(M) * 4


def scale_ld_of(M):
    return max(4, (M + 3) // 4 * 4)


def test_in_place_tile_decode_matches_the_tile_list(lib):
    # Launches too large for the per-CTA shared-memory tile list decode each tile in place instead (a
    # search over the experts' chunk prefix).  Bounding the list at 0 tiles forces that path on small
    # shapes: the 16-wide, 128-wide and split plans, the dense split-K Linear and the fused SiLU epilogue
    # must give the same bits as with the list.
    clib = lib.load()
    rng = np.random.default_rng(2024)
    K = 1024
    cases = []
    for counts, N in (([3, 0, 17, 1, 9, 2], 256), ([300, 0, 129, 513], 256), ([40, 3, 200, 0, 1, 77], 128)):
        E = len(counts)
        seg = np.concatenate([[0], np.cumsum(counts)])
        aq, a_s = _acts(rng, int(seg[-1]), K)
        packed, ws = _weights(rng, E, N, K)
        cases.append(lambda aq=aq, a_s=a_s, packed=packed, ws=ws, seg=seg: _run_grouped(lib, aq, a_s, packed, ws, seg))
    aq, a_s = _acts(rng, 1, 8192)
    packed, ws = _weights(rng, 1, 1024, 8192)
    assert lib.linear_split_k(1, 1024, 8192) > 1
    cases.append(lambda: lib.w4a8_linear(to_dev(aq), scales_to_gpu_layout(a_s), None, prepacked(lib, packed[0]),
                                         to_dev(ws[0])))
    seg = np.array([0, 300, 300, 557], dtype=np.int64)
    xq, xs = _acts(rng, 557, K)
    packed2, ws2 = _weights(rng, 3, 512, K)
    B2 = prepacked(lib, packed2)

    def fused():
        q, s, c = lib.w4a8_grouped_gemm_silu(to_dev(xq), scales_to_gpu_layout(xs), None, B2, to_dev(ws2),
                                             to_dev(seg), fused=True)
        M = int(seg[-1])  # the scale rows past M are padding the kernels never write
        return torch.cat([q.flatten(), s[:, :M].contiguous().flatten().view(torch.uint8),
                          c[:, :M].contiguous().flatten().view(torch.uint8)])

    cases.append(fused)
    ref = [f().clone() for f in cases]
    torch.cuda.synchronize()
    try:
        assert clib.w4a8_test_tile_list_limit(0) == 0
        got = [f().clone() for f in cases]
        torch.cuda.synchronize()
    finally:
        clib.w4a8_test_tile_list_limit(-1)
    assert lib.device_error() == 0
    for i, (g, r) in enumerate(zip(got, ref)):
        assert torch.equal(g, r), i


@pytest.mark.parametrize("plan_rows", ["narrow", "split", "wide"])
def test_grouped_gemm_at_the_expert_limit(lib, plan_rows):
    # 1024 experts (the largest count the kernels take: the per-CTA chunk prefix and row starts then fill
    # 8 KB of shared memory and shorten the tile list), most of them empty, the rest with few or many rows
    rng = np.random.default_rng({"narrow": 1, "split": 2, "wide": 3}[plan_rows])
    E, N, K = 1024, 128, 256
    counts = np.zeros(E, dtype=np.int64)
    used = rng.choice(E, 48, replace=False)
    if plan_rows == "narrow":
        counts[used] = rng.integers(1, 20, used.size)
    elif plan_rows == "split":
        counts[used] = rng.integers(1, 20, used.size)
        counts[used[:30]] = rng.integers(150, 400, 30)
    else:
        counts[used] = rng.integers(200, 400, used.size)
    counts[0], counts[E - 1] = 3, 257  # the first and the last expert hold rows
    seg = np.concatenate([[0], np.cumsum(counts)])
    M = int(seg[-1])
    aq, a_s = _acts(rng, M, K)
    packed, ws = _weights(rng, E, N, K)
    got = f64_of_bf16(_run_grouped(lib, aq, a_s, packed, ws, seg))
    ref = _oracle_grouped(aq, a_s, packed, ws, seg)
    err = rel_fro(got, ref)
    assert err <= 1e-3, (plan_rows, err)
    assert lib.device_error() == 0
