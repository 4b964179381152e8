"""The grouped GEMM's tile-width cost model and launch plan (host logic of the library, no GPU).

The model prices one expert's rows x per 128-row weight block in units of one 16-wide tile:
narrow tiles cost ceil(x / 16); wide tiles cost 2 per tile plus 0.004 per row padded to 16 within the
tile (the a * R + b * T form of the DeepGEMM PR #53 page's cost model, fitted to GB300 sweeps).  The
expected costs under Poisson row counts and the plans of the workloads are checked against values
worked out by hand here.
"""
import ctypes
import math
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "w4afp8_mixture_experts_gb300", "_lib", "libw4a8moe.so")


@pytest.fixture(scope="module")
def clib():
    if not os.path.exists(LIB):
        pytest.skip("library not built")
    L = ctypes.CDLL(LIB)
    L.w4a8_tile_cost.restype = ctypes.c_double
    L.w4a8_tile_cost.argtypes = [ctypes.c_int, ctypes.c_int64]
    L.w4a8_expected_tile_cost.restype = ctypes.c_double
    L.w4a8_expected_tile_cost.argtypes = [ctypes.c_int, ctypes.c_double]
    L.w4a8_grouped_gemm_plan.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_int)]
    return L


@pytest.mark.parametrize("x,narrow,wide", [
    (0, 0.0, 0.0),
    (1, 1.0, 2.0 + 0.004 * 16),
    (16, 1.0, 2.0 + 0.004 * 16),
    (17, 2.0, 2.0 + 0.004 * 32),
    (32, 2.0, 2.0 + 0.004 * 32),
    (33, 3.0, 2.0 + 0.004 * 48),
    (128, 8.0, 2.0 + 0.004 * 128),
    (129, 9.0, 4.0 + 0.004 * (128 + 16)),
    (300, 19.0, 6.0 + 0.004 * (256 + 48)),
])
def test_tile_costs(clib, x, narrow, wide):
    assert clib.w4a8_tile_cost(0, x) == pytest.approx(narrow, abs=1e-12)
    assert clib.w4a8_tile_cost(1, x) == pytest.approx(wide, abs=1e-12)


def test_crossover_is_32_rows(clib):
    # 32 rows: two narrow tiles (2) against one wide tile padded to 32 rows (2.128); 33 rows: 3 > 2.192
    assert clib.w4a8_tile_cost(0, 32) <= clib.w4a8_tile_cost(1, 32)
    assert clib.w4a8_tile_cost(0, 33) > clib.w4a8_tile_cost(1, 33)
    th = ctypes.c_int()
    clib.w4a8_grouped_gemm_plan(512, 256, 7168, ctypes.byref(th))
    assert th.value == 32


def test_expected_costs_small_means(clib):
    # With a mean far below 16 rows an expert that holds any row holds at most 16 (the tail beyond is
    # below 1e-12 at these means): E[narrow] = P(X >= 1) = 1 - exp(-lambda); E[wide] = 2.064 * P(X >= 1)
    for lam in (0.05, 0.3, 1.0):
        p1 = 1.0 - math.exp(-lam)
        assert clib.w4a8_expected_tile_cost(0, lam) == pytest.approx(p1, rel=1e-9)
        assert clib.w4a8_expected_tile_cost(1, lam) == pytest.approx(2.064 * p1, rel=1e-9)
    assert clib.w4a8_expected_tile_cost(0, 0.0) == 0.0


def test_expected_cost_mid_mean(clib):
    # lambda = 20: ceil(x / 16) counts the k >= 0 with 16 k < x, so E[ceil(X / 16)] = sum_k P(X > 16 k),
    # written out with the Poisson tail sums up to k = 4 (beyond 64 rows the probability is below 1e-15)
    lam = 20.0
    pmf = [math.exp(-lam + x * math.log(lam) - math.lgamma(x + 1)) for x in range(200)]
    tail = lambda n: sum(pmf[n + 1:])  # P(X > n)
    e_narrow = sum(tail(16 * k) for k in range(5))
    assert clib.w4a8_expected_tile_cost(0, lam) == pytest.approx(e_narrow, rel=1e-9)


@pytest.mark.parametrize("M,E,K,plan", [
    (64 * 8, 256, 7168, 1),     # decode: 2 rows per expert on average -> narrow tiles only
    (64 * 8, 256, 2048, 1),
    (8192 * 8, 256, 7168, 2),   # prefill: 256 rows per expert -> wide tiles only
    (8192 * 8, 256, 2048, 2),
    (4096 * 8, 384, 7168, 3),   # skewed: mean 85 rows, between the crossover and the wide tile -> both
    (4096 * 8, 384, 2048, 3),
    (64 * 2, 8, 256, 1),        # tiny: 16 rows per expert
])
def test_plans_of_the_workloads(clib, M, E, K, plan):
    th = ctypes.c_int()
    assert clib.w4a8_grouped_gemm_plan(M, E, K, ctypes.byref(th)) == plan


def _plan_splits_by_hand(M, N, K, sms=152):
    # the dense Linear's K splits as the estimate defines them: 16-wide tiles (4 groups per stage) up to
    # 32 rows, 128-wide tiles (2 groups per stage) above; S = 1 .. 16 minimising
    # ceil(items / SMs) * ceil(stages / S) + 2 (S > 1), partials at most a quarter of the weight bytes
    nmax, gmax = (16, 4) if M <= 32 else (128, 2)
    G = K // 128
    gps = 1
    while gps * 2 <= gmax and G % (gps * 2) == 0:
        gps *= 2
    tiles = -(-M // nmax) * (N // 128)
    if tiles >= sms:
        return 1
    stages = G // gps
    best, best_cost = 1, -(-tiles // sms) * stages
    for S in range(2, 17):
        if S > stages or S * M * N * 4 > N * K // 8:
            break
        cost = -(-tiles * S // sms) * -(-stages // S) + 2
        if cost < best_cost:
            best, best_cost = S, cost
    return best


@pytest.mark.parametrize("N,K", [(24576, 1536), (7168, 16384), (18432, 7168), (7168, 2048), (1024, 8192), (256, 32768)])
def test_linear_split_plan(clib, N, K):
    # on a host without a GPU the library plans for the GB300's 152 SMs
    clib.w4a8_linear_split_k.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    for M in (1, 13, 16, 40, 128, 130, 1024, 8192):
        S = clib.w4a8_linear_split_k(M, N, K)
        assert S == _plan_splits_by_hand(M, N, K), (M, N, K, S)
        assert 1 <= S <= 16 and (S == 1 or S * M * N * 4 <= N * K // 8)
    # the sweep's one split shape family: (7168, 16384) splits 8 ways at M = 1 and 16, twice at 128
    assert [clib.w4a8_linear_split_k(M, 7168, 16384) for M in (1, 16, 128, 1024)] == [8, 8, 2, 1]
