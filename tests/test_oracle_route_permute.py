"""Pins of routing (brute force, closed forms, invariants) and of the stable permutation."""
import math
import random

import numpy as np
import pytest

import oracle


def brute_topk(row, k):
    # every expert, sorted by (-logit, id) with Python's sort
    return [e for _, e in sorted(((-float(v), e) for e, v in enumerate(row)))[:k]]


@pytest.mark.parametrize("T,E,k", [(7, 8, 2), (5, 64, 8), (3, 384, 8), (4, 5, 5)])
def test_route_matches_brute_force(T, E, k):
    rng = np.random.default_rng(T * E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, :4] = lg[0, 0]  # a tie
    ids, w = oracle.route_topk(lg, k)
    for t in range(T):
        assert list(ids[t]) == brute_topk(lg[t], k)
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(w[t]) <= 0)
        assert len(set(ids[t].tolist())) == k


def test_route_hand_worked():
    lg = np.array([[0.0, 1.0, 3.0, 2.0],
                   [1.0, 1.0, 1.0, 1.0]], dtype=np.float32)
    ids, w = oracle.route_topk(lg, 2)
    assert ids.tolist() == [[2, 3], [0, 1]]
    e = math.e
    assert np.allclose(w[0], [e / (1 + e), 1 / (1 + e)], rtol=1e-15)
    assert np.allclose(w[1], [0.5, 0.5], rtol=0)
    ids, w = oracle.route_topk(lg, 2, renormalize=False)
    z = 1 + math.exp(-1) + math.exp(-2) + math.exp(-3)
    assert np.allclose(w[0], [1 / z, math.exp(-1) / z], rtol=1e-15)
    assert np.allclose(w[1], [0.25, 0.25], rtol=0)


def test_permute_hand_worked():
    # four tokens, top-2 of three experts; flat ids 1,0 | 0,2 | 2,1 | 0,1
    ids = np.array([[1, 0], [0, 2], [2, 1], [0, 1]], dtype=np.int32)
    seg, src2dst, dst2src = oracle.permute(ids, 3)
    assert seg.tolist() == [0, 3, 6, 8]
    assert dst2src.tolist() == [1, 2, 6, 0, 5, 7, 3, 4]
    assert src2dst.tolist() == [3, 0, 1, 6, 7, 4, 2, 5]


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (9, 4, 2), (100, 16, 4), (33, 256, 8)])
def test_permute_invariants(T, E, k):
    rng = random.Random(T + E + k)
    ids = np.array([rng.sample(range(E), k) for _ in range(T)], dtype=np.int32)
    seg, src2dst, dst2src = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    P = T * k
    assert seg[0] == 0 and seg[-1] == P and np.all(np.diff(seg) >= 0)
    assert sorted(dst2src.tolist()) == list(range(P))
    assert np.array_equal(src2dst[dst2src], np.arange(P))
    for e in range(E):
        block = dst2src[seg[e]:seg[e + 1]]
        assert np.all(flat[block] == e)
        assert np.all(np.diff(block) > 0)  # stable


def test_permute_unpermute_identity():
    # k = 1, unit weights: unpermute(permute(x)) = x
    rng = np.random.default_rng(5)
    T, E, H = 12, 5, 16
    ids = rng.integers(0, E, size=(T, 1)).astype(np.int32)
    x = rng.standard_normal((T, H))
    seg, src2dst, dst2src = oracle.permute(ids, E)
    xp = x[dst2src]
    back = oracle.unpermute_combine(xp, src2dst, np.ones((T, 1)), T, 1)
    assert np.array_equal(back, x)


def test_combine_hand_worked():
    y2 = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0], [1000.0, 2000.0]])
    src2dst = np.array([2, 0, 3, 1])  # token 0 -> rows 2, 0; token 1 -> rows 3, 1
    w = np.array([[0.5, 0.25], [0.125, 2.0]])
    out = oracle.unpermute_combine(y2, src2dst, w, 2, 2)
    assert out.tolist() == [[50.25, 100.5], [145.0, 290.0]]
