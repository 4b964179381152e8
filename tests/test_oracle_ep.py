"""Pins of the oracle's expert-parallel shard mode (expert_map; pairs of remote experts skipped).

The shard mode is the local part of an expert-parallel layer (SGLang PR #7762 page, review of
ep_moe/layer.py: routed ids translated through expert_map before the preprocess).  What fixes it
independently of the code: a hand-worked permutation, the identity map reducing to the plain layer,
and the partition property (over any split of the experts into shards, the shards' float64 outputs
add up to the whole layer's, since every routed pair lands on exactly one shard).
"""
import numpy as np
import pytest

import oracle


def test_permute_ep_hand_worked():
    # flat ids 1,0 | 0,2 | 2,1 | 0,1; expert 0 lives elsewhere, 1 -> local 0, 2 -> local 1
    ids = np.array([[1, 0], [0, 2], [2, 1], [0, 1]], dtype=np.int32)
    seg, src2dst, dst2src = oracle.permute(ids, 3, expert_map=[-1, 0, 1])
    assert seg.tolist() == [0, 3, 5]
    assert dst2src.tolist() == [0, 5, 7, 3, 4]
    assert src2dst.tolist() == [0, -1, -1, 3, 4, 1, -1, 2]


def test_permute_ep_reordered_local_ids():
    # local ids need not follow the global order: 2 -> local 0, 0 -> local 1
    ids = np.array([[1, 0], [0, 2], [2, 1], [0, 1]], dtype=np.int32)
    seg, src2dst, dst2src = oracle.permute(ids, 3, expert_map=[1, -1, 0])
    assert seg.tolist() == [0, 2, 5]
    assert dst2src.tolist() == [3, 4, 1, 2, 6]
    assert src2dst.tolist() == [-1, 2, 3, 0, 1, -1, 4, -1]


def test_permute_ep_all_remote_and_identity():
    rng = np.random.default_rng(3)
    ids = np.array([rng.permutation(6)[:3] for _ in range(5)], dtype=np.int32)
    seg, src2dst, dst2src = oracle.permute(ids, 6, expert_map=[-1] * 6)
    assert seg.tolist() == [0] and dst2src.size == 0 and np.all(src2dst == -1)
    full = oracle.permute(ids, 6)
    same = oracle.permute(ids, 6, expert_map=list(range(6)))
    for a, b in zip(full, same):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("bad", [[-2, 0, 1], [0, 1]])
def test_permute_ep_rejects_bad_maps(bad):
    with pytest.raises(ValueError):
        oracle.permute(np.zeros((2, 1), dtype=np.int32), 3, expert_map=bad)


def test_combine_skips_remote_pairs():
    y2 = np.array([[1.0, 2.0], [10.0, 20.0]])
    src2dst = np.array([1, -1, 0, -1])  # T = 2, k = 2
    w = np.array([[0.5, 0.5], [0.25, 0.75]])
    out = oracle.unpermute_combine(y2, src2dst, w, 2, 2)
    assert out.tolist() == [[5.0, 10.0], [0.25, 0.5]]


def _tiny_layer(seed=11, T=6, H=256, I=128, E=4):
    rng = np.random.default_rng(seed)
    x = oracle.round_bf16(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w13 = rng.integers(-8, 8, size=(E, 2 * I, H))
    w2 = rng.integers(-8, 8, size=(E, H, I))
    s13 = rng.uniform(0.005, 0.02, size=(E, 2 * I, H // 128)).astype(np.float32)
    s2 = rng.uniform(0.005, 0.02, size=(E, H, I // 128)).astype(np.float32)
    return x, logits, w13, w2, s13, s2


def _layer(x, logits, k, w13, w2, s13, s2, experts=None):
    """One shard holding `experts` (global ids, in local order); None: the plain layer."""
    if experts is None:
        return oracle.moe_layer(x, logits, k, lambda e: w13[e], lambda e: s13[e], lambda e: w2[e], lambda e: s2[e])
    emap = [-1] * w13.shape[0]
    for l, e in enumerate(experts):
        emap[e] = l
    g = list(experts)
    return oracle.moe_layer(x, logits, k, lambda l: w13[g[l]], lambda l: s13[g[l]], lambda l: w2[g[l]],
                            lambda l: s2[g[l]], expert_map=emap)


@pytest.mark.parametrize("shards", [[[0, 1], [2, 3]], [[3], [1, 0], [2]], [[2, 0, 3, 1]]])
def test_shards_add_up_to_the_layer(shards):
    x, logits, w13, w2, s13, s2 = _tiny_layer()
    k = 2
    full = _layer(x, logits, k, w13, w2, s13, s2)
    total = np.zeros_like(full["out_f64"])
    for experts in shards:
        part = _layer(x, logits, k, w13, w2, s13, s2, experts)
        total += part["out_f64"]
    np.testing.assert_allclose(total, full["out_f64"], rtol=1e-12, atol=1e-12)


def test_shard_without_local_pairs_is_zero():
    x, logits, w13, w2, s13, s2 = _tiny_layer(T=3, E=8)
    ids, _ = oracle.route_topk(logits, 1)
    unused = [e for e in range(8) if e not in set(ids.reshape(-1).tolist())]
    part = _layer(x, logits, 1, w13, w2, s13, s2, unused[:1])
    assert np.all(part["out"] == 0) and part["dst2src"].size == 0


def test_moe_tokens_matches_shard_layer():
    x, logits, w13, w2, s13, s2 = _tiny_layer(seed=5)
    k = 2
    experts = [3, 1]
    part = _layer(x, logits, k, w13, w2, s13, s2, experts)
    emap = [-1, 1, -1, 0]
    out, _, _ = oracle.moe_tokens(x[[0, 4]], logits[[0, 4]], k, lambda l: w13[experts[l]],
                                  lambda l: s13[experts[l]], lambda l: w2[experts[l]], lambda l: s2[experts[l]],
                                  expert_map=emap)
    assert np.array_equal(out, part["out"][[0, 4]])
