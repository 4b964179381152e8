"""The sampled full-size parity machinery, pinned on the CPU against the oracle's whole layer.

Fed the oracle's own intermediates in place of a device's, the expert-by-expert computation must find
zero stage error and reproduce the whole layer's output rows of the sampled tokens exactly.
"""
import numpy as np

import fullsize
import inputs
import oracle
from helpers import moe_experts, moe_host_inputs


def _layer_rows(cfg, seed):
    x_bits, logits = moe_host_inputs(seed, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    w13, w2 = moe_experts(seed, cfg)
    lay = oracle.moe_layer(x, logits, cfg["k"], w13.w, w13.s, w2.w, w2.s)
    return x, logits, lay


def test_expert_by_expert_sample_equals_the_layer():
    cfg = dict(T=40, H=256, I=256, E=6, k=2, zipf=1.2)
    seed = 7
    x, logits, lay = _layer_rows(cfg, seed)
    k = cfg["k"]
    sample = fullsize.pick_tokens(cfg["T"], 12, 3, lay["ids"], cfg["E"])
    pairs = (sample[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    r = lay["src2dst"][pairs]
    tok = pairs // k
    rows = dict(xq=lay["xq"][tok], xs=lay["xs"][tok], y13=lay["y13"][r], hq=lay["hq"][r], hs=lay["hs"][r],
                y2=lay["y2"][r])
    stats, out_ref = fullsize.sampled_layer_check(seed, cfg, sample, logits, rows)
    assert stats["y13"] == 0 and stats["y2"] == 0 and stats["hq_mismatch"] == 0 and stats["hq_deq"] == 0
    assert np.array_equal(out_ref, lay["out"][sample])


def test_stage_errors_are_seen():
    # a perturbed Y2 row and a flipped code must show up in the statistics
    cfg = dict(T=16, H=256, I=256, E=4, k=2, zipf=None)
    seed = 2
    x, logits, lay = _layer_rows(cfg, seed)
    k = cfg["k"]
    sample = np.arange(cfg["T"])
    pairs = (sample[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    r = lay["src2dst"][pairs]
    tok = pairs // k
    rows = dict(xq=lay["xq"][tok], xs=lay["xs"][tok], y13=lay["y13"][r], hq=lay["hq"][r].copy(),
                hs=lay["hs"][r], y2=lay["y2"][r].copy())
    rows["y2"][3] *= 1.01
    rows["hq"][5, 7] ^= 1
    stats, _ = fullsize.sampled_layer_check(seed, cfg, sample, logits, rows)
    assert stats["y13"] == 0 and stats["y2"] > 1e-3 and stats["hq_mismatch"] > 0


def test_pick_tokens():
    ids = np.zeros((100, 2), np.int32)
    s = fullsize.pick_tokens(100, 10, 0, ids, 4, extra=(50, 51))
    assert s.size == 10 and len(set(s.tolist())) == 10
    assert {0, 99, 50, 51} <= set(s.tolist()) and np.all(np.diff(s) > 0)
    assert np.array_equal(fullsize.pick_tokens(8, 10, 0, ids, 4), np.arange(8))


def test_skew_extremes():
    ids = np.array([[0, 1], [0, 2], [0, 1], [3, 0], [1, 0]], np.int32)  # counts 5, 3, 1, 1
    toks, hot, cold = fullsize.skew_extremes(ids, 5, per_expert=2, n_cold=2)
    assert hot == 0 and cold == [2, 3]
    assert set(toks) == {0, 1, 3}  # two tokens of expert 0, the token of 2, the token of 3
