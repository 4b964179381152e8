"""The oracle's pins catch plausible mistakes: each test plants one mistake in the oracle (CPU
only, through monkeypatch) and checks that at least one pin then fails.

A mistake that no pin caught would mean a function of the oracle is trusted on its own say-so.
"""
import functools

import numpy as np
import pytest

import oracle
import oracle.e4m3 as e4m3
import oracle.moe as moe
import test_oracle_e4m3 as pe
import test_oracle_gemm as pg
import test_oracle_moe as pm
import test_oracle_quant as pq
import test_oracle_route_permute as pr


def _plant(monkeypatch, name, fn, module=moe):
    """Replace oracle function `name` in its module and in the package namespace."""
    monkeypatch.setattr(module, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _caught(*pins):
    """Number of pins that fail (assertion or error) under the planted mistake."""
    failed = 0
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception:  # noqa: BLE001 - a pin failing in any way counts
            failed += 1
    return failed


# --- E4M3 codec ---------------------------------------------------------------

def test_decode_with_bias_8_is_caught(monkeypatch):
    bad = np.array([e4m3._decode_one(c) / 2.0 for c in range(256)])
    monkeypatch.setattr(e4m3, "DECODE_TABLE", bad)
    assert _caught(pe.test_decode_fixed_points, pe.test_int4_values_are_exact) > 0


def _encode_truncating(x):
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(np.nan_to_num(x)), e4m3.MAX_FINITE)
    idx = np.searchsorted(e4m3._POS_VALUES, mag, side="right") - 1  # round toward zero
    code = np.clip(idx, 0, 0x7E).astype(np.uint8)
    return (code | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))).astype(np.uint8)


def test_encode_truncating_is_caught(monkeypatch):
    monkeypatch.setattr(e4m3, "encode", _encode_truncating)
    assert _caught(pe.test_ties_to_even_and_neighbours, functools.partial(pe.test_matches_torch_cast_in_range, 0)) > 0


def test_encode_without_saturation_is_caught(monkeypatch):
    good = e4m3.encode

    def unsaturated(x):
        c = good(x)
        return np.where(np.abs(np.asarray(x, dtype=np.float64)) > e4m3.MAX_FINITE, np.uint8(0x7F), c).astype(np.uint8)

    monkeypatch.setattr(e4m3, "encode", unsaturated)
    assert _caught(pe.test_saturation) > 0


def test_encode_losing_negative_zero_is_caught(monkeypatch):
    good = e4m3.encode
    monkeypatch.setattr(e4m3, "encode", lambda x: np.where(good(x) == 0x80, np.uint8(0), good(x)).astype(np.uint8))
    assert _caught(pe.test_signed_zero) > 0


# --- quantisation -------------------------------------------------------------

def test_scale_over_447_is_caught(monkeypatch):
    monkeypatch.setattr(moe, "FP8_MAX", np.float32(447.0))
    assert _caught(pq.test_amax_maps_to_448, pq.test_matches_torch_route) > 0


def test_missing_amax_floor_is_caught(monkeypatch):
    monkeypatch.setattr(moe, "AMAX_FLOOR", np.float32(0.0))
    assert _caught(pq.test_zero_row_and_spike) > 0


# --- int4 packing and the GEMM ------------------------------------------------

def test_swapped_nibble_order_is_caught(monkeypatch):
    good = moe.unpack_int4

    def swapped(packed):
        v = good(packed)
        out = v.copy()
        out[..., 0::2], out[..., 1::2] = v[..., 1::2], v[..., 0::2]
        return out

    _plant(monkeypatch, "unpack_int4", swapped)
    assert _caught(pg.test_pack_order_hand_worked, pg.test_pack_round_trip) > 0


def _gemm_variant(drop_weight_scale=False, first_group_act_scale=False, transpose_scales=False):
    def gemm(a_codes, a_scales, w_int4, w_scales, group=moe.GROUP):
        A = e4m3.decode(a_codes)
        W = np.asarray(w_int4, dtype=np.float64)
        a_s = np.asarray(a_scales, dtype=np.float64)
        w_s = np.asarray(w_scales, dtype=np.float64)
        if transpose_scales:
            w_s = w_s[::-1]
        G = A.shape[1] // group
        y = np.zeros((A.shape[0], W.shape[0]))
        for g in range(G):
            ks = slice(g * group, (g + 1) * group)
            P = A[:, ks] @ W[:, ks].T
            sa = a_s[:, 0] if first_group_act_scale else a_s[:, g]
            sw = np.ones(W.shape[0]) if drop_weight_scale else w_s[:, g]
            y += sa[:, None] * sw[None, :] * P
        return y
    return gemm


@pytest.mark.parametrize("kind", ["drop_weight_scale", "first_group_act_scale", "transpose_scales"])
def test_gemm_mistakes_are_caught(monkeypatch, kind):
    _plant(monkeypatch, "w4a8_gemm", _gemm_variant(**{kind: True}))
    assert _caught(functools.partial(pg.test_grouped_form_equals_dense_dequantised_matmul, 5, 7, 384),
                   pg.test_brute_force_tiny, pg.test_power_of_two_scales_are_exact) > 0


def test_bf16_truncation_is_caught(monkeypatch):
    def trunc(x):
        b = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
        return b.view(np.float32).astype(np.float64)

    _plant(monkeypatch, "round_bf16", trunc)
    assert _caught(pg.test_round_bf16_matches_torch) > 0


# --- SiLU and Mul -------------------------------------------------------------

def test_silu_without_gate_factor_is_caught(monkeypatch):
    _plant(monkeypatch, "silu", lambda g: 1.0 / (1.0 + np.exp(-np.asarray(g, dtype=np.float64))))
    assert _caught(pg.test_silu_closed_forms) > 0


def test_silu_mul_swapping_gate_and_up_is_caught(monkeypatch):
    def swapped(y13):
        y = np.asarray(y13, dtype=np.float64)
        I = y.shape[1] // 2
        return moe.silu(y[:, I:]) * y[:, :I]

    _plant(monkeypatch, "silu_mul", swapped)
    assert _caught(pg.test_silu_mul_uses_gate_then_up) > 0


# --- routing, permutation, combine ---------------------------------------------

def test_route_without_renormalisation_is_caught(monkeypatch):
    good = moe.route_topk
    _plant(monkeypatch, "route_topk", lambda lg, k, renormalize=True: good(lg, k, renormalize=False))
    assert _caught(pr.test_route_hand_worked, functools.partial(pr.test_route_matches_brute_force, 7, 8, 2)) > 0


def test_route_ties_to_higher_id_are_caught(monkeypatch):
    def ties_high(logits, k, renormalize=True):
        lg = np.asarray(logits, dtype=np.float32)
        flipped = lg[:, ::-1]
        ids, w = moe.__dict__["_route_unpatched"](flipped, k, renormalize)
        return (lg.shape[1] - 1 - ids).astype(np.int32), w

    monkeypatch.setattr(moe, "_route_unpatched", moe.route_topk, raising=False)
    _plant(monkeypatch, "route_topk", ties_high)
    assert _caught(pr.test_route_hand_worked, functools.partial(pr.test_route_matches_brute_force, 7, 8, 2)) > 0


def test_unstable_permutation_is_caught(monkeypatch):
    good = moe.permute

    def unstable(topk_ids, E):
        seg, _, dst2src = good(topk_ids, E)
        d2s = dst2src.copy()
        for e in range(E):  # reverse the order inside every expert
            d2s[seg[e]:seg[e + 1]] = d2s[seg[e]:seg[e + 1]][::-1]
        s2d = np.empty_like(d2s)
        s2d[d2s] = np.arange(d2s.size, dtype=d2s.dtype)
        return seg, s2d, d2s

    _plant(monkeypatch, "permute", unstable)
    assert _caught(pr.test_permute_hand_worked, functools.partial(pr.test_permute_invariants, 9, 4, 2)) > 0


def test_combine_ignoring_routing_weights_is_caught(monkeypatch):
    good = moe.unpermute_combine
    _plant(monkeypatch, "unpermute_combine",
           lambda y2, s2d, w, T, k: good(y2, s2d, np.ones_like(np.asarray(w, dtype=np.float64)), T, k))
    assert _caught(pr.test_combine_hand_worked) > 0


def test_layer_combining_through_dst2src_is_caught(monkeypatch):
    good = moe.unpermute_combine

    def wrong_index(y2, src2dst, w, T, k):
        s2d = np.asarray(src2dst)
        d2s = np.empty_like(s2d)
        d2s[s2d] = np.arange(s2d.size, dtype=s2d.dtype)
        return good(y2, d2s, w, T, k)

    _plant(monkeypatch, "unpermute_combine", wrong_index)
    assert _caught(pm.test_hand_worked_layer) > 0


# --- expert-parallel shard mode -------------------------------------------------

import test_oracle_ep as pep  # noqa: E402


def test_ep_remote_pairs_kept_are_caught(monkeypatch):
    good = moe.permute

    def keeps_remote(topk_ids, E, expert_map=None):
        if expert_map is None:
            return good(topk_ids, E)
        return good(topk_ids, E, np.maximum(np.asarray(expert_map), 0))  # remote experts folded into local 0

    _plant(monkeypatch, "permute", keeps_remote)
    assert _caught(pep.test_permute_ep_hand_worked,
                   functools.partial(pep.test_shards_add_up_to_the_layer, [[0, 1], [2, 3]])) > 0


def test_ep_combine_reading_remote_slots_is_caught(monkeypatch):
    def no_skip(y2, src2dst, topk_w, T, k):
        y2 = np.asarray(y2, dtype=np.float64)
        w = np.asarray(topk_w, dtype=np.float64).reshape(T, k)
        s2d = np.asarray(src2dst, dtype=np.int64).reshape(T, k)
        out = np.zeros((T, y2.shape[1]))
        for j in range(k):
            out += w[:, j][:, None] * y2[s2d[:, j]]  # -1 reads the last row
        return out

    _plant(monkeypatch, "unpermute_combine", no_skip)
    assert _caught(pep.test_combine_skips_remote_pairs,
                   functools.partial(pep.test_shards_add_up_to_the_layer, [[0, 1], [2, 3]])) > 0


def test_ep_unstable_local_order_is_caught(monkeypatch):
    good = moe.permute

    def unstable(topk_ids, E, expert_map=None):
        seg, s2d, d2s = good(topk_ids, E, expert_map)
        d2s = d2s.copy()
        for e in range(seg.size - 1):
            d2s[seg[e]:seg[e + 1]] = d2s[seg[e]:seg[e + 1]][::-1]
        s2d = np.full_like(s2d, -1)
        s2d[d2s] = np.arange(d2s.size, dtype=s2d.dtype)
        return seg, s2d, d2s

    _plant(monkeypatch, "permute", unstable)
    assert _caught(pep.test_permute_ep_hand_worked, pep.test_permute_ep_reordered_local_ids) > 0
