"""Plain, slow CPU oracle of the W4AFP8 mixture-of-experts layer and dense Linear.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The CUDA library never
calls it and shares no code, table or helper with it.

Every step follows the workflow of the SGLang PR #7762 page ("support
DeepSeek-R1-W4AFP8 model with ep-moe mode", Modifications: Workflow, and the
Gemini summary "CUTLASS W4A8 MoE Kernel Integration"): routing ids, a stable
permutation of the routed (token, slot) pairs by expert, FP8 scaling of the
hidden states, an int4 x FP8 grouped GEMM for w13 with group size 128, SiLU
and Mul with FP8 re-scaling of the intermediate, the same grouped GEMM for w2,
and an unpermutation weighted by the routing weights.  The dense W4AFP8 Linear
is the same mixed-input GEMM with one weight matrix (lyraW4AFp8 page,
"LyraW4fp8": "MoE and GEMMs", Machete GEMM).

Floating point: every contraction and every non-decision step is float64.
Quantisation decisions (the FP8 code of an activation) are taken in float32,
the precision the method computes its scales in, so that codes are exact.
Rounding of the bf16 tensors on the path (Y13, Y2, the layer output) is done
once, from float64, to nearest even.

Where the pages leave a point open, the plainest reading is taken and stated at
the function that depends on it: s = amax/448 per token per 128 columns with
amax clamped to >= 1e-12; int4 element 2b in the low nibble of byte b; w13 rows
[0, I) gate, [I, 2I) up; top-k ties broken towards the lower expert index;
softmax over the logits, then the top-k weights renormalised to sum to 1.

Parity pins: see tests/test_oracle_*.py (exhaustive E4M3 codec, closed forms,
brute force on tiny inputs, dense dequantise-then-matmul, integer special
cases, and a hand-worked 2-expert / 4-token example).
"""
from __future__ import annotations

import numpy as np

from . import e4m3

GROUP = 128
AMAX_FLOOR = np.float32(1e-12)
FP8_MAX = np.float32(448.0)


# ----------------------------------------------------------------------------
# bf16 helpers

def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64.

    bf16 keeps 8 significant bits; subnormals (below 2**-126) step by 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)
    q = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    return np.where(x == 0, x, q)


def bf16_bits(x) -> np.ndarray:
    """Bit patterns (uint16) of bf16-representable float64 values."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# int4 packing

def unpack_int4(packed) -> np.ndarray:
    """uint8 [..., K/2] -> int8 [..., K].

    Byte b holds element k = 2b in bits 0-3 and k = 2b+1 in bits 4-7, each a
    two's-complement nibble (-8..7).  Lower k in the lower bits follows the
    unpack order of the SGLang PR #37796 page (Modifications: the 2-bit unpack
    is "the generalization of the 4-bit branch", shift (offs_k % n) * bits).
    """
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0x0F).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def pack_int4(values) -> np.ndarray:
    """int [..., K] in -8..7 -> uint8 [..., K/2] (inverse of unpack_int4)."""
    v = np.asarray(values, dtype=np.int16)
    if v.shape[-1] % 2:
        raise ValueError("K must be even")
    if v.min(initial=0) < -8 or v.max(initial=0) > 7:
        raise ValueError("int4 values must lie in [-8, 7]")
    n = (v & 0xF).astype(np.uint8)
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


# ----------------------------------------------------------------------------
# (1) routing

def route_topk(logits, k: int, renormalize: bool = True):
    """Softmax over router logits, top-k experts, optional renormalisation.

    The ids feed the permutation preprocess (SGLang PR #7762 page, review of
    ep_moe/kernels.py, run_cutlass_moe_ep_preproess(local_topk_ids, ...)).
    Order: descending logit, equal logits by ascending expert id.  Weights:
    p = softmax(logits) in float64; with renormalisation w_j = p_j / sum of the
    selected p, i.e. exp(l_j - l_max) / sum_sel exp(l_i - l_max).
    Returns ids int32 [T, k] and weights float64 [T, k].
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        row = lg[t].astype(np.float64)
        order = np.argsort(-row, kind="stable")  # ties keep ascending index
        sel = order[:k]
        ids[t] = sel
        ex = np.exp(row - row.max())
        w[t] = ex[sel] / (ex[sel].sum() if renormalize else ex.sum())
    return ids, w


# ----------------------------------------------------------------------------
# (2) permutation preprocess

def permute(topk_ids, E: int, expert_map=None):
    """Stable sort of the flat routed pairs f = t*k + j by expert.

    SGLang PR #7762 page, review of ep_moe/kernels.py: the preprocess sorts
    topk_ids.view(-1) with stable=True (reorder_ids), fills seg_indptr[E+1]
    (int64 segment starts of each expert) and src2dst (position of each flat
    pair in sorted order).  Returns seg_indptr int64 [E+1], src2dst int32 [P],
    dst2src int32 [P] (= reorder_ids).

    Expert-parallel shard (same page, review of ep_moe/layer.py: with an
    expert_map the routed ids are translated to this rank's local ids before
    the preprocess, which then runs over the local experts): expert_map is an
    int array [E] holding each global expert's local id on this shard, or -1
    when the expert lives elsewhere.  Reading taken: pairs mapped to -1 are
    not placed at all (src2dst = -1 for them); the local pairs, P_local of
    them, are sorted stably by local id, seg_indptr has E_local + 1 entries
    with E_local = max(expert_map) + 1, and dst2src has length P_local.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    if expert_map is None:
        local, n_local = flat, E
    else:
        emap = np.asarray(expert_map, dtype=np.int64)
        if emap.shape != (E,) or (emap.size and emap.min() < -1):
            raise ValueError("expert_map must hold E local ids or -1")
        n_local = int(emap.max()) + 1 if emap.size else 0
        local = emap[flat]
    keep = np.nonzero(local >= 0)[0]
    dst2src = keep[np.argsort(local[keep], kind="stable")].astype(np.int32)
    src2dst = np.full(flat.size, -1, dtype=np.int32)
    src2dst[dst2src] = np.arange(dst2src.size, dtype=np.int32)
    counts = np.bincount(local[keep], minlength=n_local)
    seg = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return seg, src2dst, dst2src


# ----------------------------------------------------------------------------
# (3) FP8 activation quantisation

def quant_per_token_group(x, group: int = GROUP):
    """bf16/fp32 activations [M, K] -> E4M3 codes [M, K] and fp32 scales [M, K/group].

    Per row and per group of 128 columns (the PR #7762 page: chunk_size is 128
    for the DeepSeek-R1-W4AFP8 group size): amax = max |x|, clamped to at
    least 1e-12 (the page of DeepGEMM PR #53, "SM90 FP4 MegaMoE": clamp amax
    before the reciprocal, since padded rows have amax == 0), s = amax / 448 in
    fp32, code = E4M3(x / s) rounded to nearest even and saturated at +-448
    (PR #37796 page, fp8 write path).  Both divisions are IEEE fp32.
    """
    x32 = np.asarray(x, dtype=np.float32)
    M, K = x32.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    G = K // group
    xg = x32.reshape(M, G, group)
    amax = np.abs(xg).max(axis=2) if M else np.zeros((0, G), np.float32)
    amax = np.maximum(amax, AMAX_FLOOR).astype(np.float32)
    s = (amax / FP8_MAX).astype(np.float32)
    y = (xg / s[:, :, None]).astype(np.float32)
    codes = e4m3.encode(y).reshape(M, K)
    return codes, s


def dequant(codes, s, group: int = GROUP) -> np.ndarray:
    """E4M3 codes [M, K] and scales [M, K/group] -> float64 values code * scale."""
    v = e4m3.decode(codes)
    M, K = v.shape
    return (v.reshape(M, K // group, group) * np.asarray(s, np.float64)[:, :, None]).reshape(M, K)


# ----------------------------------------------------------------------------
# (4) the int4 x FP8 GEMM with per-128-group scales

def w4a8_gemm(a_codes, a_scales, w_int4, w_scales, group: int = GROUP) -> np.ndarray:
    """y[m, n] = sum_g a_s[m, g] * w_s[n, g] * sum_{k in g} e4m3(a[m, k]) * int4(w[n, k]).

    a_codes uint8 [M, K], a_scales fp32 [M, G], w_int4 int8 [N, K] (unpacked
    values), w_scales fp32 [N, G].  float64 result [M, N].  This is the W4A8
    grouped GEMM of the PR #7762 page (cutlass_w4a8_moe, chunk_size 128) for
    one expert; the per-group partial sums are scaled and added group by group.
    """
    A = e4m3.decode(a_codes)
    W = np.asarray(w_int4, dtype=np.float64)
    a_s = np.asarray(a_scales, dtype=np.float64)
    w_s = np.asarray(w_scales, dtype=np.float64)
    M, K = A.shape
    N = W.shape[0]
    G = K // group
    y = np.zeros((M, N), dtype=np.float64)
    for g in range(G):
        ks = slice(g * group, (g + 1) * group)
        P = A[:, ks] @ W[:, ks].T
        y += a_s[:, g][:, None] * w_s[:, g][None, :] * P
    return y


def grouped_gemm(a_codes, a_scales, seg_indptr, w_of_expert, ws_of_expert):
    """Rows [seg[e], seg[e+1]) of the permuted activations times expert e's weights.

    w_of_expert(e) -> int8 [N, K]; ws_of_expert(e) -> fp32 [N, G].  float64 [P, N].
    """
    seg = np.asarray(seg_indptr, dtype=np.int64)
    E = seg.size - 1
    out = None
    for e in range(E):
        r0, r1 = int(seg[e]), int(seg[e + 1])
        if r1 == r0:
            continue
        y = w4a8_gemm(a_codes[r0:r1], a_scales[r0:r1], w_of_expert(e), ws_of_expert(e))
        if out is None:
            out = np.zeros((a_codes.shape[0], y.shape[1]), dtype=np.float64)
        out[r0:r1] = y
    return out


# ----------------------------------------------------------------------------
# (5) SiLU and Mul, then FP8 re-quantisation

def silu(g) -> np.ndarray:
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g)), float64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def silu_mul(y13) -> np.ndarray:
    """h = silu(gate) * up; gate = columns [0, I), up = columns [I, 2I) (PR #7762: SiLU and Mul)."""
    y = np.asarray(y13, dtype=np.float64)
    I = y.shape[1] // 2
    return silu(y[:, :I]) * y[:, I:]


def silu_mul_requant(y13):
    """SiLU and Mul in float64, rounded to fp32 (the kernel's precision), then step (3)."""
    h32 = silu_mul(y13).astype(np.float32)
    return quant_per_token_group(h32)


# ----------------------------------------------------------------------------
# (6) unpermute and combine

def unpermute_combine(y2, src2dst, topk_w, T: int, k: int) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y2[src2dst[t*k + j]] in float64 (PR #7762: post-reorder).

    Pairs with src2dst = -1 (routed to another expert-parallel shard) add nothing.
    """
    y2 = np.asarray(y2, dtype=np.float64)
    w = np.asarray(topk_w, dtype=np.float64).reshape(T, k)
    s2d = np.asarray(src2dst, dtype=np.int64).reshape(T, k)
    out = np.zeros((T, y2.shape[1]), dtype=np.float64)
    for j in range(k):
        here = s2d[:, j] >= 0
        out[here] += w[here, j][:, None] * y2[s2d[here, j]]
    return out


# ----------------------------------------------------------------------------
# the whole layer

def moe_layer(x_bf16, logits, k, w13_of_expert, w13s_of_expert, w2_of_expert, w2s_of_expert,
              renormalize: bool = True, expert_map=None):
    """The W4AFP8 MoE layer, step by step; returns a dict of every intermediate.

    x_bf16: float array [T, H] holding bf16 values.  w13_of_expert(e) -> int8
    [2I, H] (rows [0, I) gate, [I, 2I) up); w2_of_expert(e) -> int8 [H, I];
    the *_s functions return fp32 [N, K/128].  With an expert_map (see permute)
    the layer is one expert-parallel shard: e is a local id, only the pairs
    routed to local experts are computed, and out_f64 / out are this shard's
    share of the output (the shards' float64 shares sum to the whole layer's).
    """
    x = np.asarray(x_bf16, dtype=np.float32)
    T = x.shape[0]
    E = np.asarray(logits).shape[1]
    ids, w = route_topk(logits, k, renormalize)
    seg, src2dst, dst2src = permute(ids, E, expert_map)
    xq, xs = quant_per_token_group(x)
    tok = dst2src.astype(np.int64) // k
    a_codes, a_scales = xq[tok], xs[tok]
    if dst2src.size == 0:  # no pair routed to this shard
        return dict(ids=ids, w=w, seg=seg, src2dst=src2dst, dst2src=dst2src, xq=xq, xs=xs, y13=None,
                    hq=None, hs=None, y2=None, out_f64=np.zeros((T, x.shape[1])), out=np.zeros((T, x.shape[1])))
    y13 = round_bf16(grouped_gemm(a_codes, a_scales, seg, w13_of_expert, w13s_of_expert))
    hq, hs = silu_mul_requant(y13)
    y2 = round_bf16(grouped_gemm(hq, hs, seg, w2_of_expert, w2s_of_expert))
    out_f64 = unpermute_combine(y2, src2dst, w, T, k)
    out = round_bf16(out_f64)
    return dict(ids=ids, w=w, seg=seg, src2dst=src2dst, dst2src=dst2src, xq=xq, xs=xs,
                y13=y13, hq=hq, hs=hs, y2=y2, out_f64=out_f64, out=out)


def moe_tokens(x_bf16_rows, logits_rows, k, w13_of_expert, w13s_of_expert, w2_of_expert,
               w2s_of_expert, renormalize: bool = True, expert_map=None):
    """Layer output for a subset of tokens, one routed pair at a time.

    Each pair's values do not depend on the other tokens (quantisation is per
    token, the GEMMs are row-wise and the permutation only moves rows), so a
    sample of tokens is computed exactly as moe_layer would for those rows.
    With an expert_map, the pairs of experts mapped to -1 are skipped and the
    weight functions take local ids (one expert-parallel shard, as moe_layer).
    Returns out float64 [Ts, H] (bf16 values) and the routing (ids, w).
    """
    x = np.asarray(x_bf16_rows, dtype=np.float32)
    ids, w = route_topk(logits_rows, k, renormalize)
    xq, xs = quant_per_token_group(x)
    T, H = x.shape
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            e = int(ids[t, j])
            if expert_map is not None:
                e = int(expert_map[e])
                if e < 0:
                    continue
            y13 = round_bf16(w4a8_gemm(xq[t:t + 1], xs[t:t + 1], w13_of_expert(e), w13s_of_expert(e)))
            hq, hs = silu_mul_requant(y13)
            y2 = round_bf16(w4a8_gemm(hq, hs, w2_of_expert(e), w2s_of_expert(e)))
            acc += w[t, j] * y2[0]
        out[t] = round_bf16(acc)
    return out, ids, w


def linear(a_codes, a_scales, w_int4, w_scales) -> np.ndarray:
    """Dense W4AFP8 Linear: the mixed-input GEMM with one weight matrix, bf16 output."""
    return round_bf16(w4a8_gemm(a_codes, a_scales, w_int4, w_scales))
