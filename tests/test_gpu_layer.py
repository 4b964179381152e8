"""GPU parity of the whole W4AFP8 MoE layer.

Small workloads are compared stage by stage (every intermediate of the
w4a8_moe_forward workspace against the oracle fed the same inputs) and end to
end.  Full-size workloads are compared on a sample of tokens that the oracle
computes one routed pair at a time, with the same launch configuration the
bench times.
"""
import numpy as np
import pytest
import torch

import inputs
import oracle
from gpu_util import bf16_from_bits, bits_of_bf16, f64_of_bf16, gcorr_of, rel_fro, to_dev
from helpers import moe_experts, moe_host_inputs

pytestmark = pytest.mark.gpu


def _device_weights(lib, seed, cfg):
    H, I, E = cfg["H"], cfg["I"], cfg["E"]
    return (lib.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W13, (E, 2 * I, H // 2))),
            inputs.gpu_scales(seed, inputs.STREAM_W13_SCALE, (E, H // 128, 2 * I)),
            lib.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W2, (E, H, I // 2))),
            inputs.gpu_scales(seed, inputs.STREAM_W2_SCALE, (E, I // 128, H)))


def _run_layer(lib, seed, cfg, x_bits=None, logits=None):
    if x_bits is None:
        x_bits, logits = moe_host_inputs(seed, cfg)
    T, H, I, E, k = (cfg[n] for n in ("T", "H", "I", "E", "k"))
    w13, w13s, w2, w2s = _device_weights(lib, seed, cfg)
    L = lib.moe_workspace_layout(T, H, I, E, k)
    ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
    out = lib.w4a8_moe_forward(bf16_from_bits(x_bits), to_dev(logits), k, w13, w13s, w2, w2s, ws=ws)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out, ws, L, x_bits, logits


def _ws_view(ws, off, dtype, shape):
    n = int(np.prod(shape))
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).reshape(shape).cpu()


@pytest.mark.parametrize("name,cfg", [
    ("tiny", inputs.WORKLOADS["tiny"]),
    ("tiny-k1", dict(T=33, H=256, I=256, E=4, k=1)),
    ("one-token", dict(T=1, H=384, I=256, E=16, k=4)),
    ("k-equals-E", dict(T=20, H=128, I=128, E=3, k=3)),
    ("many-experts", dict(T=200, H=512, I=384, E=160, k=6)),
    ("prefill-tiles", dict(T=700, H=256, I=256, E=4, k=2)),
    ("wide-two-stages", dict(T=600, H=512, I=256, E=4, k=2)),
    ("expert-limit", dict(T=300, H=256, I=128, E=1024, k=8)),  # the largest expert count the layer takes
])
def test_layer_stage_by_stage(lib, name, cfg):
    seed = 3
    out, ws, L, x_bits, logits = _run_layer(lib, seed, cfg)
    T, H, I, E, k = (cfg[n] for n in ("T", "H", "I", "E", "k"))
    P = T * k
    w13h, w2h = moe_experts(seed, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    ld = L.scale_ld
    # (1) routing: ids exact, weights 1e-6
    ids = _ws_view(ws, L.topk_ids, torch.int32, (T, k)).numpy()
    tw = _ws_view(ws, L.topk_w, torch.float32, (T, k)).numpy()
    rid, rw = oracle.route_topk(logits, k)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(tw - rw) / rw) <= 1e-6
    # (2) permutation: exact
    seg = _ws_view(ws, L.seg_indptr, torch.int64, (E + 1,)).numpy()
    s2d = _ws_view(ws, L.src2dst, torch.int32, (P,)).numpy()
    d2s = _ws_view(ws, L.dst2src, torch.int32, (P,)).numpy()
    rseg, rs2d, rd2s = oracle.permute(rid, E)
    assert np.array_equal(seg, rseg) and np.array_equal(s2d, rs2d) and np.array_equal(d2s, rd2s)
    # (3) quantised permuted activations: exact
    xq = _ws_view(ws, L.xq, torch.uint8, (P, H)).numpy()
    xs = _ws_view(ws, L.xs, torch.float32, (H // 128, ld)).numpy()[:, :P].T
    xc = _ws_view(ws, L.xc, torch.float32, (H // 128, ld)).numpy()[:, :P].T
    rq, rs = oracle.quant_per_token_group(x)
    tok = rd2s // k
    assert np.array_equal(xq, rq[tok]) and np.array_equal(xs, rs[tok])
    assert np.array_equal(xc, gcorr_of(xq, xs))  # exact code sums, then one fp32 product
    # (4) w13 on the device's own inputs (identical to the oracle's): 1e-3
    ry13 = oracle.round_bf16(oracle.grouped_gemm(xq, xs, seg, w13h.w, w13h.s))
    y13 = _ws_view(ws, L.y13, torch.bfloat16, (P, 2 * I)).float().numpy().astype(np.float64)
    assert rel_fro(y13, ry13) <= 1e-3
    # (5) SiLU-and-Mul requant of the device's Y13
    hq = _ws_view(ws, L.hq, torch.uint8, (P, I)).numpy()
    hs = _ws_view(ws, L.hs, torch.float32, (I // 128, ld)).numpy()[:, :P].T
    hc = _ws_view(ws, L.hc, torch.float32, (I // 128, ld)).numpy()[:, :P].T
    assert np.array_equal(hc, gcorr_of(hq, hs))
    rhq, rhs = oracle.silu_mul_requant(y13)
    assert (hq != rhq).mean() <= 1e-3
    assert rel_fro(oracle.dequant(hq, hs), oracle.dequant(rhq, rhs)) <= 1e-3
    # (6) w2 on the device's Hq: 1e-3
    y2 = _ws_view(ws, L.y2, torch.bfloat16, (P, H)).float().numpy().astype(np.float64)
    ry2 = oracle.round_bf16(oracle.grouped_gemm(hq, hs, seg, w2h.w, w2h.s))
    assert rel_fro(y2, ry2) <= 1e-3
    # (7) combine of the device's Y2: 1e-3
    rout_stage = oracle.round_bf16(oracle.unpermute_combine(y2, s2d, tw.astype(np.float64), T, k))
    got = f64_of_bf16(out)
    assert rel_fro(got, rout_stage) <= 1e-3
    # end to end against the oracle's own chain: 2e-2
    ref = oracle.moe_layer(x, logits, k, w13h.w, w13h.s, w2h.w, w2h.s)["out"]
    err = rel_fro(got, ref)
    print(f"{name}: end-to-end rel Frobenius {err:.2e}, max abs {np.abs(got - ref).max():.3e}")
    assert err <= 2e-2
    assert np.all(np.isfinite(got))


def test_layer_zero_and_huge_rows(lib):
    cfg = dict(T=16, H=256, I=256, E=4, k=2)
    x_bits, logits = moe_host_inputs(5, cfg)
    x = inputs.bf16_bits_to_f32(x_bits).copy()
    x[0] = 0.0
    x[1] *= 1e4
    x_bits = inputs.to_bf16_bits(x)
    out, ws, L, _, _ = _run_layer(lib, 5, cfg, x_bits, logits)
    w13h, w2h = moe_experts(5, cfg)
    ref = oracle.moe_layer(inputs.bf16_bits_to_f32(x_bits), logits, 2, w13h.w, w13h.s, w2h.w, w2h.s)["out"]
    got = f64_of_bf16(out)
    assert np.all(np.isfinite(got)) and np.all(got[0] == 0)
    assert rel_fro(got, ref) <= 2e-2


# Full-size workloads in the bench's launch configuration.  decode: every token; prefill and skewed: a
# seeded sample of 256 tokens holding the first and last token (and, for the skewed routing, tokens of the
# hottest expert and of the nearly empty ones).  For every routed pair of a sampled token the device's
# Y13 and Y2 rows are compared with the oracle's GEMM of the same rows at the stage tolerance (1e-3), its
# Hq codes with the oracle's requantisation of its Y13 (the c15 gate), and the layer output with the
# oracle's own chain at the end-to-end tolerance (2e-2).  Routing ids and the permutation are compared
# for all tokens, bit for bit.
@pytest.mark.parametrize("name,n", [("decode", 64), ("prefill", 256), ("skewed", 256)])
def test_full_size_sampled_tokens(lib, name, n):
    import fullsize
    cfg = inputs.WORKLOADS[name]
    T, H, I, E, k = (cfg[c] for c in ("T", "H", "I", "E", "k"))
    P = T * k
    out, ws, L, x_bits, logits = _run_layer(lib, 0, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    allout = f64_of_bf16(out)
    assert np.all(np.isfinite(allout))
    rid, _ = oracle.route_topk(logits, k)
    assert np.array_equal(_ws_view(ws, L.topk_ids, torch.int32, (T, k)).numpy(), rid)
    rseg, rs2d, rd2s = oracle.permute(rid, E)
    seg = _ws_view(ws, L.seg_indptr, torch.int64, (E + 1,)).numpy()
    s2d = _ws_view(ws, L.src2dst, torch.int32, (P,)).numpy()
    d2s = _ws_view(ws, L.dst2src, torch.int32, (P,)).numpy()
    assert np.array_equal(seg, rseg) and np.array_equal(s2d, rs2d) and np.array_equal(d2s, rd2s)
    extra = ()
    if cfg.get("zipf"):
        extra, hot, cold = fullsize.skew_extremes(rid, E)
        counts = np.diff(seg)
        print(f"{name}: hottest expert {hot} ({counts[hot]} rows), coldest used {cold} "
              f"({counts[cold].tolist()} rows), {np.count_nonzero(counts == 0)} empty experts")
    sample = fullsize.pick_tokens(T, max(n, len(extra) + 2), 1234, rid, E, extra)
    pairs = (sample[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    r_idx = torch.from_numpy(s2d[pairs].astype(np.int64)).cuda()
    ld = L.scale_ld

    def rows_of(off, dtype, width):
        n_el = P * width
        t = ws[off:off + n_el * torch.tensor([], dtype=dtype).element_size()].view(dtype).view(P, width)
        return t.index_select(0, r_idx).cpu()

    def scale_rows(off, G):
        t = ws[off:off + G * ld * 4].view(torch.float32).view(G, ld)
        return t.index_select(1, r_idx).t().contiguous().cpu().numpy()

    rows = dict(xq=rows_of(L.xq, torch.uint8, H).numpy(), xs=scale_rows(L.xs, H // 128),
                y13=rows_of(L.y13, torch.bfloat16, 2 * I).float().numpy().astype(np.float64),
                hq=rows_of(L.hq, torch.uint8, I).numpy(), hs=scale_rows(L.hs, I // 128),
                y2=rows_of(L.y2, torch.bfloat16, H).float().numpy().astype(np.float64))
    # quantised rows of the sampled pairs: exact against the oracle's quantisation of the tokens
    rq, rs = oracle.quant_per_token_group(x[sample])
    tok = np.repeat(np.arange(sample.size), k)
    assert np.array_equal(rows["xq"], rq[tok]) and np.array_equal(rows["xs"], rs[tok])
    stats, out_ref = fullsize.sampled_layer_check(0, cfg, sample, logits, rows)
    got = allout[sample]
    err = rel_fro(got, out_ref)
    print(f"{name}: {sample.size} tokens ({pairs.size} pairs): w13 {stats['y13']:.2e}, w2 {stats['y2']:.2e}, "
          f"SiLU codes differing {stats['hq_mismatch']:.2e} (dequantised {stats['hq_deq']:.2e}), "
          f"end to end {err:.2e}, max abs {np.abs(got - out_ref).max():.3e}")
    assert stats["y13"] <= 1e-3 and stats["y2"] <= 1e-3
    assert stats["hq_mismatch"] <= 1e-3 and stats["hq_deq"] <= 1e-3
    assert err <= 2e-2
    assert lib.device_error() == 0


def test_layer_on_a_second_device(lib):
    # Launch attributes (the GEMM's and permutation's shared-memory limits) are per device: the layer must
    # also run on a device other than the first one the process used.
    if torch.cuda.device_count() < 2:
        pytest.skip("one CUDA device")
    cfg = dict(T=300, H=256, I=256, E=4, k=2)
    x_bits, logits = moe_host_inputs(4, cfg)
    w13h, w2h = moe_experts(4, cfg)
    ref = oracle.moe_layer(inputs.bf16_bits_to_f32(x_bits), logits, 2, w13h.w, w13h.s, w2h.w, w2h.s)["out"]
    for d in (0, 1):
        with torch.cuda.device(d):
            out, _, _, _, _ = _run_layer(lib, 4, cfg, x_bits, logits)
            assert rel_fro(f64_of_bf16(out), ref) <= 2e-2
