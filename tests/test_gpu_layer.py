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
    assert np.allclose(xc, gcorr_of(xq, xs), rtol=1e-5, atol=1e-30)
    # (4) w13 on the device's own inputs (identical to the oracle's): 1e-3
    y13 = _ws_view(ws, L.y13, torch.bfloat16, (P, 2 * I)).float().numpy().astype(np.float64)
    ry13 = oracle.round_bf16(oracle.grouped_gemm(xq, xs, seg, w13h.w, w13h.s))
    assert rel_fro(y13, ry13) <= 1e-3
    # (5) SiLU-and-Mul requant of the device's Y13
    hq = _ws_view(ws, L.hq, torch.uint8, (P, I)).numpy()
    hs = _ws_view(ws, L.hs, torch.float32, (I // 128, ld)).numpy()[:, :P].T
    hc = _ws_view(ws, L.hc, torch.float32, (I // 128, ld)).numpy()[:, :P].T
    assert np.allclose(hc, gcorr_of(hq, hs), rtol=1e-5, atol=1e-30)
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


@pytest.mark.parametrize("name,sample", [("decode", [0, 17, 63]), ("prefill", [0, 4095]),
                                         ("skewed", [0, 2048])])
def test_full_size_sampled_tokens(lib, name, sample):
    cfg = inputs.WORKLOADS[name]
    out, ws, L, x_bits, logits = _run_layer(lib, 0, cfg)
    w13h, w2h = moe_experts(0, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    got = f64_of_bf16(out)[sample]
    ref, ids, _ = oracle.moe_tokens(x[sample], logits[sample], cfg["k"], w13h.w, w13h.s, w2h.w, w2h.s)
    err = rel_fro(got, ref)
    print(f"{name}: sampled tokens {sample}: rel Frobenius {err:.2e}, max abs {np.abs(got - ref).max():.3e}")
    assert err <= 2e-2
    # invariants over every token: finite, routing ids exact for all tokens
    allout = f64_of_bf16(out)
    assert np.all(np.isfinite(allout))
    rid, _ = oracle.route_topk(logits, cfg["k"])
    assert np.array_equal(_ws_view(ws, L.topk_ids, torch.int32, (cfg["T"], cfg["k"])).numpy(), rid)
