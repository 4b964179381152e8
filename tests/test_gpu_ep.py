"""GPU parity of the expert-parallel shard mode (expert_map; pairs of remote experts skipped).

The permutation is compared bit for bit with the oracle's; quantisation and combine are checked on
the rows and slots the shard leaves out; the layer forward of a shard is compared with the oracle's
shard layer, stage by stage on small workloads and on sampled tokens of the full prefill shape split
over 8 shards.
"""
import numpy as np
import pytest
import torch

import inputs
import oracle
from gpu_util import bf16_from_bits, bf16_ulp_diff, bits_of_bf16, f64_of_bf16, rel_fro, to_dev
from helpers import moe_experts, moe_host_inputs
from test_gpu_layer import _device_weights, _ws_view

pytestmark = pytest.mark.gpu


def _shard_map(E, experts):
    emap = np.full(E, -1, np.int32)
    emap[np.asarray(experts)] = np.arange(len(experts), dtype=np.int32)
    return emap


def _distinct_ids(rng, T, E, k):
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


# below 8192 pairs one CTA, from 8192 the count + placement passes
@pytest.mark.parametrize("T,E,k,kind", [(5, 8, 2, "half"), (64, 256, 8, "strided"), (1000, 384, 8, "shuffled"),
                                        (1024, 256, 8, "strided"), (8192, 256, 8, "strided"),
                                        (4096, 1024, 8, "shuffled"), (3001, 7, 3, "half"), (300, 16, 4, "none"),
                                        (300, 16, 4, "all")])
def test_permute_ep(lib, T, E, k, kind):
    rng = np.random.default_rng(T + E + k)
    ids = _distinct_ids(rng, T, E, k)
    if kind == "half":
        experts = list(range(E // 2, E))
    elif kind == "strided":
        experts = list(range(3, E, 8))
    elif kind == "shuffled":
        experts = list(rng.permutation(E)[: E // 3])
    elif kind == "all":
        experts = list(rng.permutation(E))
    else:  # no local expert is routed to: map with one local id that nobody uses
        used = set(ids.reshape(-1).tolist())
        experts = [e for e in range(E) if e not in used][:1] or [E - 1]
        ids[ids == experts[0]] = (experts[0] + 1) % E if len(experts) else 0
    emap = _shard_map(E, experts)
    EL = len(experts)
    seg, s2d, d2s = lib.moe_permute_ep(to_dev(ids), E, to_dev(emap), EL)
    rs, rs2d, rd2s = oracle.permute(ids, E, emap)
    assert np.array_equal(seg.cpu().numpy(), rs)
    assert np.array_equal(s2d.cpu().numpy(), rs2d)
    d = d2s.cpu().numpy()
    PL = int(rs[-1])
    assert np.array_equal(d[:PL], rd2s) and np.all(d[PL:] == -1)
    assert lib.device_error() == 0


def test_permute_ep_flags_bad_map_entries(lib):
    ids = np.array([[0, 1], [2, 3]], np.int32)
    emap = np.array([0, 5, -1, 1], np.int32)  # 5 is out of range for E_local = 2
    seg, s2d, d2s = lib.moe_permute_ep(to_dev(ids), 4, to_dev(emap), 2)
    torch.cuda.synchronize()
    assert lib.device_error() == 2
    assert s2d.cpu().numpy()[1] == -1  # the pair is left out
    assert seg.cpu().numpy().tolist() == [0, 1, 2]


def test_quant_gather_leaves_negative_rows(lib):
    rng = np.random.default_rng(2)
    M, K = 40, 512
    x_bits = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    row_index = np.concatenate([rng.permutation(M)[:25], -np.ones(7)]).astype(np.int32)
    m_out = row_index.size
    ld = lib.scale_ld(m_out)
    q = torch.full((m_out, K), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((K // 128, ld), 7.0, dtype=torch.float32, device="cuda")
    c = torch.full((K // 128, ld), 9.0, dtype=torch.float32, device="cuda")
    x = bf16_from_bits(x_bits)
    rc = lib.load().fp8_quant_per_token_group(x.data_ptr(), M, K, to_dev(row_index).data_ptr(), 1, m_out,
                                               q.data_ptr(), s.data_ptr(), c.data_ptr(), ld,
                                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    rq, rsc = oracle.quant_per_token_group(inputs.bf16_bits_to_f32(x_bits))
    gq = q.cpu().numpy()
    gs = s.cpu().numpy()
    assert np.array_equal(gq[:25], rq[row_index[:25]])
    assert np.array_equal(gs[:, :25].T, rsc[row_index[:25]])
    assert np.all(gq[25:] == 0xAB) and np.all(gs[:, 25:m_out] == 7.0) and np.all(c.cpu().numpy()[:, 25:m_out] == 9.0)


@pytest.mark.parametrize("T,k,H", [(1, 1, 8), (64, 8, 7168), (300, 2, 256)])
def test_combine_skips_remote_slots(lib, T, k, H):
    rng = np.random.default_rng(T + k)
    P = T * k
    yb = inputs.to_bf16_bits(rng.standard_normal((P, H)).astype(np.float32))
    s2d = rng.permutation(P).astype(np.int32)
    s2d[rng.random(P) < 0.6] = -1
    if T > 1:
        s2d[:k] = -1  # a token with no local slot
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    out = lib.moe_unpermute_combine(bf16_from_bits(yb), to_dev(s2d), to_dev(w))
    ref = oracle.round_bf16(oracle.unpermute_combine(inputs.bf16_bits_to_f32(yb), s2d, w, T, k))
    got = f64_of_bf16(out)
    if T > 1:
        assert np.all(got[0] == 0)
    # the kernel sums in fp32 (slot order) and rounds to bf16, the oracle sums in float64 and rounds: the
    # two bf16 roundings are at most 2^-7 |ref| apart, plus the fp32 accumulation error, below
    # 2k * 2^-24 * sum_j |w_j y_j| (one rounding per fused step; two for a plain multiply-add)
    absum = oracle.unpermute_combine(np.abs(inputs.bf16_bits_to_f32(yb)), s2d, np.abs(w), T, k)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 2 * k * 2.0 ** -24 * absum)
    ulp = bf16_ulp_diff(bits_of_bf16(out), oracle.bf16_bits(ref))
    assert (ulp > 1).mean() <= 1e-4
    assert rel_fro(got, ref) <= 1e-3


def _run_shard(lib, seed, cfg, experts, x_bits=None, logits=None):
    if x_bits is None:
        x_bits, logits = moe_host_inputs(seed, cfg)
    T, H, I, E, k = (cfg[n] for n in ("T", "H", "I", "E", "k"))
    w13, w13s, w2, w2s = _device_weights(lib, seed, cfg)
    idx = torch.tensor(experts, dtype=torch.int64, device="cuda")
    w13, w13s, w2, w2s = (t.index_select(0, idx).contiguous() for t in (w13, w13s, w2, w2s))
    emap = _shard_map(E, experts)
    L = lib.moe_workspace_layout(T, H, I, E, k)
    ws = torch.zeros(L.total, dtype=torch.uint8, device="cuda")
    out = lib.w4a8_moe_forward_ep(bf16_from_bits(x_bits), to_dev(logits), k, to_dev(emap), w13, w13s, w2, w2s,
                                  ws=ws)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    return out, ws, L, x_bits, logits, emap


@pytest.mark.parametrize("name,cfg,experts", [
    ("tiny-shard", inputs.WORKLOADS["tiny"], [5, 0, 2]),
    ("tiny-one", inputs.WORKLOADS["tiny"], [7]),
    ("many-experts", dict(T=200, H=512, I=384, E=160, k=6), list(range(1, 160, 4))),
    ("prefill-tiles", dict(T=700, H=256, I=256, E=4, k=2), [1, 3]),
])
def test_layer_shard_stage_by_stage(lib, name, cfg, experts):
    seed = 4
    out, ws, L, x_bits, logits, emap = _run_shard(lib, seed, cfg, experts)
    T, H, I, E, k = (cfg[n] for n in ("T", "H", "I", "E", "k"))
    w13h, w2h = moe_experts(seed, cfg)
    g = list(experts)
    x = inputs.bf16_bits_to_f32(x_bits)
    ref = oracle.moe_layer(x, logits, k, lambda l: w13h.w(g[l]), lambda l: w13h.s(g[l]), lambda l: w2h.w(g[l]),
                           lambda l: w2h.s(g[l]), expert_map=emap)
    EL = len(experts)
    seg = _ws_view(ws, L.seg_indptr, torch.int64, (EL + 1,)).numpy()
    assert np.array_equal(seg, ref["seg"])
    assert np.array_equal(_ws_view(ws, L.src2dst, torch.int32, (T * k,)).numpy(), ref["src2dst"])
    PL = int(seg[-1])
    d2s = _ws_view(ws, L.dst2src, torch.int32, (T * k,)).numpy()
    assert np.array_equal(d2s[:PL], ref["dst2src"]) and np.all(d2s[PL:] == -1)
    got = f64_of_bf16(out)
    err = rel_fro(got, ref["out"]) if np.any(ref["out"]) else float(np.abs(got).max())
    print(f"{name}: {PL} of {T * k} pairs local, end-to-end rel Frobenius {err:.2e}")
    assert err <= 2e-2
    assert np.all(np.isfinite(got))
    nolocal = np.all(ref["src2dst"].reshape(T, k) < 0, axis=1)
    assert np.all(got[nolocal] == 0)


def test_shards_add_up_on_the_gpu(lib):
    # every token's shard outputs sum (in float64, before each shard's bf16 rounding differs) to within a few
    # bf16 ulps of the whole layer's output
    cfg = dict(T=96, H=256, I=256, E=8, k=3)
    seed = 6
    x_bits, logits = moe_host_inputs(seed, cfg)
    from test_gpu_layer import _run_layer
    full, *_ = _run_layer(lib, seed, cfg, x_bits, logits)
    total = np.zeros((cfg["T"], cfg["H"]))
    for experts in ([0, 3, 6], [1, 4, 7], [2, 5]):
        part, *_ = _run_shard(lib, seed, cfg, experts, x_bits, logits)
        total += f64_of_bf16(part)
    assert rel_fro(total, f64_of_bf16(full)) <= 1e-2


def test_full_prefill_shard_sampled_tokens(lib):
    # the prefill shape (T=8192, E=256, top-8) split over 8 shards; shard 3 holds experts 3, 11, 19, ...
    cfg = inputs.WORKLOADS["prefill"]
    experts = list(range(3, cfg["E"], 8))
    out, ws, L, x_bits, logits, emap = _run_shard(lib, 0, cfg, experts)
    sample = [0, 1, 4095, 8191]
    w13h, w2h = moe_experts(0, cfg)
    g = experts
    x = inputs.bf16_bits_to_f32(x_bits)
    ref, _, _ = oracle.moe_tokens(x[sample], logits[sample], cfg["k"], lambda l: w13h.w(g[l]),
                                  lambda l: w13h.s(g[l]), lambda l: w2h.w(g[l]), lambda l: w2h.s(g[l]),
                                  expert_map=emap)
    got = f64_of_bf16(out)[sample]
    err = rel_fro(got, ref)
    print(f"prefill shard 3 of 8: sampled tokens {sample}: rel Frobenius {err:.2e}")
    assert err <= 2e-2
    rs, rs2d, rd2s = oracle.permute(oracle.route_topk(logits, cfg["k"])[0], cfg["E"], emap)
    assert np.array_equal(_ws_view(ws, L.seg_indptr, torch.int64, (len(experts) + 1,)).numpy(), rs)
    assert np.array_equal(_ws_view(ws, L.src2dst, torch.int32, (cfg["T"] * cfg["k"],)).numpy(), rs2d)


@pytest.mark.parametrize("M,I,m", [(50, 256, 30), (700, 2048, 699), (64, 128, 0)])
def test_silu_rows_stops_at_device_count(lib, M, I, m):
    # rows below the device-side count are what silu_mul_requant (parity-tested against the oracle) gives;
    # rows from it on are left as they were
    rng = np.random.default_rng(M + I + m)
    gu = bf16_from_bits(inputs.to_bf16_bits(rng.standard_normal((M, 2 * I)).astype(np.float32) * 4))
    fq, fs, fc = lib.silu_mul_requant(gu)
    ld = lib.scale_ld(M)
    q = torch.full((M, I), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((I // 128, ld), 7.0, dtype=torch.float32, device="cuda")
    c = torch.full((I // 128, ld), 9.0, dtype=torch.float32, device="cuda")
    m_dev = torch.tensor([m], dtype=torch.int64, device="cuda")
    rc = lib.load().silu_mul_requant_rows(gu.data_ptr(), M, m_dev.data_ptr(), I, q.data_ptr(), s.data_ptr(),
                                          c.data_ptr(), ld, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(q[:m], fq[:m]) and torch.equal(s[:, :m], fs[:, :m]) and torch.equal(c[:, :m], fc[:, :m])
    assert bool((q[m:] == 0xAB).all()) and bool((s[:, m:M] == 7.0).all()) and bool((c[:, m:M] == 9.0).all())
