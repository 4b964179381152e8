"""Host logic of bench.py (no GPU): workload parsing, algorithmic work counts, the roofline choice, launch
counts, clock-record parsing and the DRAM-traffic lookup.

The counts are pinned to closed forms written out here from the shapes: an int4 weight is half a byte, a
per-128 fp32 scale adds 4/128 bytes per weight, so a DeepSeek-V3-shaped expert (H = 7168, I = 2048: 3·I·H
weights over w13 and w2) holds 3·I·H·(1/2 + 4/128) = 23.40 MB; the ridge of the dense Linear lies where
its bytes per FLOP meet the bandwidth / peak ratio."""
import json
import os

import numpy as np
import pytest

import bench
import inputs


def test_named_workloads_parse():
    for name in ("tiny", "decode", "prefill", "skewed"):
        got, cfg = bench.get_workload(name)
        assert got == name
        assert cfg == inputs.WORKLOADS[name]
    name, cfg = bench.get_workload("decode")
    assert (cfg["T"], cfg["H"], cfg["I"], cfg["E"], cfg["k"]) == (64, 7168, 2048, 256, 8)


def test_custom_shard_and_linear_workloads_parse():
    assert bench.get_workload("moe:128,256,512,8,2") == ("moe", dict(T=128, H=256, I=512, E=8, k=2, zipf=None))
    name, cfg = bench.get_workload("ep:prefill:8:3")
    assert name == "ep-prefill" and cfg["ep"] == (8, 3) and cfg["T"] == inputs.WORKLOADS["prefill"]["T"]
    assert "ep" not in inputs.WORKLOADS["prefill"]  # the named workload is copied, not modified
    assert bench.get_workload("linear:16,7168,2048") == ("linear", dict(M=16, N=7168, K=2048))
    with pytest.raises(KeyError):
        bench.get_workload("no-such-workload")


def test_workload_descriptions_state_the_shapes():
    d = bench.workload_desc("decode", inputs.WORKLOADS["decode"])
    assert "T=64" in d and "H=7168" in d and "E=256" in d and "top-8" in d
    _, cfg = bench.get_workload("ep:decode:8:3")
    assert "shard 3 of 8" in bench.workload_desc("ep-decode", cfg)
    assert bench.workload_desc("linear", dict(M=1, N=2, K=128)) == "dense W4AFP8 Linear M=1 N=2 K=128"


def test_expert_bytes_and_layer_flops_closed_forms():
    H, I, E, k = 7168, 2048, 256, 8
    per_expert = 3 * I * H * (0.5 + 4 / 128)
    assert per_expert == pytest.approx(23.40e6, rel=1e-3)
    c = bench.moe_counts(64, H, I, E, k, 64 * k, 1)
    assert c["layer_bytes"] - (64 * H * 2 * 2 + 64 * E * 4) == pytest.approx(per_expert, rel=0, abs=0)
    # all 256 experts: 5.99 GB of weights
    c = bench.moe_counts(0, H, I, E, k, 0, E)
    assert c["layer_bytes"] == pytest.approx(5.99e9, rel=1e-3)
    assert c["flops"] == 0 and c["w13_flops"] == 0
    # prefill: 8192 tokens x 8 pairs x 3 matrices of I x H, two FLOPs per multiply-add
    c = bench.moe_counts(8192, H, I, E, k, 8192 * k, E)
    assert c["flops"] == pytest.approx(2 * 65536 * 3 * I * H)
    assert c["flops"] / 1e12 == pytest.approx(5.77, rel=1e-3)
    assert c["w13_flops"] == pytest.approx(c["flops"] * 2 / 3)


def test_fused_w13_writes_h_instead_of_y13():
    H, I = 256, 512
    a = bench.moe_counts(4, H, I, 8, 2, 10, 3)
    b = bench.moe_counts(4, H, I, 8, 2, 10, 3, fused=True)
    # Y13 (2I bf16 per pair) replaced by I E4M3 codes + I/128 scales and corrections per pair
    assert a["w13_bytes"] - b["w13_bytes"] == 10 * (2 * I * 2 - I - 2 * (I // 128) * 4)
    assert a["w13_flops"] == b["w13_flops"] and a["flops"] == b["flops"]


def test_w13_bytes_add_activation_traffic_per_pair():
    H, I = 256, 512
    base = bench.moe_counts(4, H, I, 8, 2, 0, 3)["w13_bytes"]
    one = bench.moe_counts(4, H, I, 8, 2, 1, 3)["w13_bytes"]
    # one more pair: H codes + H/128 fp32 scales read, 2I bf16 outputs written
    assert one - base == H + (H // 128) * 4 + 2 * I * 2
    assert base == 3 * (2 * I * H // 2 + 2 * I * (H // 128) * 4)


def test_expected_touched_experts_of_the_decode_shape():
    # 64 tokens x top-8 of 256 experts: an expert is missed by one token with probability 1 - 8/256 = 31/32
    touched = 256 * (1 - (31 / 32) ** 64)
    assert touched == pytest.approx(222.4, abs=0.05)
    c = bench.moe_counts(64, 7168, 2048, 256, 8, 512, touched)
    assert c["layer_bytes"] / 1e9 == pytest.approx(5.20, abs=0.01)


def test_linear_counts_and_ridge():
    c = bench.linear_counts(1, 7168, 2048)
    assert c["flops"] == 2 * 7168 * 2048
    assert c["bytes"] == 7168 * 1024 + 7168 * 16 * 4 + 2048 + 16 * 4 + 7168 * 2
    # ridge: the M at which bytes / 6.8 TB/s equals FLOPs / 3.4 PFLOP/s, about 160-170 rows at these widths
    hbm, peak = 6806.2, 2 * 1710.9

    def bound(M):
        c = bench.linear_counts(M, 18432, 7168)
        return bench.roofline_core(c["bytes"], c["flops"], 1.0, hbm, peak)["bound"]
    assert bound(128) == "hbm" and bound(1024) == "tensor"
    ridge = next(M for M in range(1, 4096) if bound(M) == "tensor")
    assert 120 <= ridge <= 220


def test_roofline_core_picks_the_larger_bound():
    # 1 GB in 1 ms = 1000 GB/s; 1 TFLOP in 1 ms = 1000 TFLOP/s
    r = bench.roofline_core(1e9, 1e9, 1.0, 2000.0, 4000.0)
    assert r == {"bound": "hbm", "achieved": 1000.0, "peak": 2000.0, "unit": "GB/s", "frac": 0.5}
    r = bench.roofline_core(1e6, 1e12, 1.0, 2000.0, 4000.0)
    assert r == {"bound": "tensor", "achieved": 1000.0, "peak": 4000.0, "unit": "TFLOP/s", "frac": 0.25}
    # equal times: the HBM bound is taken
    assert bench.roofline_core(2e9, 4e12, 1.0, 2000.0, 4000.0)["bound"] == "hbm"


def test_launch_counts():
    # seven stages; the permutation's count pass from 8192 pairs; one more launch per split GEMM plan
    assert bench.moe_launches_per_step(7, False, [1, 1]) == 7
    assert bench.moe_launches_per_step(7, True, [2, 2]) == 8
    assert bench.moe_launches_per_step(7, True, [3, 3]) == 10
    assert bench.moe_launches_per_step(7, False, [3, 2]) == 8


def test_throughput_is_whole_job():
    assert bench.throughput(640, 2, 20.0) == pytest.approx(64000.0)
    assert bench.throughput(64, 1, 1.0) == pytest.approx(64000.0)


def _sampler_with(tmp_path, lines, uuid="GPU-a"):
    s = bench.ClockSampler(uuid)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = object()  # a sampler that ran
    return s


def test_clock_summary_median_reasons_and_device_filter(tmp_path):
    na = "Not Active"
    lines = [
        f"0, GPU-a, 2070, 2070, 900.5, 0x0, {na}, {na}, {na}, {na}",
        f"0, GPU-a, 1950, 2070, 1380.0, 0x4, {na}, {na}, {na}, Active",
        f"0, GPU-a, 2070, 2070, 1000.0, 0x0, {na}, {na}, {na}, {na}",
        f"1, GPU-b, 300, 2070, 100.0, 0x8, Active, {na}, {na}, {na}",  # another GPU: ignored
        "garbage line",
    ]
    s = _sampler_with(tmp_path, lines).summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["samples"] == 3 and s["power_w_max"] == 1380.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_tolerates_missing_power_and_no_samples(tmp_path):
    na = "Not Active"
    s = _sampler_with(tmp_path, [f"0, GPU-a, 2070, 2070, [N/A], 0x0, {na}, {na}, {na}, {na}"]).summary()
    assert s["sm_mhz"] == 2070.0 and s["power_w_max"] is None and s["reasons"] == []
    assert _sampler_with(tmp_path, ["nothing here"]).summary() is None
    s = bench.ClockSampler("GPU-a")
    assert s.summary() is None  # nvidia-smi never started


def test_traffic_lookup_is_keyed_by_the_gemm_source(monkeypatch, tmp_path):
    p = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(p) as f:
        d = json.load(f)
    key = next(kk for kk, v in d.items() if isinstance(v, dict) and "bytes_per_launch" in v)
    ent = d[key]
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: ent["source_hash"])
    assert bench.ncu_traffic(key) == ent["bytes_per_launch"]
    assert bench.ncu_traffic("no-such-launch") is None
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic(key) is None  # counters of an older kernel are not reported


def test_gemm_source_hash_covers_the_kernel_sources():
    h = bench.gemm_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0


def test_peaks_file_has_the_fields_the_bench_reads():
    peaks, src = bench.load_peaks()
    for f in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
        assert peaks[f] > 0
    assert src in ("measured", "fallback")


def test_default_cpu_sample_sizes():
    assert bench.default_cpu_tokens("tiny") == 64
    assert bench.default_cpu_tokens("decode") == 1
    assert bench.default_cpu_tokens("ep-prefill") == 1
    assert np.isfinite(bench.throughput(1, 1, 1.0))


class _FakeNvml:
    """Stands in for libnvidia-ml: fixed clocks and power, a reason bitmask that changes per call."""

    def __init__(self, reasons):
        self.reasons = list(reasons)
        self.calls = 0

    def nvmlInit_v2(self):
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, handle):
        return 0 if uuid == b"GPU-x" else 1

    def nvmlDeviceGetMaxClockInfo(self, h, kind, out):
        out._obj.value = 2070
        return 0

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        out._obj.value = 1900 + 10 * (self.calls % 3)
        return 0

    def nvmlDeviceGetPowerUsage(self, h, out):
        out._obj.value = 1200000 + 1000 * self.calls
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = self.reasons[self.calls % len(self.reasons)]
        self.calls += 1
        return 0


def test_nvml_sampler_with_a_fake_library():
    fake = _FakeNvml([0x0, 0x4, 0x1])  # idle and power cap bits; idle is not a throttle reason
    s = bench.NvmlSampler("GPU-x", period_s=0.001, nvml=fake)
    with s:
        pass
    out = s.summary()
    assert out["sm_max_mhz"] == 2070 and out["samples"] >= 2
    assert out["reasons"] == (["sw_power_cap"] if out["samples"] >= 2 else [])
    assert 1900 <= out["sm_mhz"] <= 1920 and out["power_w_max"] >= 1200.0
    with pytest.raises(OSError):
        bench.NvmlSampler("GPU-other", nvml=_FakeNvml([0]))


def test_clock_rows_summary_names_the_rejecting_reasons():
    rows = [(2070, 900.0, 0x0), (1800, 1400.0, 0x8 | 0x4), (1500, 1390.0, 0x40), (None, None, 0x20)]
    out = bench.summarize_clock_rows(rows, 2070, bench.NvmlSampler.REASONS)
    assert out["sm_mhz"] == 1800 and out["power_w_max"] == 1400.0 and out["samples"] == 4
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_oracle_over_host_cores_runs_rounds_together():
    # two spawn-started processes, one token each of the tiny layer, two rounds
    cfg = dict(inputs.WORKLOADS["tiny"])
    rounds, tokens, cores = bench.oracle_on_host_cores("tiny", cfg, 0, 1, 2, cores=2)
    assert len(rounds) == 2 and tokens == 2 and cores == 2
    assert all(0.0 < r < 60.0 for r in rounds)


def test_e2e_copies_and_pipelining_rule():
    # tiny: 32 KiB in, 2 KiB of logits, 32 KiB out -> copies in order; decode: 0.92 MiB of x + 64 KiB of
    # logits in, 0.88 MiB out -> overlapped with the layer; prefill likewise
    assert bench.e2e_bytes(64, 256, 8) == (64 * 256 * 2 + 64 * 8 * 4, 64 * 256 * 2)
    assert not bench.e2e_pipelined(*bench.e2e_bytes(64, 256, 8))
    assert bench.e2e_bytes(64, 7168, 256) == (983040, 917504)
    assert bench.e2e_pipelined(*bench.e2e_bytes(64, 7168, 256))
    assert bench.e2e_pipelined(*bench.e2e_bytes(8192, 7168, 256))
