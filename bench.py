"""Benchmark of the W4AFP8 MoE layer (and the dense W4AFP8 Linear) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload decode|prefill|skewed|tiny|moe:T,H,I,E,k|ep:<workload>:R:r|linear:M,N,K]

One step = one pass of the whole hot path over one batch of synthetic input:
routing -> permutation -> FP8 quantisation (each token's row scattered to its
routed places) -> w13 grouped GEMM -> SiLU-and-Mul requantisation -> w2 grouped
GEMM -> combine, all through the C ABI (ep:...: one expert-parallel shard, the
pairs of experts r, r+R, ... only).  Prints one JSON line (rank 0).  Default workload: the DeepSeek-V3/R1-
shaped prefill layer (T=8192, H=7168, I=2048, E=256, top-8; 5.77 TFLOP per step, reported against the
FP8 tensor roofline), weights 6.0 GB (larger than L2, so every step streams them from HBM).  The same
line carries the decode layer (T=64, same experts, against the HBM roofline) under "decode", measured in
the same process on the same weights.

--impl reference times the CPU oracle (numpy, float64) over the host's cores (one process with one BLAS
thread per core, spawn-started) on a bounded sample of the same workload (a few tokens per core per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

if "--impl" in sys.argv and "reference" in sys.argv:
    for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import inputs  # noqa: E402

METRIC = "W4AFP8 MoE layer tokens/s + TFLOP/s on 1 GB300; % of HBM / FP8 roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="prefill: leave out the decode layer's keys")
    ap.add_argument("--fused-w13", action="store_true",
                    help="time w13 with the SiLU-and-Mul requantisation fused into its epilogue")
    ap.add_argument("--sustain-s", type=float, default=1.5,
                    help="seconds of untimed steps after the timed region with the clocks sampled (0: none)")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="tokens per oracle step (0: automatic)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")  # driver-written on the GPU pool
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def workload_desc(name, cfg):
    if name == "linear":
        return f"dense W4AFP8 Linear M={cfg['M']} N={cfg['N']} K={cfg['K']}"
    z = f", router logits + Zipf({cfg['zipf']}) bias" if cfg.get("zipf") else ""
    ep = ""
    if cfg.get("ep"):
        R, r = cfg["ep"]
        ep = (f"; expert-parallel shard {r} of {R} (experts {r}, {r + R}, ...; only the pairs routed to them, "
              f"tokens/s counts all T tokens of the shard's call)")
    return (f"{name} MoE layer: T={cfg['T']} H={cfg['H']} I={cfg['I']} E={cfg['E']} top-{cfg['k']}, "
            f"int4 weights + fp32 scales per 128 K, FP8 E4M3 activations per token per 128{z}{ep}")


def get_workload(spec):
    if spec.startswith("linear"):
        M, N, K = (int(v) for v in spec.split(":")[1].split(","))
        return "linear", dict(M=M, N=N, K=K)
    if spec.startswith("moe:"):  # moe:T,H,I,E,k  (custom shape, e.g. small profiling cases)
        T, H, I, E, k = (int(v) for v in spec.split(":")[1].split(","))
        return "moe", dict(T=T, H=H, I=I, E=E, k=k, zipf=None)
    if spec.startswith("ep:"):  # ep:<workload>:R:r  shard r of R (experts r, r+R, ...) of a named workload
        _, base, R, r = spec.split(":")
        cfg = dict(inputs.WORKLOADS[base])
        cfg["ep"] = (int(R), int(r))
        return f"ep-{base}", cfg
    return spec, dict(inputs.WORKLOADS[spec])


# ---------------------------------------------------------------------------
# clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"w4a8moe_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                rows.append(parts)
        if not rows:
            return None
        def num(v):  # nvidia-smi prints "[N/A]" for a field it cannot read
            return float(v) if v.replace(".", "", 1).isdigit() else None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[4]) for r in rows if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": num(rows[0][3]),
                "power_w_max": max(pw) if pw else None, "samples": len(rows), "reasons": reasons}


class NvmlSampler:
    """SM clock, power and clock-event reasons read through NVML (libnvidia-ml, read-only queries) every
    `period_s` seconds on a background thread while the timed region runs; summary() as ClockSampler's."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_slowdown"}

    def __init__(self, uuid, period_s=0.01, nvml=None):
        import ctypes
        self.uuid, self.period_s = uuid, period_s
        self.rows = []
        self.nv = nvml if nvml is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if not uuid or self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(self.nv.nvmlDeviceGetMaxClockInfo, 1)

    def _uint(self, fn, *args):
        import ctypes
        v = ctypes.c_uint()
        return v.value if fn(self.h, *args, ctypes.byref(v)) == 0 else None

    def sample(self):
        import ctypes
        r = ctypes.c_ulonglong()
        reasons = r.value if self.reasons_fn(self.h, ctypes.byref(r)) == 0 else 0
        pw = self._uint(self.nv.nvmlDeviceGetPowerUsage)
        self.rows.append((self._uint(self.nv.nvmlDeviceGetClockInfo, 1), None if pw is None else pw / 1e3,
                          reasons))

    def _loop(self):
        while not self.stop.wait(self.period_s):
            self.sample()

    def __enter__(self):
        import threading
        self.stop = threading.Event()
        self.sample()
        self.th = threading.Thread(target=self._loop, daemon=True)
        self.th.start()
        return self

    def __exit__(self, *a):
        self.stop.set()
        self.th.join()
        self.sample()

    def summary(self):
        return summarize_clock_rows(self.rows, self.max_mhz, self.REASONS)


def summarize_clock_rows(rows, max_mhz, reason_bits):
    """Median SM clock, peak power and the throttle reasons seen in (sm_mhz, power_w, reason bitmask) rows."""
    sm = [r[0] for r in rows if r[0] is not None]
    pw = [r[1] for r in rows if r[1] is not None]
    reasons = sorted({name for r in rows for bit, name in reason_bits.items() if r[2] & bit})
    return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max_mhz,
            "power_w_max": max(pw) if pw else None, "samples": len(rows), "reasons": reasons,
            "source": "NVML every 10 ms"}


def clock_sampler(dev):
    """NVML sampler when libnvidia-ml answers, else nvidia-smi every 200 ms."""
    try:
        return NvmlSampler(device_uuid(dev))
    except (OSError, AttributeError):
        return ClockSampler(device_uuid(dev))


def device_uuid(dev):
    try:
        import torch
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def gemm_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "w4afp8_mixture_experts_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary, if current."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(key)
    if not ent or ent.get("source_hash") != gemm_source_hash():
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: every rank runs the whole layer on its own batch)

def reduce_max(value: float, device) -> float:
    """Max over ranks of a per-rank time (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    return world * units_per_rank / (max_ms / 1e3)


# ---------------------------------------------------------------------------
# algorithmic work and rooflines (host arithmetic only)

def moe_counts(T, H, I, E, k, P, n_touched, fused=False):
    """Algorithmic work of one MoE layer step over P routed pairs, n_touched of the E experts holding any.

    FLOPs count the routed pairs only (no padding).  Bytes count the int4 weights and fp32 per-128 scales of
    the touched experts once, plus x and the router logits read and the output written.  The w13 launch
    reads its experts' weights and scales, the pairs' E4M3 codes and per-128 scales, and writes Y13 in bf16.
    """
    w13_w = n_touched * (2 * I * H // 2 + 2 * I * (H // 128) * 4)
    w2_w = n_touched * (H * I // 2 + H * (I // 128) * 4)
    # with SiLU-and-Mul fused into w13's epilogue the launch writes the requantised h (codes, scales and
    # corrections) instead of Y13
    out13 = P * I + 2 * (I // 128) * P * 4 if fused else P * 2 * I * 2
    return {"flops": 2.0 * P * (2 * I * H + I * H),
            "layer_bytes": w13_w + w2_w + T * H * 2 + T * E * 4 + T * H * 2,
            "w13_bytes": w13_w + P * H + (H // 128) * P * 4 + out13,
            "w13_flops": 2.0 * P * 2 * I * H}


def linear_counts(M, N, K):
    """Algorithmic work of one dense W4AFP8 Linear call: int4 weights + fp32 scales, E4M3 codes + scales of
    the M rows, bf16 output."""
    G = K // 128
    return {"flops": 2.0 * M * N * K, "bytes": N * K // 2 + N * G * 4 + M * K + M * G * 4 + M * N * 2}


def moe_launches_per_step(n_stages, two_pass_permute, gemm_plans):
    """Kernels one layer step launches: one per stage, plus the permutation's count pass from 8192 pairs,
    plus a second launch for each grouped GEMM whose plan (w4a8_grouped_gemm_plan: 1 narrow tiles, 2 wide
    tiles, 3 both over disjoint experts) is the split one."""
    return n_stages + (1 if two_pass_permute else 0) + sum(1 for p in gemm_plans if p == 3)


def w13_fuses(lib, pairs, experts, H):
    """Whether the layer's w13 launch carries the SiLU-and-Mul requantisation (the wide-tile plan with two or
    more stages of two 128-K groups per tile)."""
    import ctypes
    th = ctypes.c_int()
    G = H // 128
    gps = 2 if G % 2 == 0 else 1
    return int(lib.w4a8_grouped_gemm_plan(pairs, experts, H, ctypes.byref(th))) == 2 and G // gps >= 2


def gemm_plans(lib, pairs, experts, H, I):
    """The launch plans of the layer's w13 (K = H) and w2 (K = I) grouped GEMMs."""
    import ctypes
    th = ctypes.c_int()
    return [int(lib.w4a8_grouped_gemm_plan(pairs, experts, K, ctypes.byref(th))) for K in (H, I)]


def roofline_core(alg_bytes, flops, ms, hbm_gbs, tensor_tflops):
    """The bound that applies (the larger of bytes / bandwidth and FLOPs / peak) and the fraction of it that
    one launch of `ms` milliseconds reaches."""
    sec = ms / 1e3
    if alg_bytes / (hbm_gbs * 1e9) >= flops / (tensor_tflops * 1e12):
        ach = alg_bytes / sec / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(ach / hbm_gbs, 4)}
    ach = flops / sec / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": tensor_tflops, "unit": "TFLOP/s",
            "frac": round(ach / tensor_tflops, 4)}


# ---------------------------------------------------------------------------
# our implementation

class MoeRunner:
    """Device buffers of one MoE layer and the seven C-ABI calls of one step."""

    def __init__(self, cfg, seed, dev, weights=None):
        import torch

        import w4afp8_mixture_experts_gb300 as m
        self.m = m
        self.lib = m.load()
        self.dev = dev
        self.cfg = cfg
        T, H, I, E, k = (cfg[x] for x in ("T", "H", "I", "E", "k"))
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        if weights is not None:  # another workload's experts of the same shape (same seed)
            self.w13, self.w13s, self.w2, self.w2s = weights
        else:
            # weights are prepacked once after generation (the post-load processing step), untimed
            self.w13 = m.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W13, (E, 2 * I, H // 2),
                                                                     dev))
            self.w13s = inputs.gpu_scales(seed, inputs.STREAM_W13_SCALE, (E, H // 128, 2 * I), dev)
            self.w2 = m.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W2, (E, H, I // 2), dev))
            self.w2s = inputs.gpu_scales(seed, inputs.STREAM_W2_SCALE, (E, I // 128, H), dev)
        self.ep = cfg.get("ep")
        self.EL = E
        self.emap = None
        if self.ep:  # one expert-parallel shard: experts r, r+R, ... (local ids in that order)
            R, r = self.ep
            experts = list(range(r, E, R))
            idx = torch.tensor(experts, dtype=torch.int64, device=dev)
            self.w13, self.w13s, self.w2, self.w2s = (t.index_select(0, idx).contiguous()
                                                      for t in (self.w13, self.w13s, self.w2, self.w2s))
            emap = np.full(E, -1, np.int32)
            emap[experts] = np.arange(len(experts), dtype=np.int32)
            self.emap = torch.from_numpy(emap).to(dev)
            self.EL = len(experts)
        x_bits = inputs.activations_bf16(seed, T, H)
        logits = inputs.router_logits(seed, T, E, cfg.get("zipf"))
        self.x_pin = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        self.lg_pin = torch.from_numpy(logits).pin_memory()
        self.x = self.x_pin.to(dev)
        self.lg = self.lg_pin.to(dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.out_pin = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
        self.L = m.moe_workspace_layout(T, H, I, E, k)
        self.ws = torch.empty(self.L.total, dtype=torch.uint8, device=dev)
        b = self.ws.data_ptr()
        L = self.L
        self.p = {n: b + getattr(L, n) for n in ("topk_ids", "topk_w", "seg_indptr", "src2dst", "dst2src",
                                                 "xq", "xs", "xc", "y13", "hq", "hs", "hc", "y2", "permute_ws")}
        self.permute_ws_bytes = int(m.load().w4a8_workspace_bytes(1, T * k, 0, 0, self.EL))
        self.ld = L.scale_ld
        # --fused-w13: w13 through w4a8_grouped_gemm_silu, the SiLU-and-Mul requantisation in its epilogue where
        # the plan allows (w4a8_moe_forward keeps the separate kernel, which measured faster)
        self.fused = bool(cfg.get("fused_w13")) and (not self.ep) and w13_fuses(self.lib, T * k, E, H)

    def stages(self, stream):
        """The seven calls of one step, as closures (each returns a status)."""
        lib, p, T, H, I, E, k, ld = self.lib, self.p, self.T, self.H, self.I, self.E, self.k, self.ld
        P = T * k
        x, lg, out = self.x.data_ptr(), self.lg.data_ptr(), self.out.data_ptr()
        w13, w13s, w2, w2s = (t.data_ptr() for t in (self.w13, self.w13s, self.w2, self.w2s))
        if self.ep:  # the seven calls of w4a8_moe_forward_ep
            EL, emap = self.EL, self.emap.data_ptr()
            m_dev = p["seg_indptr"] + 8 * EL  # seg_indptr[E_local]: the shard's routed pairs
            return [
                ("route", lambda: lib.moe_route_topk(lg, T, E, k, 1, p["topk_ids"], p["topk_w"], stream)),
                ("permute", lambda: lib.moe_permute_ep(p["topk_ids"], T, k, E, emap, EL, p["seg_indptr"],
                                                       p["src2dst"], p["dst2src"], p["permute_ws"],
                                                       self.permute_ws_bytes, stream)),
                ("quant", lambda: lib.fp8_quant_scatter_per_token_group(x, T, H, p["src2dst"], k, P, p["xq"],
                                                                        p["xs"], p["xc"], ld, stream)),
                ("w13", lambda: lib.w4a8_grouped_gemm(p["xq"], p["xs"], p["xc"], ld, w13, w13s, p["seg_indptr"], EL,
                                                      2 * I, H, P, p["y13"], None, 0, stream)),
                ("silu_requant", lambda: lib.silu_mul_requant_rows(p["y13"], P, m_dev, I, p["hq"], p["hs"], p["hc"],
                                                                   ld, stream)),
                ("w2", lambda: lib.w4a8_grouped_gemm(p["hq"], p["hs"], p["hc"], ld, w2, w2s, p["seg_indptr"], EL, H,
                                                     I, P, p["y2"], None, 0, stream)),
                ("combine", lambda: lib.moe_unpermute_combine(p["y2"], p["src2dst"], p["topk_w"], T, k, H, out,
                                                              stream)),
            ]
        head = [
            ("route", lambda: lib.moe_route_topk(lg, T, E, k, 1, p["topk_ids"], p["topk_w"], stream)),
            ("permute", lambda: lib.moe_permute(p["topk_ids"], T, k, E, p["seg_indptr"], p["src2dst"],
                                                p["dst2src"], p["permute_ws"], self.permute_ws_bytes, stream)),
            ("quant", lambda: lib.fp8_quant_scatter_per_token_group(x, T, H, p["src2dst"], k, P, p["xq"], p["xs"],
                                                                    p["xc"], ld, stream)),
        ]
        if self.fused:  # w13 with the SiLU-and-Mul requantisation in its epilogue, as w4a8_moe_forward runs it
            mid = [("w13", lambda: lib.w4a8_grouped_gemm_silu(p["xq"], p["xs"], p["xc"], ld, w13, w13s,
                                                              p["seg_indptr"], E, I, H, P, p["hq"], p["hs"],
                                                              p["hc"], ld, p["y13"], self.L.hq - self.L.y13,
                                                              stream))]
        else:
            mid = [("w13", lambda: lib.w4a8_grouped_gemm(p["xq"], p["xs"], p["xc"], ld, w13, w13s, p["seg_indptr"],
                                                         E, 2 * I, H, P, p["y13"], None, 0, stream)),
                   ("silu_requant", lambda: lib.silu_mul_requant(p["y13"], P, I, p["hq"], p["hs"], p["hc"], ld,
                                                                 stream))]
        return head + mid + [
            ("w2", lambda: lib.w4a8_grouped_gemm(p["hq"], p["hs"], p["hc"], ld, w2, w2s, p["seg_indptr"], E, H, I,
                                                 P, p["y2"], None, 0, stream)),
            ("combine", lambda: lib.moe_unpermute_combine(p["y2"], p["src2dst"], p["topk_w"], T, k, H, out,
                                                          stream)),
        ]

    def forward(self, x, lg, out, stream):
        """One call of the public layer entry point (or its expert-parallel form) on device buffers."""
        if self.ep:
            return self.lib.w4a8_moe_forward_ep(x.data_ptr(), lg.data_ptr(), self.T, self.H, self.I, self.E,
                                                self.k, 1, self.emap.data_ptr(), self.EL, self.w13.data_ptr(),
                                                self.w13s.data_ptr(), self.w2.data_ptr(), self.w2s.data_ptr(),
                                                out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), stream)
        return self.lib.w4a8_moe_forward(x.data_ptr(), lg.data_ptr(), self.T, self.H, self.I, self.E, self.k, 1,
                                         self.w13.data_ptr(), self.w13s.data_ptr(), self.w2.data_ptr(),
                                         self.w2s.data_ptr(), out.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
                                         stream)

    def forward_host(self, stream):
        """e2e, one step alone: pinned host inputs -> device -> whole layer -> pinned host output."""
        self.x.copy_(self.x_pin, non_blocking=True)
        self.lg.copy_(self.lg_pin, non_blocking=True)
        rc = self.forward(self.x, self.lg, self.out, stream)
        self.out_pin.copy_(self.out, non_blocking=True)
        return rc

    def touched_experts(self):
        import torch
        seg = torch.empty(self.EL + 1, dtype=torch.int64)
        seg.copy_(self.ws[self.L.seg_indptr:self.L.seg_indptr + 8 * (self.EL + 1)].view(torch.int64))
        s = seg.numpy()
        return int(np.count_nonzero(np.diff(s))), s


def run_ours(args, name, cfg):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    seed = args.seed + rank
    if name == "linear":
        return run_linear(args, cfg, dev, world, rank, peaks, peak_src)
    if args.fused_w13:
        cfg = dict(cfg, fused_w13=True)
    r = MoeRunner(cfg, seed, dev)
    res = measure_moe(r, name, cfg, args, dev, world, peaks, peak_src)
    if not args.no_e2e:
        res["e2e"] = e2e_moe(r, args, dev, world)
    if name == "prefill" and not args.no_decode:
        # the decode half of the metric: the same experts (same seed, same tensors), 64 tokens
        dcfg = dict(inputs.WORKLOADS["decode"])
        rd = MoeRunner(dcfg, seed, dev, weights=(r.w13, r.w13s, r.w2, r.w2s))
        d = measure_moe(rd, "decode", dcfg, args, dev, world, peaks, peak_src)
        keep = ("value", "unit", "ms_per_step", "steps", "tflops", "layer_roofline", "stages_ms", "roofline",
                "gpu_launches", "clocks")
        res["decode"] = {"workload": d["config"]["workload"], "experts_touched": d["config"]["experts_touched"],
                         **{kk: d[kk] for kk in keep}}
        if not args.no_e2e:
            res["decode"]["e2e"] = e2e_moe(rd, args, dev, world)
    res["clocks_sustained"] = sustained_clocks(r, dev, args.sustain_s)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(name, args.workload, args)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def sustained_clocks(r, dev, seconds):
    """Steps back to back for about `seconds` after the timed region (untimed), with the clocks sampled:
    the clock and power state of the GPU under this workload's sustained load."""
    import torch
    if seconds <= 0:
        return None
    stream = torch.cuda.current_stream(dev)
    st = r.stages(stream.cuda_stream)
    t = time.perf_counter()
    with clock_sampler(dev) as clk:
        n = 0
        while time.perf_counter() - t < seconds:
            for _ in range(10):
                for nm, fn in st:
                    if fn():
                        raise RuntimeError(f"{nm}: {r.lib.w4a8_last_error().decode()}")
            n += 10
            torch.cuda.synchronize(dev)
    out = clk.summary() or {}
    out["steps"] = n
    return out


def measure_moe(r, name, cfg, args, dev, world, peaks, peak_src):
    """W warm-up steps, then exactly K timed steps of the seven stages back to back; the result line."""
    import torch
    import torch.distributed as dist
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    st = r.stages(sp)

    def check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: {r.lib.w4a8_last_error().decode()}")

    for _ in range(args.warmup):
        for nm, fn in st:
            check(fn(), nm)
    torch.cuda.synchronize(dev)
    n_touched, seg = r.touched_experts()

    K = args.steps
    nst = len(st)
    iw13 = [nm for nm, _ in st].index("w13")
    # Timed region: the stages back to back (each kernel's launch overlaps the previous one's tail,
    # programmatic dependent launch); events only around the dominant w13 launch, for its roofline.
    w13_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with clock_sampler(dev) as clk:
        t0.record(stream)
        for i in range(K):
            for j, (nm, fn) in enumerate(st):
                if j == iw13:
                    w13_ev[i][0].record(stream)
                check(fn(), nm)
                if j == iw13:
                    w13_ev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    w13_timed_ms = float(np.mean([w13_ev[i][0].elapsed_time(w13_ev[i][1]) for i in range(K)]))
    # stage breakdown from a separate, untimed pass with an event after every stage
    nb = min(K, 10)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(nb)]
    for i in range(nb):
        evs[i][0].record(stream)
        for j, (nm, fn) in enumerate(st):
            check(fn(), nm)
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    stage_ms = {nm: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nb)]))
                for j, (nm, _) in enumerate(st)}
    ms = reduce_max(ms, dev)
    T, H, I, E, k = r.T, r.H, r.I, r.E, r.k
    P = int(seg[-1])  # routed pairs computed (all T*k, or the shard's)
    ms_step = ms / K
    value = throughput(T * K, world, ms)
    cnt = moe_counts(T, H, I, E, k, P, n_touched, fused=r.fused)
    flops, layer_bytes = cnt["flops"], cnt["layer_bytes"]
    # dominant kernel: the w13 grouped GEMM, timed inside the long step (sustained tensor peak)
    roof = roofline_core(cnt["w13_bytes"], cnt["w13_flops"], w13_timed_ms, peaks["hbm_gbs"],
                         FP8_OVER_BF16 * peaks["bf16_tflops_sustained"])
    roof.update({"traffic": ncu_traffic(f"{name}:w13"),
                 "kernel": "w4a8_gemm_kernel (w13 grouped GEMM" + (", SiLU-and-Mul requantisation fused)" if r.fused
                                                                    else ")")})
    if roof["bound"] == "hbm":
        roof.update({"algorithmic_bytes": int(cnt["w13_bytes"]), "peak_source": f"{peak_src} hbm_gbs"})
    else:
        roof.update({"algorithmic_flops": cnt["w13_flops"],
                     "peak_source": f"{peak_src} bf16_tflops_sustained x 2 (nominal fp8/bf16 dense ratio)"})
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x int4 -> f32 (bf16 out)", "data": "synthetic",
        "config": {"workload": workload_desc(name, cfg), "T": T, "H": H, "I": I, "E": E, "k": k,
                   "routed_pairs": P, "experts_touched": n_touched,
                   "max_rows_per_expert": int(np.diff(seg).max()),
                   "l2": "no flush: the expert weights (%.2f GB) exceed L2, every step streams them from HBM"
                         % ((r.w13.numel() + r.w2.numel() + 4 * (r.w13s.numel() + r.w2s.numel())) / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tflops": round(flops / (ms_step / 1e3) / 1e12, 2),
        "layer_roofline": {"algorithmic_bytes": int(layer_bytes),
                           "hbm_gbs": round(layer_bytes / (ms_step / 1e3) / 1e9, 1),
                           "hbm_frac": round(layer_bytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                           "fp8_frac": round(flops / (ms_step / 1e3) / 1e12 /
                                             (FP8_OVER_BF16 * peaks["bf16_tflops_sustained"]), 4)},
        "stages_ms": {kk: round(v, 4) for kk, v in stage_ms.items()},
        "stages_note": "stage breakdown from a separate pass with an event after every stage; the timed "
                       "region runs the stages back to back with events only around w13",
        "roofline": roof,
        "gpu_launches": moe_launches_per_step(nst, r.permute_ws_bytes > 0, gemm_plans(r.lib, T * k, r.EL, H, I)) * K,
        "clocks": clk.summary(),
    }


def e2e_bytes(T, H, E):
    """Bytes a layer step copies in (bf16 x and fp32 router logits) and out (bf16 output)."""
    return T * H * 2 + T * E * 4, T * H * 2


def e2e_pipelined(h2d, d2h):
    """Whether the e2e loop overlaps the copies with the layer: from 1 MiB of copies per step."""
    return h2d + d2h >= (1 << 20)


def e2e_moe(r, args, dev, world):
    """The metric end to end as a serving loop runs it: every step copies its inputs from pinned host memory
    to the device, runs the layer through the public entry point and copies its output back to pinned host
    memory.  When a step moves at least 1 MiB between host and device, inputs and outputs are double-buffered
    on the device and the copies run on two more streams (inputs, outputs), so step i+1's inputs arrive and
    step i-1's output leaves while step i computes; smaller steps (whose copies take less than the
    cross-stream waits would) run copy, layer, copy in order on one stream.  Each step's own copies are
    inside the timed region (from the first input copy to the last output copy)."""
    import torch
    import torch.distributed as dist
    h2d, d2h = e2e_bytes(r.T, r.H, r.E)
    if not e2e_pipelined(h2d, d2h):
        return e2e_moe_serial(r, args, dev, world, h2d, d2h)
    stream = torch.cuda.current_stream(dev)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)  # input and output copies: neither waits on the other
    xs = [r.x, torch.empty_like(r.x)]
    lgs = [r.lg, torch.empty_like(r.lg)]
    outs = [r.out, torch.empty_like(r.out)]
    pins = [r.out_pin, torch.empty_like(r.out_pin).pin_memory()]
    ready = [torch.cuda.Event() for _ in range(2)]  # inputs of the buffer copied in
    done = [torch.cuda.Event() for _ in range(2)]   # the layer's call on the buffer finished
    freed = [torch.cuda.Event() for _ in range(2)]  # the buffer's output copied out
    for e in done + freed:
        e.record(stream)

    def run(steps):
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(cin):
                cin.wait_event(done[b])  # the step two back has read this input buffer
                xs[b].copy_(r.x_pin, non_blocking=True)
                lgs[b].copy_(r.lg_pin, non_blocking=True)
                ready[b].record(cin)
            stream.wait_event(ready[b])
            stream.wait_event(freed[b])  # the step two back's output has left this output buffer
            rc = r.forward(xs[b], lgs[b], outs[b], stream.cuda_stream)
            if rc:
                raise RuntimeError(r.lib.w4a8_last_error().decode())
            done[b].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(done[b])
                pins[b].copy_(outs[b], non_blocking=True)
                freed[b].record(cout)

    run(2)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cin)  # before the first input copy
    run(args.steps)
    cout.wait_stream(cin)
    b.record(cout)  # after the last output copy
    torch.cuda.synchronize(dev)
    ms = reduce_max(a.elapsed_time(b), dev)
    return {"value": round(throughput(r.T * args.steps, world, ms), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "w4a8_moe_forward (one C call per step) + cudaMemcpyAsync from/to pinned host on input and output "
                   "copy streams, double-buffered: the next step's input and the previous step's output copies "
                   "overlap a step"}


def e2e_moe_serial(r, args, dev, world, h2d, d2h):
    """e2e for small steps: input copy, layer, output copy in order on one stream, every step."""
    import torch
    import torch.distributed as dist
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        r.forward_host(stream.cuda_stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        rc = r.forward_host(stream.cuda_stream)
        if rc:
            raise RuntimeError(r.lib.w4a8_last_error().decode())
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = reduce_max(a.elapsed_time(b), dev)
    return {"value": round(throughput(r.T * args.steps, world, ms), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "w4a8_moe_forward (one C call per step) + cudaMemcpyAsync from/to pinned host, in order on one "
                   "stream"}


def run_linear(args, cfg, dev, world, rank, peaks, peak_src):
    import torch

    import w4afp8_mixture_experts_gb300 as m
    lib = m.load()
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    G = K // 128
    # several weight copies so that consecutive steps do not hit L2
    copies = max(1, int(np.ceil(2 * 129e6 / (N * K // 2))))
    Ws = [m.w4a8_prepack_weights(inputs.gpu_packed_int4(args.seed + c, inputs.STREAM_LIN_W, (N, K // 2), dev))
          for c in range(copies)]
    Ss = [inputs.gpu_scales(args.seed + c, inputs.STREAM_LIN_SCALE, (G, N), dev) for c in range(copies)]
    rng = np.random.default_rng(args.seed)
    x = torch.from_numpy(inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32)).view(np.int16)).view(
        torch.bfloat16).to(dev)
    aq, a_s, a_c = m.fp8_quant_per_token_group(x)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    need = m.linear_workspace_bytes(M, N, K)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream

    def step(i, stream=sp):
        return lib.w4a8_linear(aq.data_ptr(), a_s.data_ptr(), a_c.data_ptr(), a_s.shape[1], Ws[i % copies].data_ptr(),
                               Ss[i % copies].data_ptr(), M, N, K, C.data_ptr(), ws.data_ptr(), need, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    Kst = args.steps
    # events only around the K calls: the calls are launched back to back, as a model would, so a
    # call's launch and prologue overlap the previous call (programmatic dependent launch)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with clock_sampler(dev) as clk:
        evs[0].record()
        for i in range(Kst):
            rc = step(i)
            if rc:
                raise RuntimeError(lib.w4a8_last_error().decode())
        evs[1].record()
        torch.cuda.synchronize(dev)
    eager_ms = evs[0].elapsed_time(evs[1])
    # The same K calls captured once in a CUDA graph and replayed: a call of a few microseconds is then
    # timed without the host's submission (a Python call per kernel, which a thread switch can stall)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cs = torch.cuda.current_stream(dev).cuda_stream
        for i in range(Kst):
            if step(i, cs):
                raise RuntimeError(lib.w4a8_last_error().decode())
    graph.replay()
    torch.cuda.synchronize(dev)
    with clock_sampler(dev) as clk:
        evs[2].record()
        graph.replay()
        evs[3].record()
        torch.cuda.synchronize(dev)
    ms = evs[2].elapsed_time(evs[3])
    ms_step = ms / Kst
    cnt = linear_counts(M, N, K)
    tf = cnt["flops"] / (ms_step / 1e3) / 1e12
    # a call timed alone: the burst tensor peak
    roof = roofline_core(cnt["bytes"], cnt["flops"], ms_step, peaks["hbm_gbs"], FP8_OVER_BF16 * peaks["bf16_tflops"])
    roof.update({"traffic": ncu_traffic(f"linear:{M},{N},{K}"),
                 "kernel": "w4a8_gemm_kernel (dense; per call, incl. the split-K reduce when S > 1)",
                 "peak_source": peak_src})
    res = {"metric": METRIC, "value": round(M / (ms_step / 1e3), 2), "unit": "tokens/s", "n_gpus": world,
           "steps": Kst, "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x int4 -> f32 (bf16 out)", "data": "synthetic",
           "config": {"workload": workload_desc("linear", cfg), "l2": f"{copies} rotating weight copies",
                      "timing": "the K calls replayed from a CUDA graph captured once (eager_ms_per_step: the same "
                                "calls launched one by one from Python)"},
           "eager_ms_per_step": round(eager_ms / Kst, 5),
           "tflops": round(tf, 2), "roofline": roof, "gpu_launches": Kst * (2 if m.linear_split_k(M, N, K) > 1 else 1),
           "split_k": m.linear_split_k(M, N, K), "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(res), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)

def oracle_sample(name, cfg, seed, tokens):
    """Host inputs and weights of a token sample (token indices `tokens`); returns a closure running the
    oracle on it.  The weights are generated here, before any timing (model parameters in memory)."""
    import oracle
    from helpers import moe_experts, moe_host_inputs
    x_bits, logits = moe_host_inputs(seed, cfg)
    x = inputs.bf16_bits_to_f32(x_bits)
    w13, w2 = moe_experts(seed, cfg)
    sel = np.asarray(tokens)
    ids, _ = oracle.route_topk(logits[sel], cfg["k"])
    emap, glob = None, np.arange(cfg["E"])
    if cfg.get("ep"):  # one expert-parallel shard: local id l is global expert r + l*R
        R, r = cfg["ep"]
        glob = np.arange(r, cfg["E"], R)
        emap = np.full(cfg["E"], -1, np.int64)
        emap[glob] = np.arange(glob.size)
    used = [int(e) for e in np.unique(ids) if emap is None or emap[e] >= 0]
    loc = {(int(emap[e]) if emap is not None else e): e for e in used}
    cache13 = {l: (w13.w(e), w13.s(e)) for l, e in loc.items()}
    cache2 = {l: (w2.w(e), w2.s(e)) for l, e in loc.items()}
    xs, lgs = x[sel], logits[sel]

    def run():
        return oracle.moe_tokens(xs, lgs, cfg["k"], lambda e: cache13[e][0], lambda e: cache13[e][1],
                                 lambda e: cache2[e][0], lambda e: cache2[e][1], expert_map=emap)
    return run


def _oracle_worker(name, cfg, seed, tokens, core, rounds, barrier, out):
    """One host core of the CPU baseline: prepares its tokens' sample, then for each round waits for every
    worker (barrier) and times the oracle on its tokens."""
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    try:
        mine = sorted(os.sched_getaffinity(0))
        os.sched_setaffinity(0, {mine[core % len(mine)]})
    except (AttributeError, OSError):
        pass
    run = oracle_sample(name, cfg, seed, tokens)
    for _ in range(rounds):
        barrier.wait()
        t = time.perf_counter()
        run()
        out.put(time.perf_counter() - t)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_on_host_cores(name, cfg, seed, per_core, rounds, cores=None):
    """The oracle over `cores` processes (spawn start; one BLAS thread each), `per_core` tokens each, the
    cores' token samples disjoint; every round starts on all cores together.  Returns the wall time of
    each round (the slowest core's) and the number of tokens a round processes."""
    import multiprocessing as mp
    cores = cores or host_cores()
    T = cfg["T"]
    ctx = mp.get_context("spawn")
    barrier, out = ctx.Barrier(cores), ctx.Queue()
    procs = []
    for c in range(cores):
        tokens = [(c * per_core + i) % T for i in range(per_core)]
        p = ctx.Process(target=_oracle_worker, args=(name, cfg, seed, tokens, c, rounds, barrier, out), daemon=True)
        p.start()
        procs.append(p)
    per_round = []
    for _ in range(rounds):
        per_round.append(max(out.get(timeout=900) for _ in range(cores)))
    for p in procs:
        p.join(timeout=60)
    return per_round, cores * per_core, cores


def default_cpu_tokens(name):
    return {"tiny": 64}.get(name, 1)


def run_reference(args, name, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if name == "linear":
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the MoE workloads"}))
        return
    n = args.cpu_tokens or default_cpu_tokens(name)
    rounds, tokens, cores = oracle_on_host_cores(name, cfg, args.seed, n, args.warmup + args.steps)
    times = rounds[args.warmup:]
    tot = sum(times)
    value = tokens * len(times) / tot
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / len(times), 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": workload_desc(name, cfg)},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"{tokens} token(s) of the workload per step, {n} on each of {cores} host "
                                      f"cores ({n * cfg['k']} routed pairs per core"
                                      f"{', those of the shard computed' if cfg.get('ep') else ''}), numpy "
                                      f"float64, one BLAS thread per process, rounds started together"},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def cpu_baseline(name, spec, args):
    """The oracle over the host's cores on a bounded sample (~10-30 s), in a child process."""
    n = {"tiny": 8}.get(name, 4 if name.startswith("ep-") else 2)
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", spec, "--steps", "1",
           "--warmup", "0", "--cpu-tokens", str(n), "--seed", str(args.seed)]
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(v, None)
    try:
        out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900).stdout.strip().splitlines()
        d = json.loads(out[-1])
        return d["cpu_baseline"]
    except Exception as e:  # reported, never fatal for the GPU number
        return {"value": None, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle", "sample": f"failed: {e}"}


def main():
    args = parse()
    name, cfg = get_workload(args.workload)
    if args.impl == "reference":
        run_reference(args, name, cfg)
    else:
        run_ours(args, name, cfg)


if __name__ == "__main__":
    main()
