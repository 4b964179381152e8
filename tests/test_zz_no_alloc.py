"""The layer entry point that allocates nothing, for callers that cannot allocate device memory.

Such callers (a plugin whose host application owns every device allocation, a
C program that must not allocate after start-up) pass only inputs and outputs;
w4a8_moe_forward_noalloc keeps the intermediates in a fixed array inside the
library.  This test calls it through the C ABI twice in a row and checks each
result against w4a8_moe_forward given an ordinary workspace.  The file sorts
last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import inputs
from gpu_util import bf16_from_bits, f64_of_bf16, rel_fro, to_dev
from helpers import moe_host_inputs

pytestmark = pytest.mark.gpu

CFGS = [dict(T=64, H=256, I=512, E=8, k=2), dict(T=24, H=1024, I=768, E=16, k=4)]


def _weights(lib, seed, cfg):
    H, I, E = cfg["H"], cfg["I"], cfg["E"]
    return (lib.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W13, (E, 2 * I, H // 2))),
            inputs.gpu_scales(seed, inputs.STREAM_W13_SCALE, (E, H // 128, 2 * I)),
            lib.w4a8_prepack_weights(inputs.gpu_packed_int4(seed, inputs.STREAM_W2, (E, H, I // 2))),
            inputs.gpu_scales(seed, inputs.STREAM_W2_SCALE, (E, I // 128, H)))


def _noalloc(clib, x, lg, cfg, w, out):
    T, H, I, E, k = (cfg[n] for n in ("T", "H", "I", "E", "k"))
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = [ctypes.c_void_p(t.data_ptr()) for t in (x, lg) + w + (out,)]
    return clib.w4a8_moe_forward_noalloc(p[0], p[1], T, H, I, E, k, 1, p[2], p[3], p[4], p[5], p[6], st)


def test_noalloc_matches_workspace_entry_point(lib):
    clib = lib.load()
    assert clib.w4a8_moe_noalloc_scratch_bytes() == 64 << 20
    for seed, cfg in enumerate(CFGS):
        x_bits, logits = moe_host_inputs(seed, cfg)
        x, lg = bf16_from_bits(x_bits), to_dev(logits)
        w = _weights(lib, seed, cfg)
        ref = f64_of_bf16(lib.w4a8_moe_forward(x, lg, cfg["k"], *w))
        outs = [torch.full((cfg["T"], cfg["H"]), float("nan"), dtype=torch.bfloat16, device="cuda")
                for _ in range(3)]
        # a first call on the device sets the entry point up (and may be when the driver first places the
        # library's fixed array in device memory); the two checked calls after it must not take any
        assert _noalloc(clib, x, lg, cfg, w, outs[0]) == 0, clib.w4a8_last_error()
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        for call in (1, 2):  # the shared array keeps the previous call's contents
            assert _noalloc(clib, x, lg, cfg, w, outs[call]) == 0, clib.w4a8_last_error()
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before
        for call in (1, 2):
            got = f64_of_bf16(outs[call])
            assert np.all(np.isfinite(got))
            assert rel_fro(got, ref) <= 1e-3, (seed, call)
    assert lib.device_error() == 0


def test_noalloc_rejects_layers_beyond_the_array(lib):
    clib = lib.load()
    cfg = dict(T=4096, H=7168, I=2048, E=8, k=8)  # ~1 GB of intermediates
    need = clib.w4a8_moe_workspace_bytes(cfg["T"], cfg["H"], cfg["I"], cfg["E"], cfg["k"])
    assert need > clib.w4a8_moe_noalloc_scratch_bytes()
    x = torch.zeros((cfg["T"], cfg["H"]), dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros((cfg["T"], cfg["E"]), dtype=torch.float32, device="cuda")
    w = (torch.zeros(16, dtype=torch.uint8, device="cuda"),) * 4
    out = torch.zeros_like(x)
    assert _noalloc(clib, x, lg, cfg, w, out) == 1  # W4A8_ERR_INVALID_ARG, nothing launched
    assert b"at most" in clib.w4a8_last_error()
