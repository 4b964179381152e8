"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module holds no arithmetic of the W4AFP8 MoE method.  It only makes
numbers:

* Large tensors that must be identical on the host and on the GPU (the packed
  int4 expert weights and their fp32 group scales) come from one
  counter-based generator, SplitMix64 (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014), used in counter
  mode: word ``i`` of stream ``s`` under seed ``seed`` is
  ``mix64(key(seed, s) + (i + 1) * GAMMA)``.  The CUDA twin of these
  functions lives in ``inputs/gen.cu`` and is tested against this file.
* Small host tensors (activations, router logits) come from numpy's PCG64
  ``Generator`` and are copied to the device.

Derived values:
  packed int4 byte  = top 8 bits of the word  (two independent uniform nibbles,
                      i.e. int4 values uniform on [-8, 7] in two's complement)
  uniform u in [0,1) = (word >> 40) * 2**-24  (exact in fp32)
  scale             = fp32(lo) + fp32(span) * fp32(u)   (two fp32 roundings,
                      no fused multiply-add), lo = 0.005, span = 0.015
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

SCALE_LO = np.float32(0.005)
SCALE_SPAN = np.float32(0.015)

# Stream ids, one per synthetic tensor kind.
STREAM_W13 = 1
STREAM_W13_SCALE = 2
STREAM_W2 = 3
STREAM_W2_SCALE = 4
STREAM_LIN_W = 5
STREAM_LIN_SCALE = 6


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Stafford's Mix13 constants), on uint64 arrays."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of one counter stream: mix64(GAMMA * (seed * 2**16 + stream + 1))."""
    base = np.uint64(((int(seed) << 16) + int(stream) + 1) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        return mix64(np.array([base * GAMMA], dtype=np.uint64))[0]


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Words start .. start+count-1 of one stream (uint64)."""
    key = stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + idx * GAMMA)


def packed_int4(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Bytes start .. start+count-1 of a packed int4 tensor (uint8)."""
    return (words(seed, stream, start, count) >> np.uint64(56)).astype(np.uint8)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """24-bit uniforms in [0, 1) as float32 (exact)."""
    w = words(seed, stream, start, count) >> np.uint64(40)
    return w.astype(np.float32) * np.float32(2.0 ** -24)


def scales(seed: int, stream: int, start: int, count: int,
           lo: np.float32 = SCALE_LO, span: np.float32 = SCALE_SPAN) -> np.ndarray:
    """fp32 scales uniform in [lo, lo+span): fp32(lo) + fp32(span)*u, two roundings."""
    u = uniform01(seed, stream, start, count)
    prod = (np.float32(span) * u).astype(np.float32)
    return (np.float32(lo) + prod).astype(np.float32)


# ----------------------------------------------------------------------------
# Host tensors from PCG64 (activations, router logits).

def normal_f32(seed: int, shape, stream: int = 0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64([int(seed), int(stream)]))
    return rng.standard_normal(size=shape, dtype=np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations_bf16(seed: int, T: int, H: int) -> np.ndarray:
    """x ~ N(0,1), rounded to bf16; returned as uint16 bit patterns [T, H]."""
    return to_bf16_bits(normal_f32(seed, (T, H), stream=11))


def zipf_bias(seed: int, E: int, s: float = 1.2) -> np.ndarray:
    """Additive log-popularity bias: bias[e] = ln p_{pi(e)}, p_r ~ r^-s, pi a seeded permutation."""
    rng = np.random.Generator(np.random.PCG64([int(seed), 13]))
    perm = rng.permutation(E)
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    return np.log(p[perm]).astype(np.float32)


def router_logits(seed: int, T: int, E: int, zipf: float | None = None) -> np.ndarray:
    """Router logits fp32 [T, E]: N(0,1), plus a Zipf(s) popularity bias when zipf is set."""
    lg = normal_f32(seed, (T, E), stream=12)
    if zipf is not None:
        lg = (lg + zipf_bias(seed, E, zipf)[None, :]).astype(np.float32)
    return lg


# ----------------------------------------------------------------------------
# Workload shapes (synthetic stand-ins for the DeepSeek-V3/R1-class MoE layer).

WORKLOADS = {
    "tiny": dict(T=64, H=256, I=512, E=8, k=2, zipf=None),
    "decode": dict(T=64, H=7168, I=2048, E=256, k=8, zipf=None),
    "prefill": dict(T=8192, H=7168, I=2048, E=256, k=8, zipf=None),
    "skewed": dict(T=4096, H=7168, I=2048, E=384, k=8, zipf=1.2),
}

LINEAR_M = (1, 16, 128, 1024, 8192)
LINEAR_NK = ((24576, 1536), (7168, 16384), (18432, 7168), (7168, 2048))


def expert_weight_bytes(seed: int, stream: int, E: int, N: int, K: int, experts) -> dict:
    """Packed int4 bytes of selected experts of a [E, N, K/2] tensor: {e: uint8 [N, K/2]}."""
    per = N * (K // 2)
    return {int(e): packed_int4(seed, stream, int(e) * per, per).reshape(N, K // 2)
            for e in experts}


def expert_scales(seed: int, stream: int, E: int, N: int, K: int, experts) -> dict:
    """fp32 group scales of selected experts of a [E, K/128, N] tensor: {e: fp32 [K/128, N]}."""
    G = K // 128
    per = G * N
    return {int(e): scales(seed, stream, int(e) * per, per).reshape(G, N) for e in experts}


# ----------------------------------------------------------------------------
# Device twin (inputs/gen.cu): the same streams, filled on the GPU.

import os as _os  # noqa: E402

_GEN_SRC = _os.path.join(_os.path.dirname(_os.path.abspath(__file__)), "gen.cu")
_GEN_LIB = _os.path.join(_os.path.dirname(_os.path.abspath(__file__)), "_lib", "libw4a8gen.so")
_gen = None


def build_gen() -> str:
    from w4afp8_mixture_experts_gb300.build import build_shared
    return build_shared([_GEN_SRC], _GEN_LIB, [])


def _genlib():
    global _gen
    if _gen is None:
        import ctypes
        if not _os.path.exists(_GEN_LIB):
            raise RuntimeError(f"{_GEN_LIB} is missing: run inputs.build_gen()")
        lib = ctypes.CDLL(_GEN_LIB)
        lib.w4a8gen_fill_int4.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                          ctypes.c_uint32, ctypes.c_void_p]
        lib.w4a8gen_fill_scales.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                            ctypes.c_uint32, ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
        _gen = lib
    return _gen


def gpu_packed_int4(seed: int, stream: int, shape, device="cuda", start: int = 0):
    """torch uint8 tensor of `shape` on the GPU: bytes start.. of the stream."""
    import ctypes

    import torch
    t = torch.empty(shape, dtype=torch.uint8, device=device)
    st = ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    rc = _genlib().w4a8gen_fill_int4(ctypes.c_void_p(t.data_ptr()), start, t.numel(), seed, stream, st)
    if rc:
        raise RuntimeError(f"w4a8gen_fill_int4 failed ({rc})")
    return t


def gpu_scales(seed: int, stream: int, shape, device="cuda", start: int = 0):
    """torch fp32 tensor of `shape` on the GPU: scales start.. of the stream."""
    import ctypes

    import torch
    t = torch.empty(shape, dtype=torch.float32, device=device)
    st = ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    rc = _genlib().w4a8gen_fill_scales(ctypes.c_void_p(t.data_ptr()), start, t.numel(), seed, stream,
                                       float(SCALE_LO), float(SCALE_SPAN), st)
    if rc:
        raise RuntimeError(f"w4a8gen_fill_scales failed ({rc})")
    return t
