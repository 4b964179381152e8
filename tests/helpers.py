"""Glue between the seeded generators and the oracle (host side only)."""
import functools

import numpy as np

import inputs
import oracle


class HostExperts:
    """Lazily regenerated expert weights of one workload, in the oracle's layout.

    Packed int4 [E, N, K/2] and fp32 scales [E, K/128, N] come from the
    counter-based generator; the oracle wants int8 [N, K] and fp32 [N, K/128].
    """

    def __init__(self, seed, E, N, K, w_stream, s_stream):
        self.seed, self.E, self.N, self.K = seed, E, N, K
        self.w_stream, self.s_stream = w_stream, s_stream

    @functools.lru_cache(maxsize=16)
    def packed(self, e):
        per = self.N * (self.K // 2)
        return inputs.packed_int4(self.seed, self.w_stream, e * per, per).reshape(self.N, self.K // 2)

    def w(self, e):
        return oracle.unpack_int4(self.packed(int(e)))

    @functools.lru_cache(maxsize=64)
    def s(self, e):
        G = self.K // 128
        per = G * self.N
        return np.ascontiguousarray(
            inputs.scales(self.seed, self.s_stream, int(e) * per, per).reshape(G, self.N).T)


def moe_experts(seed, cfg):
    H, I, E = cfg["H"], cfg["I"], cfg["E"]
    w13 = HostExperts(seed, E, 2 * I, H, inputs.STREAM_W13, inputs.STREAM_W13_SCALE)
    w2 = HostExperts(seed, E, H, I, inputs.STREAM_W2, inputs.STREAM_W2_SCALE)
    return w13, w2


def moe_host_inputs(seed, cfg):
    x_bits = inputs.activations_bf16(seed, cfg["T"], cfg["H"])
    logits = inputs.router_logits(seed, cfg["T"], cfg["E"], cfg.get("zipf"))
    return x_bits, logits
